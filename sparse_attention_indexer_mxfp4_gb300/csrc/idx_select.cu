// idx_select.cu -- per-row top-k (cluster radix select), candidate mask and
// top-k -> ragged slot map, with their C ABI entry points.
#include <cooperative_groups.h>
#include <algorithm>
#include <cstdint>

#include "idx_internal.h"

namespace cg = cooperative_groups;

namespace idx {
namespace {

// ------------------------------------------------------------------ top-k
//
// Passage: vLLM page rocm_paged_mxfp4_indexer, _topk -- top-k over each
// row's [0, lengths[row]), -1 padding.  The design is our own: each row is
// handled by one thread-block cluster of C CTAs.  CTA c of the cluster copies
// its slice of the row into shared memory once, as order-preserving 32-bit
// keys (non-finite values become key 0 and are never selected), and the
// cluster then runs a three-digit (11/11/10 bit) radix select: each CTA
// histograms its slice for the current digit, the C histograms are summed
// through distributed shared memory, and every CTA finds the same digit of
// the k-th largest key.  Finally every CTA writes its selected indices in
// ascending index order at offsets given by a cluster prefix sum.  Elements
// equal to the k-th largest key are taken lowest index first, so the
// selected set is unique.  All waits are hardware cluster barriers that every
// CTA reaches on the same, data-independent path.

constexpr int kTopkThreads = 512;
constexpr int kMaxCluster = 8;  // portable cluster size
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t float_key(float v)
{
    uint32_t b = __float_as_uint(v);
    if (!isfinite(v))
        return 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Block-wide exclusive scan of one uint32 per thread; returns the exclusive
// prefix, *total gets the sum.  Uses wsum[kTopkWarps + 1].
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *wsum, uint32_t *total)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t x = v;
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t n = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += n;
    }
    if (lane == 31)
        wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        uint32_t s = lane < kTopkWarps ? wsum[lane] : 0u;
        uint32_t incl = s;
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += n;
        }
        if (lane < kTopkWarps)
            wsum[lane] = incl - s;
        if (lane == 31)
            wsum[kTopkWarps] = incl;
    }
    __syncthreads();
    uint32_t r = wsum[w] + x - v;
    *total = wsum[kTopkWarps];
    __syncthreads();
    return r;
}

struct TopkShared {
    uint32_t hist[2][2048];
    uint32_t wsum[kTopkWarps + 1];
    uint32_t counts[4];  // valid, greater, equal (this CTA)
    uint32_t sel[4];     // digit found, remaining k, ...
};

__global__ void __launch_bounds__(kTopkThreads)
    topk_cluster_kernel(const float *__restrict__ logits, int64_t ld, int rows,
                        const int32_t *__restrict__ lengths, int k, int32_t *__restrict__ out,
                        int64_t ld_out, int slice_cap)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int row = blockIdx.x / C;
    extern __shared__ __align__(16) uint8_t dsm[];
    TopkShared &sh = *reinterpret_cast<TopkShared *>(dsm);
    uint32_t *keys = reinterpret_cast<uint32_t *>(dsm + sizeof(TopkShared));
    const int tid = threadIdx.x;

    const bool row_ok = row < rows;  // every CTA of a cluster shares the row
    int len = row_ok ? lengths[row] : 0;
    len = max(0, min(len, (int)ld));
    const int per = (len + C - 1) / C;
    const int lo = min(len, crank * per);
    const int hi = min(len, lo + per);
    const int n = hi - lo;  // <= slice_cap by construction of the launch
    (void)slice_cap;

    // load the slice as keys, count valid keys, digit-1 histogram
    for (int i = tid; i < 2 * 2048; i += kTopkThreads)
        (&sh.hist[0][0])[i] = 0u;
    __syncthreads();
    uint32_t nvalid = 0;
    const float *src = logits + (size_t)(row_ok ? row : 0) * ld + lo;
    for (int i = tid; i < n; i += kTopkThreads) {
        uint32_t key = float_key(__ldg(src + i));
        keys[i] = key;
        if (key) {
            ++nvalid;
            atomicAdd(&sh.hist[0][key >> 21], 1u);
        }
    }
    uint32_t tot;
    (void)block_excl_scan(nvalid, sh.wsum, &tot);
    if (tid == 0)
        sh.counts[0] = tot;
    cluster.sync();
    uint32_t total_valid = 0;
    for (int r = 0; r < C; ++r)
        total_valid += cluster.map_shared_rank(&sh, r)->counts[0];

    // radix select of the threshold key T and the number of ties to take
    uint32_t prefix = 0, prefix_mask = 0;
    uint32_t krem = (uint32_t)k;
    bool take_all = total_valid <= (uint32_t)k;
    const int shifts[3] = {21, 10, 0};
    const int nbins[3] = {2048, 2048, 1024};
    for (int pass = 0; pass < 3 && !take_all; ++pass) {
        uint32_t *h = sh.hist[pass & 1];
        if (pass > 0) {
            for (int i = tid; i < 2048; i += kTopkThreads)
                h[i] = 0u;
            __syncthreads();
            const uint32_t dmask = (uint32_t)nbins[pass] - 1u;
            for (int i = tid; i < n; i += kTopkThreads) {
                uint32_t key = keys[i];
                if (key && (key & prefix_mask) == prefix)
                    atomicAdd(&h[(key >> shifts[pass]) & dmask], 1u);
            }
            cluster.sync();
        }
        // summed histogram; thread t owns 4 bins in descending order
        const int nb = nbins[pass];
        uint32_t loc[4];
        uint32_t lsum = 0;
        for (int j = 0; j < 4; ++j) {
            int b = nb - 1 - (tid * 4 + j);
            uint32_t s = 0;
            if (b >= 0)
                for (int r = 0; r < C; ++r)
                    s += cluster.map_shared_rank(h, r)[b];
            loc[j] = s;
            lsum += s;
        }
        uint32_t before = block_excl_scan(lsum, sh.wsum, &tot);
        for (int j = 0; j < 4; ++j) {
            int b = nb - 1 - (tid * 4 + j);
            if (b >= 0 && before < krem && before + loc[j] >= krem) {
                sh.sel[0] = (uint32_t)b;
                sh.sel[1] = krem - before;
            }
            before += loc[j];
        }
        __syncthreads();
        const uint32_t digit = sh.sel[0];
        krem = sh.sel[1];
        prefix |= digit << shifts[pass];
        prefix_mask |= ((uint32_t)nb - 1u) << shifts[pass];
        __syncthreads();
    }
    // T = prefix (full key); select key > T, plus the first krem keys == T.
    const uint32_t T = take_all ? 0u : prefix;
    const uint32_t ties = take_all ? 0u : krem;

    // per-CTA counts of greater and equal keys, cluster prefix sums
    uint32_t ngt = 0, neq = 0;
    for (int i = tid; i < n; i += kTopkThreads) {
        uint32_t key = keys[i];
        ngt += key > T;
        neq += (key == T) && key;
    }
    uint32_t cgt, ceq;
    (void)block_excl_scan(ngt, sh.wsum, &cgt);
    (void)block_excl_scan(neq, sh.wsum, &ceq);
    if (tid == 0) {
        sh.counts[1] = cgt;
        sh.counts[2] = ceq;
    }
    cluster.sync();
    uint32_t gt_before = 0, eq_before = 0, total_sel = 0;
    for (int r = 0; r < C; ++r) {
        const TopkShared *o = cluster.map_shared_rank(&sh, r);
        const uint32_t g = o->counts[1], e = o->counts[2];
        if (r < crank) {
            gt_before += g;
            eq_before += e;
        }
        total_sel += g;
    }
    // ties: the first `ties` equal keys in index order across the cluster
    const uint32_t my_quota = eq_before >= ties ? 0u : min(ceq, ties - eq_before);
    uint32_t ties_before = min(eq_before, ties);
    total_sel += ties;
    const uint32_t base = gt_before + ties_before;

    // ordered compaction of this CTA's selection
    uint32_t written = 0, eq_seen = 0;
    int32_t *orow = out + (size_t)(row_ok ? row : 0) * ld_out;
    for (int start = 0; start < n; start += kTopkThreads) {
        int i = start + tid;
        uint32_t key = i < n ? keys[i] : 0u;
        uint32_t is_eq = (key == T && key) ? 1u : 0u;
        uint32_t tot_eq;
        uint32_t eq_rank = eq_seen + block_excl_scan(is_eq, sh.wsum, &tot_eq);
        uint32_t take = (key > T) || (is_eq && eq_rank < my_quota) ? 1u : 0u;
        uint32_t tot_take;
        uint32_t pos = written + block_excl_scan(take, sh.wsum, &tot_take);
        if (take && row_ok)
            orow[base + pos] = lo + i;
        written += tot_take;
        eq_seen += tot_eq;
    }
    // -1 padding of [total_sel, k), spread over the cluster
    if (row_ok)
        for (int j = (int)total_sel + crank * kTopkThreads + tid; j < k; j += C * kTopkThreads)
            orow[j] = -1;
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// ---------------------------------------------------------- candidate mask
//
// Passage: vLLM page rocm_aiter_mla_sparse, _apply_candidate_mask_strided:
// keep column t of row r iff ks <= t < ke and block (t - ks) / block_size is
// a candidate of row r / row_repeat; write -inf elsewhere in [0, ke).  Each
// CTA rebuilds the row's candidate bitmap in shared memory and only writes.

__global__ void candidate_mask_kernel(float *__restrict__ logits, int64_t ld, int rows, int width,
                                      const int32_t *__restrict__ row_ks,
                                      const int32_t *__restrict__ row_ke,
                                      const int32_t *__restrict__ cand, int64_t cand_stride,
                                      int num_cand, int block_size, int row_repeat, int words)
{
    extern __shared__ uint32_t bm[];
    const int r = blockIdx.x;
    if (r >= rows)
        return;
    for (int i = threadIdx.x; i < words; i += blockDim.x)
        bm[i] = 0u;
    __syncthreads();
    const int32_t *cr = cand + (size_t)(r / row_repeat) * cand_stride;
    for (int e = threadIdx.x; e < num_cand; e += blockDim.x) {
        int id = cr[e];
        if (id >= 0 && id < words * 32)
            atomicOr(&bm[id >> 5], 1u << (id & 31));
    }
    __syncthreads();
    const int ke = max(0, min(row_ke[r], width));
    const int ks = row_ks ? max(0, min(row_ks[r], ke)) : 0;
    const int chunk = (width + gridDim.y - 1) / gridDim.y;
    const int c0 = blockIdx.y * chunk;
    const int c1 = min(ke, c0 + chunk);
    float *row = logits + (size_t)r * ld;
    for (int t = c0 + threadIdx.x; t < c1; t += blockDim.x) {
        bool keep = false;
        if (t >= ks) {
            int b = (t - ks) / block_size;
            keep = b < words * 32 && ((bm[b >> 5] >> (b & 31)) & 1u);
        }
        if (!keep)
            row[t] = -INFINITY;
    }
}

// ------------------------------------------------------------- slot map
//
// Passage: vLLM page rocm_aiter_mla_sparse, build_prefill_topk_ragged_indices
// and page rocm_aiter_mla, _expand_page_indices_kernel: position p of
// sequence b lives at slot block_table[b, p / P] * P + p % P.

__device__ __forceinline__ int slot_of(int p, int b, const int32_t *bt, int64_t bt_stride,
                                       int max_blocks, int P, int num_pages)
{
    if (p < 0)
        return -1;
    const int lp = p / P;
    if (lp >= max_blocks)
        return -2;
    const int pg = bt[(size_t)b * bt_stride + lp];
    if (pg < 0 || pg >= num_pages)
        return -2;
    return pg * P + (p - lp * P);
}

constexpr int kSlotThreads = 256;

__global__ void __launch_bounds__(kSlotThreads)
    slot_count_kernel(const int32_t *__restrict__ topk, int64_t ld, int rows, int k,
                      const int32_t *__restrict__ row_to_seq, int next_n,
                      const int32_t *__restrict__ bt, int64_t bt_stride, int max_blocks, int P,
                      int num_pages, int32_t *__restrict__ lens, unsigned int *status)
{
    __shared__ uint32_t wsum[kSlotThreads / 32];
    const int r = blockIdx.x;
    const int b = row_to_seq ? row_to_seq[r] : r / next_n;
    uint32_t cnt = 0, bad = 0;
    for (int j = threadIdx.x; j < k; j += kSlotThreads) {
        int s = slot_of(topk[(size_t)r * ld + j], b, bt, bt_stride, max_blocks, P, num_pages);
        cnt += s >= 0;
        bad += s == -2;
    }
    for (int o = 16; o > 0; o >>= 1)
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if ((threadIdx.x & 31) == 0)
        wsum[threadIdx.x >> 5] = cnt;
    if (bad)
        atomicOr(status, 1u);
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int i = 0; i < kSlotThreads / 32; ++i)
            t += wsum[i];
        lens[r] = (int32_t)t;
    }
}

__global__ void __launch_bounds__(1024) indptr_scan_kernel(const int32_t *__restrict__ lens, int rows,
                                                           int32_t *__restrict__ indptr)
{
    __shared__ int32_t wsum[32];
    __shared__ int32_t carry;
    if (threadIdx.x == 0) {
        carry = 0;
        indptr[0] = 0;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int base = 0; base < rows; base += 1024) {
        int i = base + threadIdx.x;
        int v = i < rows ? lens[i] : 0;
        int x = v;
        for (int o = 1; o < 32; o <<= 1) {
            int nb = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += nb;
        }
        if (lane == 31)
            wsum[w] = x;
        __syncthreads();
        if (w == 0) {
            int s = wsum[lane];
            int incl = s;
            for (int o = 1; o < 32; o <<= 1) {
                int nb = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += nb;
            }
            wsum[lane] = incl - s;
        }
        __syncthreads();
        int c = carry;
        if (i < rows)
            indptr[i + 1] = c + wsum[w] + x;
        __syncthreads();
        if (threadIdx.x == 1023)
            carry = c + wsum[w] + x;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kSlotThreads)
    slot_write_kernel(const int32_t *__restrict__ topk, int64_t ld, int rows, int k,
                      const int32_t *__restrict__ row_to_seq, int next_n,
                      const int32_t *__restrict__ bt, int64_t bt_stride, int max_blocks, int P,
                      int num_pages, const int32_t *__restrict__ indptr,
                      int32_t *__restrict__ slots)
{
    __shared__ uint32_t wsum[kSlotThreads / 32 + 1];
    const int r = blockIdx.x;
    const int b = row_to_seq ? row_to_seq[r] : r / next_n;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int32_t *dst = slots + indptr[r];
    uint32_t written = 0;
    for (int start = 0; start < k; start += kSlotThreads) {
        int j = start + threadIdx.x;
        int s = j < k ? slot_of(topk[(size_t)r * ld + j], b, bt, bt_stride, max_blocks, P,
                                num_pages)
                      : -1;
        uint32_t keep = s >= 0;
        uint32_t ball = __ballot_sync(0xffffffffu, keep);
        uint32_t in_warp = __popc(ball & ((1u << lane) - 1u));
        if (lane == 0)
            wsum[w] = __popc(ball);
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t acc = 0;
            for (int i = 0; i < kSlotThreads / 32; ++i) {
                uint32_t t = wsum[i];
                wsum[i] = acc;
                acc += t;
            }
            wsum[kSlotThreads / 32] = acc;
        }
        __syncthreads();
        if (keep)
            dst[written + wsum[w] + in_warp] = s;
        written += wsum[kSlotThreads / 32];
        __syncthreads();
    }
}

} // namespace
} // namespace idx

using namespace idx;

extern "C" idx_status idx_topk(const float *logits, int64_t ld, int rows, const int32_t *lengths,
                               int k, int32_t *out_idx, int64_t ld_out, void *ws, size_t ws_bytes,
                               idx_stream_t stream)
{
    (void)ws;
    (void)ws_bytes;
    if (rows < 0 || k < 0 || ld < 0 || ld_out < k)
        return IDX_ERR_INVALID_ARG;
    if (rows == 0 || k == 0)
        return IDX_OK;
    if (!logits || !lengths || !out_idx || ld <= 0)
        return IDX_ERR_INVALID_ARG;
    const int nsm = sm_count();
    // cluster size: slice of the widest possible row within ~96 KB, and enough
    // CTAs to cover the machine twice
    int C = 1;
    const long long width = ld;
    while (C < kMaxCluster && (width + C - 1) / C * 4 > 96 * 1024)
        C <<= 1;
    while (C < kMaxCluster && (long long)rows * C < 2LL * nsm &&
           (width + 2 * C - 1) / (2 * C) >= 256)
        C <<= 1;
    const long long slice = (width + C - 1) / C;
    const size_t smem = sizeof(TopkShared) + (size_t)slice * 4;
    if (smem > 227 * 1024)
        return IDX_ERR_UNSUPPORTED;
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && C > 8)
        e = cudaFuncSetAttribute(topk_cluster_kernel,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess)
        return IDX_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * C));
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel, logits, ld, rows, lengths, k, out_idx,
                           ld_out, (int)slice);
    return launch_status(e);
}

extern "C" idx_status idx_apply_candidate_mask(float *logits, int64_t ld, int rows, int width,
                                               const int32_t *row_ks, const int32_t *row_ke,
                                               const int32_t *candidate_blocks,
                                               int64_t cand_stride, int num_cand, int block_size,
                                               int row_repeat, idx_stream_t stream)
{
    if (rows < 0 || width < 0 || ld < width || num_cand < 0 || block_size <= 0 ||
        row_repeat <= 0 || cand_stride < num_cand)
        return IDX_ERR_INVALID_ARG;
    if (rows == 0 || width == 0)
        return IDX_OK;
    if (!logits || !row_ke || (num_cand > 0 && !candidate_blocks))
        return IDX_ERR_INVALID_ARG;
    const int nblk = (width + block_size - 1) / block_size;
    const int words = (nblk + 31) / 32;
    const size_t smem = (size_t)words * 4;
    if (smem > 227 * 1024)
        return IDX_ERR_UNSUPPORTED;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(candidate_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return IDX_ERR_CUDA;
    const int cols = (int)std::min<long long>(64, (width + 4095) / 4096);
    dim3 grid(rows, cols < 1 ? 1 : cols);
    candidate_mask_kernel<<<grid, 256, smem, (cudaStream_t)stream>>>(
        logits, ld, rows, width, row_ks, row_ke, candidate_blocks, cand_stride, num_cand,
        block_size, row_repeat, words);
    return launch_status(cudaGetLastError());
}

extern "C" idx_status idx_topk_to_ragged_slots(const int32_t *topk, int64_t ld, int rows, int k,
                                               const int32_t *row_to_seq, int next_n,
                                               const int32_t *block_table, int64_t bt_stride,
                                               int max_blocks, int page_size, int num_pages,
                                               int32_t *slots, int32_t *indptr, int32_t *lens,
                                               idx_stream_t stream)
{
    if (rows < 0 || k < 0 || ld < k || page_size <= 0 || max_blocks < 0 || num_pages < 0 ||
        bt_stride < max_blocks || (!row_to_seq && next_n <= 0))
        return IDX_ERR_INVALID_ARG;
    if (!indptr)
        return IDX_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (rows == 0)
        return launch_status(cudaMemsetAsync(indptr, 0, sizeof(int32_t), s));
    if (!lens || (k > 0 && (!topk || !slots || !block_table)))
        return IDX_ERR_INVALID_ARG;
    unsigned int *status = device_status_ptr();
    if (!status)
        return IDX_ERR_CUDA;
    slot_count_kernel<<<rows, kSlotThreads, 0, s>>>(topk, ld, rows, k, row_to_seq, next_n,
                                                    block_table, bt_stride, max_blocks,
                                                    page_size, num_pages, lens, status);
    indptr_scan_kernel<<<1, 1024, 0, s>>>(lens, rows, indptr);
    slot_write_kernel<<<rows, kSlotThreads, 0, s>>>(topk, ld, rows, k, row_to_seq, next_n,
                                                    block_table, bt_stride, max_blocks,
                                                    page_size, num_pages, indptr, slots);
    return launch_status(cudaGetLastError());
}
