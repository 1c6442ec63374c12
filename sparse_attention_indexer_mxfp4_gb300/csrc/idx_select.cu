// idx_select.cu -- per-row top-k (radix select; chunked over the GPU for long
// rows), candidate mask and
// top-k -> ragged slot map, with their C ABI entry points.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "idx_internal.h"
#include "idx_topk.cuh"
#include "idx_topk_chunked.cuh"
#include "idx_topk_cluster.cuh"
#include "idx_topk_short.cuh"
#include "idx_topk_cand.cuh"

namespace idx {
namespace {

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
    for (int i = threadIdx.x; i < words; i += blockDim.x)
        bm[i] = 0u;
    pdl_wait();  // the logits, ranges and candidates may come from the kernel before this one
    pdl_launch_dependents();
    if (r >= rows)
        return;
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

// Page geometry of the slot map: P tokens per page, shift = log2(P) when P
// is a power of two, else -1.
struct SlotGeom {
    const int32_t *bt;
    int64_t bt_stride;
    int max_blocks, P, shift, num_pages;
};

constexpr int kSlotThreads = 256;
constexpr int kSlotSteps = 8;  // entries per thread loaded before any is used

// Top-k entries j = base + i * kSlotThreads + tid (i < kSlotSteps) of one
// row, -1 past k; the loads are all issued before any is used.
__device__ __forceinline__ void row_pos(const int32_t *trow, int k, int base,
                                        int (&p)[kSlotSteps])
{
    #pragma unroll
    for (int i = 0; i < kSlotSteps; ++i) {
        const int j = base + i * kSlotThreads + (int)threadIdx.x;
        p[i] = j < k ? __ldg(trow + j) : -1;
    }
}

// Slots of positions p of one sequence whose block-table row is btrow:
// >= 0 a slot, -1 no entry, -2 an invalid position (logical page beyond
// max_blocks or page id outside the pool).
template <int N>
__device__ __forceinline__ void pos_slots(const int (&p)[N], const int32_t *btrow,
                                          const SlotGeom &g, int (&s)[N])
{
    int lp[N], pg[N];
    #pragma unroll
    for (int i = 0; i < N; ++i) {
        lp[i] = p[i] < 0 ? -1 : (g.shift >= 0 ? p[i] >> g.shift : p[i] / g.P);
        pg[i] = lp[i] >= 0 && lp[i] < g.max_blocks ? __ldg(btrow + lp[i]) : -1;
    }
    #pragma unroll
    for (int i = 0; i < N; ++i) {
        if (p[i] < 0)
            s[i] = -1;
        else if (lp[i] >= g.max_blocks || pg[i] < 0 || pg[i] >= g.num_pages)
            s[i] = -2;
        else
            s[i] = pg[i] * g.P + (p[i] - lp[i] * g.P);
    }
}

__global__ void __launch_bounds__(kSlotThreads)
    slot_count_kernel(const int32_t *__restrict__ topk, int64_t ld, int rows, int k,
                      const int32_t *__restrict__ row_to_seq, int next_n, SlotGeom g,
                      int32_t *__restrict__ lens, unsigned int *status)
{
    __shared__ uint32_t wsum[kSlotThreads / 32];
    pdl_wait();
    pdl_launch_dependents();
    const int r = blockIdx.x;
    const int b = row_to_seq ? row_to_seq[r] : r / next_n;
    const int32_t *trow = topk + (size_t)r * ld;
    uint32_t cnt = 0, bad = 0;
    const int32_t *btrow = g.bt + (size_t)b * g.bt_stride;
    for (int base = 0; base < k; base += kSlotSteps * kSlotThreads) {
        int p[kSlotSteps], sl[kSlotSteps];
        row_pos(trow, k, base, p);
        pos_slots(p, btrow, g, sl);
        #pragma unroll
        for (int i = 0; i < kSlotSteps; ++i) {
            cnt += sl[i] >= 0;
            bad += sl[i] == -2;
        }
    }
    for (int o = 16; o > 0; o >>= 1)
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if ((threadIdx.x & 31) == 0)
        wsum[threadIdx.x >> 5] = cnt;
    if (bad)
        atomicOr(status, kDevBadPage);
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int i = 0; i < kSlotThreads / 32; ++i)
            t += wsum[i];
        lens[r] = (int32_t)t;
    }
}

// Up to this many rows each write CTA adds up the earlier rows' counts
// itself (at most rows / kSlotThreads loads a thread, from L2); above it a
// scan kernel writes indptr first, since the direct sums grow as rows^2.
constexpr int kSlotDirectRows = 4096;

__global__ void __launch_bounds__(1024) indptr_scan_kernel(const int32_t *__restrict__ lens, int rows,
                                                           int32_t *__restrict__ indptr)
{
    __shared__ int32_t wsum[32];
    __shared__ int32_t carry;
    pdl_wait();
    pdl_launch_dependents();
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

// Ordered write of one row's valid slots.  The row's offset is indptr[r]
// when the scan kernel ran (scanned != 0); otherwise it is the sum of the
// earlier rows' counts, which the CTA adds up itself and publishes as
// indptr[r + 1] (CTA 0 also writes indptr[0] = 0).  Entry order is (step i,
// warp, lane); a ballot gives each lane its rank inside the warp and step,
// and warp 0 scans the (step, warp) counts once per batch of kSlotSteps
// steps.
__global__ void __launch_bounds__(kSlotThreads)
    slot_write_kernel(const int32_t *__restrict__ topk, int64_t ld, int rows, int k,
                      const int32_t *__restrict__ row_to_seq, int next_n, SlotGeom g,
                      const int32_t *__restrict__ lens, int32_t *__restrict__ indptr,
                      int scanned, int32_t *__restrict__ slots)
{
    constexpr int NW = kSlotThreads / 32;
    static_assert(kSlotSteps * NW == 64, "warp 0 scans 64 (step, warp) counts");
    __shared__ uint32_t tab[kSlotSteps * NW + 1];
    __shared__ uint32_t red[NW];
    pdl_wait();
    pdl_launch_dependents();
    const int r = blockIdx.x;
    const int b = row_to_seq ? row_to_seq[r] : r / next_n;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    const int32_t *trow = topk + (size_t)r * ld;
    // the first batch's loads go out before the offset is summed
    const int32_t *btrow = g.bt + (size_t)b * g.bt_stride;
    int p[kSlotSteps], sl[kSlotSteps];
    row_pos(trow, k, 0, p);
    pos_slots(p, btrow, g, sl);
    uint32_t off = 0;
    if (scanned) {
        off = (uint32_t)indptr[r];
    } else {
        uint32_t part = 0;
        for (int i = threadIdx.x; i < r; i += kSlotThreads)
            part += (uint32_t)lens[i];
        for (int o = 16; o > 0; o >>= 1)
            part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0)
            red[w] = part;
        __syncthreads();
        for (int i = 0; i < NW; ++i)
            off += red[i];
        if (threadIdx.x == 0) {
            indptr[r + 1] = (int32_t)(off + (uint32_t)lens[r]);
            if (r == 0)
                indptr[0] = 0;
        }
    }
    int32_t *dst = slots + off;
    uint32_t written = 0;
    for (int base = 0; base < k; base += kSlotSteps * kSlotThreads) {
        if (base > 0) {
            row_pos(trow, k, base, p);
            pos_slots(p, btrow, g, sl);
        }
        uint32_t ball[kSlotSteps];
        #pragma unroll
        for (int i = 0; i < kSlotSteps; ++i) {
            ball[i] = __ballot_sync(0xffffffffu, sl[i] >= 0);
            if (lane == i)
                tab[i * NW + w] = __popc(ball[i]);
        }
        __syncthreads();
        if (w == 0) {
            const uint32_t a0 = tab[2 * lane], a1 = tab[2 * lane + 1];
            uint32_t x = a0 + a1;
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t n = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o)
                    x += n;
            }
            const uint32_t ex = x - (a0 + a1);
            tab[2 * lane] = ex;
            tab[2 * lane + 1] = ex + a0;
            if (lane == 31)
                tab[kSlotSteps * NW] = x;
        }
        __syncthreads();
        #pragma unroll
        for (int i = 0; i < kSlotSteps; ++i)
            if (sl[i] >= 0)
                dst[written + tab[i * NW + w] + __popc(ball[i] & lt)] = sl[i];
        written += tab[kSlotSteps * NW];
        __syncthreads();
    }
}

// Slot map in one launch, for the row counts of a decode step: one
// thread-block cluster of C CTAs, CTA q taking rows [q R, q R + R).  Each CTA
// stages its rows' block-table rows in shared memory, forms its rows' slots
// (at most kScPairs per thread, in registers), counts the valid ones per
// (row, step, warp) and scans them per row; after a cluster barrier each CTA
// adds up the lower ranks' totals through distributed shared memory for its
// first offset, then writes its rows' lens, indptr and slots in entry order.
// A second barrier, arrived at once the totals are read and waited on at
// the end, keeps every CTA's shared memory alive until the others are done
// with it.  Entry e of a row is held by thread e % 1024 at step e / 1024;
// pair u of a thread is (row u / E, step u % E).
constexpr int kScThreads = 1024;
constexpr int kScWarps = kScThreads / 32;
constexpr int kScPairs = 4;            // (row, step) pairs per CTA
constexpr int kScMaxBt = 32768;        // staged block-table words per CTA

struct ScShared {
    uint32_t tab[kScPairs * kScWarps];  // valid slots per (pair, warp), then offsets
    uint32_t rowcnt[kScPairs];
    uint32_t rowoff[kScPairs];  // offset of each row within the CTA's rows
    uint32_t total;             // the CTA's valid slots (read by higher ranks)
    uint32_t base;              // the lower ranks' valid slots
};

__global__ void __launch_bounds__(kScThreads, 1)
    slot_cluster_kernel(const int32_t *__restrict__ topk, int64_t ld, int rows, int k,
                        const int32_t *__restrict__ row_to_seq, int next_n, SlotGeom g, int R,
                        int32_t *__restrict__ slots, int32_t *__restrict__ indptr,
                        int32_t *__restrict__ lens, unsigned int *status)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    ScShared &sh = *reinterpret_cast<ScShared *>(dsm);
    int32_t *sbt = reinterpret_cast<int32_t *>(dsm + sizeof(ScShared));  // [row][max_blocks]
    cooperative_groups::cluster_group cl = cooperative_groups::this_cluster();
    const int q = (int)cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int E = (k + kScThreads - 1) / kScThreads;
    const int r0 = q * R, nr = max(0, min(R, rows - r0));
    const int npair = nr * E;
    pdl_wait();  // the top-k rows may come from the kernel before this one
    pdl_launch_dependents();
    int pos[kScPairs];
    #pragma unroll
    for (int u = 0; u < kScPairs; ++u) {
        const int j = u / E, e = (u - j * E) * kScThreads + tid;
        pos[u] = u < npair && e < k ? __ldg(topk + (size_t)(r0 + j) * ld + e) : -1;
    }
    // block-table rows of the CTA's rows, while the top-k entries are in flight
    for (int j = 0; j < nr; ++j) {
        const int b = row_to_seq ? __ldg(row_to_seq + r0 + j) : (r0 + j) / next_n;
        const int32_t *btrow = g.bt + (size_t)b * g.bt_stride;
        for (int i = tid; i < g.max_blocks; i += kScThreads)
            sbt[j * g.max_blocks + i] = __ldg(btrow + i);
    }
    __syncthreads();
    int sl[kScPairs];
    uint32_t bad = 0;
    #pragma unroll
    for (int u = 0; u < kScPairs; ++u) {
        const int j = u / E;
        sl[u] = -1;
        if (pos[u] >= 0) {
            const int lp = g.shift >= 0 ? pos[u] >> g.shift : pos[u] / g.P;
            const int pg = lp < g.max_blocks ? sbt[j * g.max_blocks + lp] : -1;
            if (lp >= g.max_blocks || pg < 0 || pg >= g.num_pages)
                bad = 1;
            else
                sl[u] = pg * g.P + (pos[u] - lp * g.P);
        }
        const uint32_t ball = __ballot_sync(0xffffffffu, sl[u] >= 0);
        if (lane == 0 && u < npair)
            sh.tab[u * kScWarps + w] = __popc(ball);
    }
    if (bad)
        atomicOr(status, kDevBadPage);
    __syncthreads();
    // per row: exclusive offsets of its (step, warp) counts in that order
    // (lane l holds entries l E .. l E + E - 1, E <= 4) and the row's count
    if (w < nr) {
        uint32_t *t = sh.tab + w * E * kScWarps;
        uint32_t v[kScPairs], sum = 0;
        #pragma unroll
        for (int e = 0; e < kScPairs; ++e) {
            v[e] = e < E ? t[lane * E + e] : 0u;
            sum += v[e];
        }
        uint32_t tot;
        uint32_t run = topk_detail::warp_excl(sum, lane, &tot);
        #pragma unroll
        for (int e = 0; e < kScPairs; ++e) {
            if (e < E)
                t[lane * E + e] = run;
            run += v[e];
        }
        if (lane == 0)
            sh.rowcnt[w] = tot;
    }
    __syncthreads();
    if (w == 0) {
        const uint32_t c = lane < nr ? sh.rowcnt[lane] : 0u;
        uint32_t tot;
        const uint32_t ex = topk_detail::warp_excl(c, lane, &tot);
        if (lane < nr)
            sh.rowoff[lane] = ex;
        if (lane == 0)
            sh.total = tot;
    }
    cl.sync();  // every CTA's total is published
    if (w == 0) {
        uint32_t v = lane < q ? *cl.map_shared_rank(&sh.total, lane) : 0u;
        v = __reduce_add_sync(0xffffffffu, v);
        if (lane == 0)
            sh.base = v;
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");  // done reading others
    __syncthreads();
    const uint32_t base = sh.base;
    if (tid < nr) {
        lens[r0 + tid] = (int32_t)sh.rowcnt[tid];
        indptr[r0 + tid + 1] = (int32_t)(base + sh.rowoff[tid] + sh.rowcnt[tid]);
    }
    if (q == 0 && tid == 0)
        indptr[0] = 0;
    const uint32_t lt = (1u << lane) - 1u;
    #pragma unroll
    for (int u = 0; u < kScPairs; ++u) {
        const uint32_t ball = __ballot_sync(0xffffffffu, sl[u] >= 0);
        if (sl[u] >= 0)
            slots[base + sh.rowoff[u / E] + sh.tab[u * kScWarps + w] + __popc(ball & lt)] = sl[u];
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ top-k

idx_status topk_launch_per_row(const float *logits, int64_t ld, int rows,
                               const int32_t *lengths, int k, int32_t *out, int64_t ld_out,
                               int vec_ok, cudaStream_t s)
{
    namespace T = topk_detail;
    const size_t smem = sizeof(T::Shared);
    static int configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return IDX_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(T::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return IDX_ERR_CUDA;
        configured[dev] = 1;
    }
    return launch_status(launch_pdl(T::topk_kernel, dim3(rows), dim3(T::kThreads), smem, s,
                                    logits, ld, rows, lengths, k, out, ld_out, vec_ok));
}

// Rows of at most 8192 keys: one 256-thread CTA per row, keys in registers.
idx_status topk_launch_short(const float *logits, int64_t ld, int rows, const int32_t *lengths,
                             int k, int32_t *out, int64_t ld_out, int vec_ok, cudaStream_t s)
{
    namespace T = topk_short;
    return launch_status(launch_pdl(T::topk_short_kernel, dim3(rows), dim3(T::kThreads), 0, s,
                                    logits, ld, rows, lengths, k, out, ld_out, vec_ok));
}

// Rows of up to 262144 keys: one cluster of ceil(ld / 32768) CTAs per row,
// when those CTAs (one per SM) fit the GPU in one wave: the clusters run
// side by side and every row ends after one cluster's time.  More rows than
// that are spread better over the GPU by the chunked path.
// IDX_ERR_UNSUPPORTED when the call is outside that range or no such
// cluster can be resident on the device.
idx_status topk_launch_cluster(const float *logits, int64_t ld, int rows, const int32_t *lengths,
                               int k, int32_t *out, int64_t ld_out, int vec_ok, cudaStream_t s,
                               const SlotCount *sc = nullptr)
{
    namespace T = topk_cluster;
    const int C = (int)((ld + T::kChunk - 1) / T::kChunk);
    if (C < 1 || C > T::kMaxCluster || (long long)rows * C > sm_count())
        return IDX_ERR_UNSUPPORTED;
    const size_t smem = sizeof(T::Shared);
    static int configured[64] = {};
    static int resident[64][T::kMaxCluster + 1] = {};  // 0 unknown, 1 yes, -1 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return IDX_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(T::topk_cluster_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return IDX_ERR_CUDA;
        configured[dev] = 1;
    }
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * C));
    cfg.blockDim = dim3(T::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!resident[dev][C]) {
        int n = 0;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, T::topk_cluster_kernel, &cfg);
        if (e != cudaSuccess)
            (void)cudaGetLastError();
        resident[dev][C] = e == cudaSuccess && n > 0 ? 1 : -1;
    }
    if (resident[dev][C] < 0)
        return IDX_ERR_UNSUPPORTED;
    cfg.numAttrs = 2;  // launched programmatically after the kernel before it
    SlotCount none = {};
    return launch_status(cudaLaunchKernelEx(&cfg, T::topk_cluster_kernel, logits, ld, rows,
                                            lengths, k, out, ld_out, vec_ok, sc ? *sc : none));
}

} // namespace

// Resident phase CTAs per SM of the chunked top-k on the current device
// (0 on error, -1 without cooperative launch).
static int chunked_grid_per_sm()
{
    namespace C = topk_chunked;
    static int grid_per_sm[64] = {};  // 0 = not known yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    if (!grid_per_sm[dev]) {
        int coop = 0, n = 0;
        if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
            return 0;
        if (!coop)
            return -1;
        if (cudaFuncSetAttribute(C::phases_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kPhaseDynSmem) != cudaSuccess)
            return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, C::phases_kernel, C::kThreads,
                                                          C::kPhaseDynSmem) != cudaSuccess ||
            n < 1)
            return 0;
        grid_per_sm[dev] = n;
    }
    return grid_per_sm[dev];
}

// The chunked top-k's plan kernel: clears the row histograms and counters
// (and, with zero_cvalid, the per-chunk valid counts) and lists the live
// chunks.  IDX_ERR_UNSUPPORTED without cooperative launch.
idx_status topk_chunked_plan(const int32_t *lengths, int64_t ld, int rows, void *ws,
                             int zero_cvalid, cudaStream_t s)
{
    namespace C = topk_chunked;
    const int g = chunked_grid_per_sm();
    if (g < 0)
        return IDX_ERR_UNSUPPORTED;
    if (g == 0)
        return IDX_ERR_CUDA;
    const int P = (int)((ld + C::kCh - 1) / C::kCh);
    C::Ws w;
    C::ws_layout(ws, rows, P, &w);
    const long long zero_vec4 = ((long long)rows * (2048 + 2) + 3) / 4;
    const int g_plan = (int)std::max<long long>(
        1, std::min<long long>(sm_count(), (zero_vec4 + C::kPlanThreads - 1) / C::kPlanThreads));
    return launch_status(launch_pdl(C::plan_kernel, dim3(g_plan), dim3(C::kPlanThreads), 0, s,
                                    lengths, ld, rows, P, w, zero_cvalid));
}

// The chunked top-k's phases (one cooperative launch; every CTA resident).
// hist_done: the row histograms and the valid counts were written by the
// kernel before (the logits kernel's histogram variant), so the phases start
// at the filter.
idx_status topk_chunked_phases(const float *logits, int64_t ld, int rows, const int32_t *lengths,
                               int k, int32_t *out, int64_t ld_out, void *ws, int vec_ok,
                               int hist_done, cudaStream_t s)
{
    namespace C = topk_chunked;
    const int g = chunked_grid_per_sm();
    if (g < 0)
        return IDX_ERR_UNSUPPORTED;
    if (g == 0)
        return IDX_ERR_CUDA;
    unsigned int *status = device_status_ptr();
    if (!status)
        return IDX_ERR_CUDA;
    const int P = (int)((ld + C::kCh - 1) / C::kCh);
    C::PhaseArgs a;
    a.logits = logits;
    a.ld = ld;
    a.lengths = lengths;
    a.R = rows;
    a.P = P;
    a.k = k;
    a.out = out;
    a.ld_out = ld_out;
    a.vec_ok = vec_ok;
    a.hist_done = hist_done;
    a.status = status;
    C::ws_layout(ws, rows, P, &a.ws);
    // every CTA resident (the phases wait on one another), no more CTAs
    // than there can be items or rows
    const long long cap = (long long)g * sm_count();
    const long long want = std::max<long long>((long long)rows * P, rows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::max<long long>(1, std::min(cap, want)));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kPhaseDynSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_status(cudaLaunchKernelEx(&cfg, C::phases_kernel, a));
}

// Where a chunked top-k over (rows, ld) keeps its row histograms, valid
// counts and per-chunk valid counts inside ws; returns the chunks per row.
int topk_chunked_counts(void *ws, int rows, int64_t ld, uint32_t **hist, uint32_t **valid,
                        uint32_t **cvalid)
{
    namespace C = topk_chunked;
    const int P = (int)((ld + C::kCh - 1) / C::kCh);
    C::Ws w;
    C::ws_layout(ws, rows, P, &w);
    *hist = w.hist;
    *valid = w.valid;
    *cvalid = w.cvalid;
    return P;
}

// Whether idx_topk takes the chunked path for these arguments.
bool topk_takes_chunked(const float *logits, int64_t ld, int rows, int k, const void *ws,
                        size_t ws_bytes)
{
    const size_t need = idx_topk_workspace_size(rows, ld, k);
    (void)logits;
    return ws && need > 0 && ws_bytes >= need && aligned16(ws) && ld > topk_chunked::kCh &&
           chunked_grid_per_sm() > 0;
}

namespace {

// Chunked top-k over the caller's workspace: the plan kernel, then one
// cooperative launch of the phases (see idx_topk_chunked.cuh).  Returns
// IDX_ERR_UNSUPPORTED when the device has no cooperative launch.
idx_status topk_launch_chunked(const float *logits, int64_t ld, int rows,
                               const int32_t *lengths, int k, int32_t *out, int64_t ld_out,
                               void *ws, int vec_ok, cudaStream_t s)
{
    const idx_status st = topk_chunked_plan(lengths, ld, rows, ws, 0, s);
    if (st != IDX_OK)
        return st;
    return topk_chunked_phases(logits, ld, rows, lengths, k, out, ld_out, ws, vec_ok, 0, s);
}

} // namespace
} // namespace idx

using namespace idx;

extern "C" size_t idx_topk_workspace_size(int rows, int64_t ld, int k)
{
    (void)k;
    namespace C = idx::topk_chunked;
    if (rows <= 0 || ld <= 0 || ld > INT32_MAX)
        return 0;
    const int64_t P = (ld + C::kCh - 1) / C::kCh;
    if (P > C::kMaxChunks || (int64_t)rows * P > INT32_MAX)
        return 0;
    return C::ws_bytes(rows, (int)P);
}

extern "C" idx_status idx_topk(const float *logits, int64_t ld, int rows, const int32_t *lengths,
                               int k, int32_t *out_idx, int64_t ld_out, void *ws, size_t ws_bytes,
                               idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_topk");
    if (rows < 0 || k < 0 || ld < 0 || ld_out < k || ld > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    if (rows == 0 || k == 0)
        return IDX_OK;
    if (!logits || !lengths || !out_idx || ld <= 0)
        return IDX_ERR_INVALID_ARG;
    const int vec_ok = (ld % 4 == 0) && aligned16(logits);
    cudaStream_t s = (cudaStream_t)stream;
    if (ld <= topk_short::kMaxLen)
        return topk_launch_short(logits, ld, rows, lengths, k, out_idx, ld_out, vec_ok, s);
    if (ld <= topk_cluster::kMaxLen) {
        const idx_status st =
            topk_launch_cluster(logits, ld, rows, lengths, k, out_idx, ld_out, vec_ok, s);
        if (st != IDX_ERR_UNSUPPORTED)
            return st;
    }
    const size_t need = idx_topk_workspace_size(rows, ld, k);
    if (ws && need > 0 && ws_bytes >= need && aligned16(ws) && ld > topk_chunked::kCh) {
        const idx_status st =
            topk_launch_chunked(logits, ld, rows, lengths, k, out_idx, ld_out, ws, vec_ok, s);
        if (st != IDX_ERR_UNSUPPORTED)
            return st;
    }
    return topk_launch_per_row(logits, ld, rows, lengths, k, out_idx, ld_out, vec_ok, s);
}

extern "C" idx_status idx_topk_candidates(const float *logits, int64_t ld, int rows,
                                          const int32_t *lengths, const int32_t *row_ks,
                                          const int32_t *candidate_blocks, int64_t cand_stride,
                                          int num_cand, int block_size, int row_repeat, int k,
                                          int32_t *out_idx, int64_t ld_out, idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_topk_candidates");
    namespace T = idx::topk_cand;
    if (rows < 0 || k < 0 || ld < 0 || ld_out < k || ld > INT32_MAX || num_cand < 0 ||
        block_size <= 0 || row_repeat <= 0 || cand_stride < num_cand)
        return IDX_ERR_INVALID_ARG;
    if (rows == 0 || k == 0)
        return IDX_OK;
    if (!logits || !lengths || !out_idx || (num_cand > 0 && !candidate_blocks))
        return IDX_ERR_INVALID_ARG;
    if (num_cand > T::kMaxIds || (long long)num_cand * block_size > T::kMaxKeys)
        return IDX_ERR_UNSUPPORTED;
    const int vec4 = ld % 4 == 0 && block_size % 4 == 0 && aligned16(logits);
    // register runs per thread: four up to 8192 candidate keys, else eight
    const bool small = (long long)num_cand * block_size <= 4LL * T::kThreads * T::kStepsSmall;
    auto kern = small ? T::topk_cand_kernel<T::kStepsSmall> : T::topk_cand_kernel<T::kStepsLarge>;
    return launch_status(launch_pdl(kern, dim3(rows), dim3(T::kThreads), 0, (cudaStream_t)stream,
                                    logits, ld, rows, lengths, row_ks, candidate_blocks,
                                    cand_stride, num_cand, block_size, row_repeat, k, out_idx,
                                    ld_out, vec4));
}

extern "C" idx_status idx_apply_candidate_mask(float *logits, int64_t ld, int rows, int width,
                                               const int32_t *row_ks, const int32_t *row_ke,
                                               const int32_t *candidate_blocks,
                                               int64_t cand_stride, int num_cand, int block_size,
                                               int row_repeat, idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_apply_candidate_mask");
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
    return launch_status(launch_pdl(candidate_mask_kernel, grid, dim3(256), smem,
                                    (cudaStream_t)stream, logits, ld, rows, width, row_ks, row_ke,
                                    candidate_blocks, cand_stride, num_cand, block_size,
                                    row_repeat, words));
}

namespace idx {
namespace {

// The one-launch slot map, when its cluster holds the call: at most 4 (row,
// 1024-entry step) pairs and 32768 staged block-table words per CTA, in
// clusters of 16 CTAs where the device can hold them (else 8).  Past that
// the count and write kernels, which spread the rows over the GPU, measured
// faster (64 rows of 2048 entries: 7.6 us a step for the cluster at 8 pairs
// a CTA against 6.0 us; 32 rows: 4.0 us against 6.2 us).
// IDX_ERR_UNSUPPORTED otherwise.
// Largest slot_cluster_kernel cluster the current device holds (16, else
// 8; -1 none; 0 when the device query fails), with cfg's shared memory,
// block and attributes set up for it.
int slot_cluster_max(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&attr)[2])
{
    static int cmax[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    const size_t smem_max = sizeof(ScShared) + (size_t)kScMaxBt * 4;
    cfg.blockDim = dim3(kScThreads);
    cfg.dynamicSmemBytes = smem_max;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!cmax[dev]) {
        if (cudaFuncSetAttribute(slot_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_max) != cudaSuccess)
            return 0;
        if (cudaFuncSetAttribute(slot_cluster_kernel,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            (void)cudaGetLastError();
        cmax[dev] = -1;
        for (int C : {16, 8}) {
            attr[0].val.clusterDim.x = (unsigned)C;
            cfg.gridDim = dim3((unsigned)C);
            int n = 0;
            const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, slot_cluster_kernel, &cfg);
            if (e != cudaSuccess)
                (void)cudaGetLastError();
            if (e == cudaSuccess && n > 0) {
                cmax[dev] = C;
                break;
            }
        }
    }
    return cmax[dev];
}

// Rows per CTA of the one-launch slot map for this call: 0 when it does not
// take the call (more than kScPairs (row, step) pairs or kScMaxBt staged
// block-table words a CTA, or no such cluster on the device), -1 when the
// device query fails.
int slot_cluster_rows(int rows, int k, int max_blocks, cudaLaunchConfig_t &cfg,
                      cudaLaunchAttribute (&attr)[2])
{
    const int cmax = slot_cluster_max(cfg, attr);
    if (cmax == 0)
        return -1;
    if (cmax < 0 || k < 1)
        return 0;
    const int E = (k + kScThreads - 1) / kScThreads;
    const int R = (rows + cmax - 1) / cmax;
    return R * E > kScPairs || (long long)R * max_blocks > kScMaxBt ? 0 : R;
}

// The one-launch slot map; IDX_ERR_UNSUPPORTED where it does not take the
// call (slot_cluster_rows).
idx_status slots_launch_cluster(const int32_t *topk, int64_t ld, int rows, int k,
                                const int32_t *row_to_seq, int next_n, const SlotGeom &g,
                                int32_t *slots, int32_t *indptr, int32_t *lens,
                                unsigned int *status, cudaStream_t s)
{
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    const int R = slot_cluster_rows(rows, k, g.max_blocks, cfg, attr);
    if (R < 0)
        return IDX_ERR_CUDA;
    if (R == 0)
        return IDX_ERR_UNSUPPORTED;
    const int C = (rows + R - 1) / R;
    attr[0].val.clusterDim.x = (unsigned)C;
    cfg.gridDim = dim3((unsigned)C);
    cfg.dynamicSmemBytes = sizeof(ScShared) + (size_t)R * g.max_blocks * 4;
    cfg.stream = s;
    cfg.numAttrs = 2;  // launched programmatically after the kernel before it
    return launch_status(cudaLaunchKernelEx(&cfg, slot_cluster_kernel, topk, ld, rows, k,
                                            row_to_seq, next_n, g, R, slots, indptr, lens,
                                            status));
}

} // namespace
} // namespace idx

namespace idx {
namespace {

// Checks and page geometry of a slot-map call (idx_topk_to_ragged_slots).
idx_status slot_args(int64_t ld, int rows, int k, const int32_t *row_to_seq, int next_n,
                     const int32_t *block_table, int64_t bt_stride, int max_blocks,
                     int page_size, int num_pages, const int32_t *topk, int32_t *slots,
                     int32_t *indptr, int32_t *lens, SlotGeom *g)
{
    if (rows < 0 || k < 0 || ld < k || page_size <= 0 || max_blocks < 0 || num_pages < 0 ||
        bt_stride < max_blocks || (!row_to_seq && next_n <= 0))
        return IDX_ERR_INVALID_ARG;
    if (!indptr)
        return IDX_ERR_INVALID_ARG;
    if (rows > 0 && (!lens || (k > 0 && (!topk || !slots || !block_table))))
        return IDX_ERR_INVALID_ARG;
    g->bt = block_table;
    g->bt_stride = bt_stride;
    g->max_blocks = max_blocks;
    g->P = page_size;
    g->shift = -1;
    for (int i = 0; i < 31; ++i)
        if ((1 << i) == page_size)
            g->shift = i;
    g->num_pages = num_pages;
    return IDX_OK;
}

// The ordered write of the slot map (with the scan kernel first above
// kSlotDirectRows rows), after lens holds every row's valid slots.
cudaError_t slots_launch_write(const int32_t *topk, int64_t ld, int rows, int k,
                               const int32_t *row_to_seq, int next_n, const SlotGeom &g,
                               int32_t *slots, int32_t *indptr, const int32_t *lens,
                               cudaStream_t s)
{
    const int scanned = rows > kSlotDirectRows;
    cudaError_t e = cudaSuccess;
    if (scanned)
        e = launch_pdl(indptr_scan_kernel, dim3(1), dim3(1024), 0, s, lens, rows, indptr);
    if (e == cudaSuccess)
        e = launch_pdl(slot_write_kernel, dim3(rows), dim3(kSlotThreads), 0, s, topk, ld, rows, k,
                       row_to_seq, next_n, g, lens, indptr, scanned, slots);
    return e;
}

} // namespace
} // namespace idx

extern "C" idx_status idx_topk_to_ragged_slots(const int32_t *topk, int64_t ld, int rows, int k,
                                               const int32_t *row_to_seq, int next_n,
                                               const int32_t *block_table, int64_t bt_stride,
                                               int max_blocks, int page_size, int num_pages,
                                               int32_t *slots, int32_t *indptr, int32_t *lens,
                                               idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_topk_to_ragged_slots");
    SlotGeom g;
    const idx_status st0 = slot_args(ld, rows, k, row_to_seq, next_n, block_table, bt_stride,
                                     max_blocks, page_size, num_pages, topk, slots, indptr, lens,
                                     &g);
    if (st0 != IDX_OK)
        return st0;
    cudaStream_t s = (cudaStream_t)stream;
    if (rows == 0)
        return launch_status(cudaMemsetAsync(indptr, 0, sizeof(int32_t), s));
    unsigned int *status = device_status_ptr();
    if (!status)
        return IDX_ERR_CUDA;
    {
        const idx_status st = slots_launch_cluster(topk, ld, rows, k, row_to_seq, next_n, g,
                                                   slots, indptr, lens, status, s);
        if (st != IDX_ERR_UNSUPPORTED)
            return st;
    }
    cudaError_t e = launch_pdl(slot_count_kernel, dim3(rows), dim3(kSlotThreads), 0, s, topk, ld,
                               rows, k, row_to_seq, next_n, g, lens, status);
    if (e == cudaSuccess)
        e = slots_launch_write(topk, ld, rows, k, row_to_seq, next_n, g, slots, indptr,
                               (const int32_t *)lens, s);
    return launch_status(e);
}

extern "C" idx_status idx_topk_ragged_slots(const float *logits, int64_t ld, int rows,
                                            const int32_t *lengths, int k, int32_t *out_idx,
                                            int64_t ld_out, void *ws, size_t ws_bytes,
                                            const int32_t *row_to_seq, int next_n,
                                            const int32_t *block_table, int64_t bt_stride,
                                            int max_blocks, int page_size, int num_pages,
                                            int32_t *slots, int32_t *indptr, int32_t *lens,
                                            idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_topk_ragged_slots");
    if (rows < 0 || k < 0 || ld < 0 || ld_out < k || ld > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    if (rows > 0 && k > 0 && (!logits || !lengths || !out_idx || ld <= 0))
        return IDX_ERR_INVALID_ARG;
    SlotGeom g;
    const idx_status st0 = slot_args(ld_out, rows, k, row_to_seq, next_n, block_table, bt_stride,
                                     max_blocks, page_size, num_pages, out_idx, slots, indptr,
                                     lens, &g);
    if (st0 != IDX_OK)
        return st0;
    cudaStream_t s = (cudaStream_t)stream;
    // rows of 8193 .. 262144 keys on the cluster top-k, which counts each
    // row's valid slots as it writes the row: then only the ordered write
    // of the slot map runs (unless the one-launch slot map takes the call:
    // it is the shorter of the two)
    int sc_rows = 0;
    if (rows > 0 && k > 0) {
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = {};
        sc_rows = slot_cluster_rows(rows, k, max_blocks, cfg, attr);
        if (sc_rows < 0)
            return IDX_ERR_CUDA;
    }
    if (rows > 0 && k > 0 && sc_rows == 0 && ld > topk_short::kMaxLen &&
        ld <= topk_cluster::kMaxLen) {
        unsigned int *status = device_status_ptr();
        if (!status)
            return IDX_ERR_CUDA;
        SlotCount sc;
        sc.bt = g.bt;
        sc.bt_stride = g.bt_stride;
        sc.max_blocks = g.max_blocks;
        sc.P = g.P;
        sc.shift = g.shift;
        sc.num_pages = g.num_pages;
        sc.row_to_seq = row_to_seq;
        sc.next_n = next_n;
        sc.lens = lens;
        sc.status = status;
        const int vec_ok = (ld % 4 == 0) && aligned16(logits);
        const idx_status st = topk_launch_cluster(logits, ld, rows, lengths, k, out_idx, ld_out,
                                                  vec_ok, s, &sc);
        if (st == IDX_OK)
            return launch_status(slots_launch_write(out_idx, ld_out, rows, k, row_to_seq, next_n,
                                                    g, slots, indptr, (const int32_t *)lens, s));
        if (st != IDX_ERR_UNSUPPORTED)
            return st;
    }
    const idx_status st = idx_topk(logits, ld, rows, lengths, k, out_idx, ld_out, ws, ws_bytes,
                                   stream);
    if (st != IDX_OK)
        return st;
    return idx_topk_to_ragged_slots(out_idx, ld_out, rows, k, row_to_seq, next_n, block_table,
                                    bt_stride, max_blocks, page_size, num_pages, slots, indptr,
                                    lens, stream);
}

// ------------------------------------------------ row ends and tail fill
//
// Row ends: ke of row j of sequence b is context_lens[b] - next_n + j + 1
// (one length per sequence: each of the next_n query tokens of an MTP step
// sees the context up to itself) or context_lens[b * next_n + j] (one
// length per row), clamped to [0, width] -- the rule the paged logits
// kernel applies to its own rows (vLLM page rocm_aiter_mla_sparse,
// rocm_fp8_paged_mqa_logits_triton, ctx_per_row).  Tail fill: -inf over
// [ke, width) of every row, as the stage-1 path of rocm_fp8_paged_mqa_logits
// fills its whole workspace with -inf before scoring.

namespace idx {

__global__ void __launch_bounds__(256) row_ends_kernel(const int32_t *__restrict__ ctx,
                                                       int ctx_per_row, int rows, int next_n,
                                                       int width, int32_t *__restrict__ out)
{
    pdl_wait();  // out may still be read by the kernel before this one
    pdl_launch_dependents();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows)
        return;
    const int e = ctx_per_row ? ctx[r] : ctx[r / next_n] - next_n + r % next_n + 1;
    out[r] = min(max(e, 0), width);
}

// Grid (column blocks, rows), both strided; four columns a store where the
// row and the tail start allow it.
__global__ void __launch_bounds__(256) fill_tail_kernel(float *__restrict__ logits, int64_t ld,
                                                        int rows,
                                                        const int32_t *__restrict__ row_ends,
                                                        int width, int vec)
{
    pdl_wait();  // the logits and row ends may come from the kernel before this one
    pdl_launch_dependents();
    for (int r = blockIdx.y; r < rows; r += gridDim.y) {
        const int e = min(max(row_ends[r], 0), width);
        float *row = logits + (size_t)r * ld;
        // scalar up to a multiple of 4 (with four-column stores), else to the end
        const int e4 = vec ? min((e + 3) & ~3, width) : width;
        for (int t = e + blockIdx.x * 256 + threadIdx.x; t < e4; t += gridDim.x * 256)
            row[t] = -INFINITY;
        if (vec) {
            const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            for (int t = e4 + 4 * (blockIdx.x * 256 + threadIdx.x); t + 4 <= width;
                 t += 4 * gridDim.x * 256)
                *reinterpret_cast<float4 *>(row + t) = ninf;
            const int w4 = e4 + (width - e4) / 4 * 4;  // scalar tail past the last full quad
            for (int t = w4 + blockIdx.x * 256 + threadIdx.x; t < width; t += gridDim.x * 256)
                row[t] = -INFINITY;
        }
    }
}

} // namespace idx

extern "C" idx_status idx_row_ends(const int32_t *context_lens, int ctx_per_row, int B,
                                   int next_n, int max_model_len, int32_t *row_ends,
                                   idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_row_ends");
    if (B < 0 || next_n <= 0 || max_model_len < 0)
        return IDX_ERR_INVALID_ARG;
    const long long rows = (long long)B * next_n;
    if (rows == 0)
        return IDX_OK;
    if (!context_lens || !row_ends || rows > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    return launch_status(launch_pdl(row_ends_kernel, dim3((unsigned)((rows + 255) / 256)),
                                    dim3(256), 0, (cudaStream_t)stream, context_lens,
                                    ctx_per_row ? 1 : 0, (int)rows, next_n, max_model_len,
                                    row_ends));
}

extern "C" idx_status idx_fill_logits_tail(float *logits, int64_t ld, int rows,
                                           const int32_t *row_ends, int width,
                                           idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_fill_logits_tail");
    if (rows < 0 || width < 0 || ld < width)
        return IDX_ERR_INVALID_ARG;
    if (rows == 0 || width == 0)
        return IDX_OK;
    if (!logits || !row_ends)
        return IDX_ERR_INVALID_ARG;
    const int vec = (ld % 4 == 0) && aligned16(logits);
    const dim3 grid((unsigned)std::min(64, (width + 4 * 256 - 1) / (4 * 256)),
                    (unsigned)std::min(rows, 65535));
    return launch_status(launch_pdl(fill_tail_kernel, grid, dim3(256), 0, (cudaStream_t)stream,
                                    logits, ld, rows, row_ends, width, vec));
}

// ---------------------------------------------------- bounded-wait expiry
//
// A diagnostic that makes the library's bounded waits run out, so that a
// test can check the path every pipeline takes when a wait never completes:
// the wait returns after its limit, the device status gets IDX_DEV_TIMEOUT,
// the kernel ends, and the context stays usable.  which = 0: the mbarrier
// wait of the logits pipeline (mbar_wait) on a barrier no thread arrives
// on; which = 1: the grid barrier of the chunked top-k (grid_sync) in a
// launch of two CTAs of which only the first arrives.

namespace idx {

__device__ uint32_t g_expiry_ctrl[2];

__global__ void wait_expiry_kernel(int which, uint64_t limit_ns, unsigned *status)
{
    if (which == 0) {
        __shared__ __align__(8) uint64_t bar;
        __shared__ int abort;
        if (threadIdx.x == 0) {
            mbar_init(&bar, 1);
            abort = 0;
            fence_mbar_init();
        }
        __syncthreads();
        if (threadIdx.x == 0)
            (void)mbar_wait(&bar, 0u, &abort, status, limit_ns);
        __syncthreads();
        return;
    }
    if (blockIdx.x != 0)  // the CTA that never arrives
        return;
    __shared__ uint32_t abort_sh;
    if (threadIdx.x == 0)
        abort_sh = 0u;
    __syncthreads();
    (void)topk_chunked::grid_sync(g_expiry_ctrl, status, &abort_sh, limit_ns);
}

} // namespace idx

extern "C" idx_status idx_debug_wait_expiry(int which, uint64_t limit_ns, idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_debug_wait_expiry");
    if ((which != 0 && which != 1) || limit_ns == 0 || limit_ns > 10000000000ull)
        return IDX_ERR_INVALID_ARG;
    unsigned int *status = device_status_ptr();
    if (!status)
        return IDX_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (which == 1) {  // the barrier's arrival count starts at zero
        void *ctrl = nullptr;
        if (cudaGetSymbolAddress(&ctrl, g_expiry_ctrl) != cudaSuccess ||
            cudaMemsetAsync(ctrl, 0, sizeof(g_expiry_ctrl), s) != cudaSuccess)
            return IDX_ERR_CUDA;
    }
    wait_expiry_kernel<<<which == 0 ? 1 : 2, 128, 0, s>>>(which, limit_ns, status);
    return launch_status(cudaGetLastError());
}

// ------------------------------------------------ top-k without allocation
//
// idx_topk_noalloc runs the chunked top-k over one fixed array per device
// instead of caller scratch, for callers that can neither pass scratch nor
// allocate it when they call.  The array is part of this library's device
// image; its address is looked up with the device current and cached per
// (device, context): a new primary context after a device reset gets a new
// lookup.

static __device__ __align__(256) unsigned char g_topk_scratch[IDX_TOPK_NOALLOC_MAX_BYTES];

namespace {

std::mutex g_scratch_mu;
void *g_scratch_ptr[64];
CUcontext g_scratch_ctx[64];

// The driver's cuCtxGetCurrent, through the runtime's entry-point query (the
// library links no driver library).
CUresult (*ctx_getter())(CUcontext *)
{
    static CUresult (*fn)(CUcontext *) = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CUresult (*)(CUcontext *)>(p);
    });
    return fn;
}

idx_status topk_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return IDX_ERR_CUDA;
    auto get_ctx = ctx_getter();
    if (!get_ctx)
        return IDX_ERR_CUDA;
    // the context current on this thread (null before the runtime has bound
    // one); the cached address is valid only in the context it was taken in
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS)
        return IDX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;  // the lookup binds the device's primary context
        if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || !p)
            return IDX_ERR_CUDA;
        if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx)
            return IDX_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return IDX_OK;
}

} // namespace

extern "C" idx_status idx_topk_noalloc(const float *logits, int64_t ld, int rows,
                                       const int32_t *lengths, int k, int32_t *out_idx,
                                       int64_t ld_out, idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_topk_noalloc");
    if (rows < 0 || k < 0 || ld < 0 || ld_out < k || ld > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    if (rows == 0 || k == 0)
        return IDX_OK;
    if (!logits || !lengths || !out_idx || ld <= 0)
        return IDX_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const int vec_ok = (ld % 4 == 0) && aligned16(logits);
    if (ld <= topk_short::kMaxLen)  // rows a CTA or a cluster holds need no scratch
        return topk_launch_short(logits, ld, rows, lengths, k, out_idx, ld_out, vec_ok, s);
    if (ld <= topk_cluster::kMaxLen) {
        const idx_status st =
            topk_launch_cluster(logits, ld, rows, lengths, k, out_idx, ld_out, vec_ok, s);
        if (st != IDX_ERR_UNSUPPORTED)
            return st;
    }
    // the chunked path over the fixed array when the call fits it; otherwise
    // (too many rows for the array, rows too long for the chunked path, no
    // cooperative launch) the scratch-free kernel that streams each row
    const size_t need = idx_topk_workspace_size(rows, ld, k);
    if (need > 0 && need <= (size_t)IDX_TOPK_NOALLOC_MAX_BYTES && ld > topk_chunked::kCh) {
        void *ws = nullptr;
        const idx_status st = topk_scratch(&ws);
        if (st != IDX_OK)
            return st;
        const idx_status sc =
            topk_launch_chunked(logits, ld, rows, lengths, k, out_idx, ld_out, ws, vec_ok, s);
        if (sc != IDX_ERR_UNSUPPORTED)
            return sc;
    }
    return topk_launch_per_row(logits, ld, rows, lengths, k, out_idx, ld_out, vec_ok, s);
}
