// idx_select.cu -- per-row top-k (radix select; chunked over the GPU for long
// rows), candidate mask and
// top-k -> ragged slot map, with their C ABI entry points.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "idx_internal.h"
#include "idx_topk.cuh"
#include "idx_topk_chunked.cuh"

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
    T::topk_kernel<<<rows, T::kThreads, smem, s>>>(logits, ld, rows, lengths, k, out, ld_out,
                                                   vec_ok);
    return launch_status(cudaGetLastError());
}

// Chunked top-k over the caller's workspace: the plan kernel, then one
// cooperative launch of the phases (see idx_topk_chunked.cuh).  Returns
// IDX_ERR_UNSUPPORTED when the device has no cooperative launch.
idx_status topk_launch_chunked(const float *logits, int64_t ld, int rows,
                               const int32_t *lengths, int k, int32_t *out, int64_t ld_out,
                               void *ws, int vec_ok, cudaStream_t s)
{
    namespace C = topk_chunked;
    static int grid_per_sm[64] = {};  // resident phase CTAs per SM, 0 = not known yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return IDX_ERR_CUDA;
    if (!grid_per_sm[dev]) {
        int coop = 0, n = 0;
        if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
            return IDX_ERR_CUDA;
        if (!coop)
            return IDX_ERR_UNSUPPORTED;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, C::phases_kernel, C::kThreads, 0) !=
                cudaSuccess ||
            n < 1)
            return IDX_ERR_CUDA;
        grid_per_sm[dev] = n;
    }
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
    a.status = status;
    C::ws_layout(ws, rows, P, &a.ws);
    const long long zero_vec4 = ((long long)rows * (2048 + 2) + 3) / 4;
    const int g_plan = (int)std::max<long long>(
        1, std::min<long long>(sm_count(), (zero_vec4 + C::kPlanThreads - 1) / C::kPlanThreads));
    C::plan_kernel<<<g_plan, C::kPlanThreads, 0, s>>>(lengths, ld, rows, a.ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return IDX_ERR_CUDA;
    // every CTA resident (the phases wait on one another), no more CTAs
    // than there can be items or rows
    const long long cap = (long long)grid_per_sm[dev] * sm_count();
    const long long want = std::max<long long>((long long)rows * P, rows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::max<long long>(1, std::min(cap, want)));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, C::phases_kernel, a);
    return launch_status(e);
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
    if (rows < 0 || k < 0 || ld < 0 || ld_out < k || ld > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    if (rows == 0 || k == 0)
        return IDX_OK;
    if (!logits || !lengths || !out_idx || ld <= 0)
        return IDX_ERR_INVALID_ARG;
    const int vec_ok = (ld % 4 == 0) && aligned16(logits);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t need = idx_topk_workspace_size(rows, ld, k);
    if (ws && need > 0 && ws_bytes >= need && aligned16(ws) && ld > topk_chunked::kCh) {
        const idx_status st =
            topk_launch_chunked(logits, ld, rows, lengths, k, out_idx, ld_out, ws, vec_ok, s);
        if (st != IDX_ERR_UNSUPPORTED)
            return st;
    }
    return topk_launch_per_row(logits, ld, rows, lengths, k, out_idx, ld_out, vec_ok, s);
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

// ------------------------------------------------ top-k without allocation
//
// idx_topk_noalloc runs the chunked top-k over one fixed array per device
// instead of caller scratch, for callers that can neither pass scratch nor
// allocate it when they call.  The array is part of this library's device
// image; its address is looked up once per device, with that device
// current, and cached.

static __device__ __align__(256) unsigned char g_topk_scratch[IDX_TOPK_NOALLOC_MAX_BYTES];

namespace {

std::mutex g_scratch_mu;
void *g_scratch_ptr[64];

idx_status topk_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return IDX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || !p)
            return IDX_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return IDX_OK;
}

} // namespace

extern "C" idx_status idx_topk_noalloc(const float *logits, int64_t ld, int rows,
                                       const int32_t *lengths, int k, int32_t *out_idx,
                                       int64_t ld_out, idx_stream_t stream)
{
    if (rows < 0 || k < 0 || ld < 0 || ld_out < k || ld > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    if (rows == 0 || k == 0)
        return IDX_OK;
    if (!logits || !lengths || !out_idx || ld <= 0)
        return IDX_ERR_INVALID_ARG;
    const size_t need = idx_topk_workspace_size(rows, ld, k);
    if (need == 0)
        return IDX_ERR_UNSUPPORTED;
    if (need > (size_t)IDX_TOPK_NOALLOC_MAX_BYTES)
        return IDX_ERR_WORKSPACE;
    void *ws = nullptr;
    const idx_status st = topk_scratch(&ws);
    if (st != IDX_OK)
        return st;
    const int vec_ok = (ld % 4 == 0) && aligned16(logits);
    return topk_launch_chunked(logits, ld, rows, lengths, k, out_idx, ld_out, ws, vec_ok,
                               (cudaStream_t)stream);
}
