// idx_api.cu -- C ABI entry points of the logits kernels, argument checks,
// TMA descriptor encoding and the device status word.
#include <climits>
#include <cstdio>
#include <cudaTypedefs.h>
#include <mutex>

#include "idx_internal.h"
#include "idx_logits_kernel.cuh"

namespace idx {

__device__ unsigned int g_idx_status;

namespace {

constexpr int kMaxDevices = 64;

int current_device()
{
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

PFN_cuTensorMapEncodeTiled_v12000 tma_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

} // namespace

unsigned int *device_status_ptr()
{
    static unsigned int *ptrs[kMaxDevices] = {};
    static std::mutex mu;
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_idx_status) != cudaSuccess)
            return nullptr;
        ptrs[dev] = static_cast<unsigned int *>(p);
    }
    return ptrs[dev];
}

int sm_count()
{
    static int counts[kMaxDevices] = {};
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices)
        return 1;
    if (counts[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        counts[dev] = n > 0 ? n : 1;
    }
    return counts[dev];
}

bool encode_tma_u8(CUtensorMap *map, int rank, const void *base, const uint64_t *dims,
                   const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swz)
{
    auto fn = tma_encoder();
    if (!fn)
        return false;
    cuuint64_t gdim[5], gstr[4];
    cuuint32_t bdim[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank)
            gstr[i] = strides_bytes[i];
    }
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void *>(base),
                    gdim, gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

constexpr size_t kMaxSmem = 227 * 1024;
// Units a CTA is charged for starting a row group of a paged call (see
// locate_units), for 128-key tiles: about the latency of a group start over
// the time of a tile.  256-key tiles measured best with no charge.
constexpr int kGroupCost128 = 5;
constexpr int kMaxSmemBytes = 227 * 1024;

// BM: whether this instantiation also has the block-maxima variant (dense
// walks of one- and two-row groups, the candidate source's shapes).
// nctas: the grid size, or 0 for one persistent CTA per resident slot: the
// CTAs the occupancy calculator places on an SM for this kernel and shared
// memory, times the SMs (capped at max_ctas).
template <int FMT, int H, int G, int S, int NA, int TK, bool BM>
cudaError_t launch_logits_t(const LogitsArgs &a0, const CUtensorMap &tmK, const CUtensorMap &tmQ,
                            const CUtensorMap &tmS, int nctas, long long max_ctas,
                            cudaStream_t stream)
{
    using C = LogitsCfg<FMT, H, G, S, NA, TK>;
    LogitsArgs a = a0;
    a.tile_shift = TK == 256 ? 8 : 7;
    a.group_cost = a.paged && TK == 128 ? kGroupCost128 : 0;
    size_t smem = (size_t)C::fixed_bytes() + (size_t)2 * G * a.cand_words * 4;
    // variant: 0 dense, 1 gather plan, 2 dense with block maxima, 3 dense
    // with digit-1 histograms, 4 both
    const int variant = a.plan ? 1 : (a.bmax ? 2 : 0) + (a.hist ? (a.bmax ? 2 : 3) : 0);
    decltype(&logits_kernel<FMT, H, G, S, NA, TK, false>) kern = nullptr;
    if (variant == 1)
        kern = logits_kernel<FMT, H, G, S, NA, TK, true>;
    else if (variant == 0)
        kern = logits_kernel<FMT, H, G, S, NA, TK, false>;
    else if constexpr (BM) {
        if (variant == 2)
            kern = logits_kernel<FMT, H, G, S, NA, TK, false, true>;
        else if (variant == 3)
            kern = logits_kernel<FMT, H, G, S, NA, TK, false, false, true>;
        else
            kern = logits_kernel<FMT, H, G, S, NA, TK, false, true, true>;
    }
    if (!kern)
        return cudaErrorNotSupported;
    if (a.hist)
        smem += 16 + hist_smem_bytes<G, NA>();
    if (smem > kMaxSmem)
        return cudaErrorNotSupported;
    // raise each kernel's dynamic shared memory limit once per device
    static int configured[5][kMaxDevices] = {};
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!configured[variant][dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kMaxSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured[variant][dev] = 1;
    }
    if (nctas <= 0) {
        // resident CTAs per SM for this kernel and shared memory, cached per
        // (variant, device) with the shared memory it was asked for
        static int occ[5][kMaxDevices] = {};
        static size_t occ_smem[5][kMaxDevices] = {};
        if (!occ[variant][dev] || occ_smem[variant][dev] != smem) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, smem) !=
                    cudaSuccess ||
                n < 1)
                return cudaErrorNotSupported;
            occ[variant][dev] = n;
            occ_smem[variant][dev] = smem;
        }
        const long long want = (long long)occ[variant][dev] * sm_count();
        nctas = (int)std::max<long long>(1, std::min(want, max_ctas));
    }
    return launch_pdl(kern, dim3(nctas), dim3(C::THREADS), smem, stream, a, tmK, tmQ, tmS);
}

// Shared memory the launch needs; 0 if the combination has no kernel.
template <int FMT, int H, int G, int S, int NA, int TK>
size_t logits_smem_t(int cand_words)
{
    return (size_t)LogitsCfg<FMT, H, G, S, NA, TK>::fixed_bytes() + (size_t)2 * G * cand_words * 4;
}


// Dispatch on (format, heads, rows per group) to the compiled instantiations.
cudaError_t launch_logits(int fmt, int H, int G, const LogitsArgs &a, const CUtensorMap &tmK,
                          const CUtensorMap &tmQ, const CUtensorMap &tmS, int nctas,
                          long long max_ctas, cudaStream_t s, bool *supported)
{
    *supported = true;
    if (H == 64 && fmt == kFmtFp8) {
        switch (G) {
        case 1: return launch_logits_t<kFmtFp8, 64, 1, 4, 2, 256, true>(a, tmK, tmQ, tmS, nctas, max_ctas, s);
        case 2:
            // under a gather plan, 128-key tiles: candidate blocks of 128 keys
            // then fill whole tiles and stages
            if (a.plan)
                return launch_logits_t<kFmtFp8, 64, 2, 6, 3, 128, false>(a, tmK, tmQ, tmS, nctas, max_ctas, s);
            return launch_logits_t<kFmtFp8, 64, 2, 4, 2, 256, true>(a, tmK, tmQ, tmS, nctas, max_ctas, s);
        case 4:
            if (a.bmax)
                break;  // no block-maxima variant for four-row groups
            return launch_logits_t<kFmtFp8, 64, 4, 8, 2, 128, false>(a, tmK, tmQ, tmS, nctas, max_ctas, s);
        }
    } else if (H == 64 && fmt == kFmtMxfp4) {
        switch (G) {
        case 1: return launch_logits_t<kFmtMxfp4, 64, 1, 8, 2, 256, true>(a, tmK, tmQ, tmS, nctas, max_ctas, s);
        case 2: return launch_logits_t<kFmtMxfp4, 64, 2, 12, 3, 128, true>(a, tmK, tmQ, tmS, nctas, max_ctas, s);
        }
    }
    *supported = false;
    return cudaSuccess;
}

// log2 of the keys per tile of the instantiation launch_logits picks.
int logits_tile_shift(int fmt, int G, bool plan)
{
    if (fmt == kFmtFp8)
        return G == 4 || (G == 2 && plan) ? 7 : 8;
    return G == 2 ? 7 : 8;
}

// Gather-plan geometry for a row width: box bits for 64-key boxes and a
// tile list long enough for 128-key tiles (the most tiles any instantiation
// has); the plan kernel's shared memory also holds the tile bits.
void plan_geom(int width, int *box_words, int *plan_words, int *tile_words)
{
    const int tiles = (width + kMmaM - 1) / kMmaM;
    const int boxes = (width + kHalfKeys - 1) / kHalfKeys;
    *box_words = (boxes + 31) / 32;
    *tile_words = (tiles + 31) / 32;
    *plan_words = (1 + *box_words + tiles + 3) / 4 * 4;
}

cudaError_t launch_plan(const LogitsArgs &a, int groups, int tile_words, cudaStream_t s)
{
    const size_t smem = (size_t)(a.box_words + tile_words) * 4;
    const dim3 grid(groups, a.plan_fill ? kPlanSlices : 1);  // slices only split the fill
    if (a.tile_shift == 8)
        return launch_pdl(cand_plan_kernel<8>, grid, dim3(kPlanThreads), smem, s, a);
    return launch_pdl(cand_plan_kernel<7>, grid, dim3(kPlanThreads), smem, s, a);
}

size_t logits_smem(int fmt, int H, int G, int cand_words)
{
    if (H == 64 && fmt == kFmtFp8) {
        switch (G) {
        case 1: return logits_smem_t<kFmtFp8, 64, 1, 4, 2, 256>(cand_words);
        case 2:
            return std::max(logits_smem_t<kFmtFp8, 64, 2, 4, 2, 256>(cand_words),
                            logits_smem_t<kFmtFp8, 64, 2, 6, 3, 128>(cand_words));
        case 4: return logits_smem_t<kFmtFp8, 64, 4, 8, 2, 128>(cand_words);
        }
    } else if (H == 64 && fmt == kFmtMxfp4) {
        switch (G) {
        case 1: return logits_smem_t<kFmtMxfp4, 64, 1, 8, 2, 256>(cand_words);
        case 2: return logits_smem_t<kFmtMxfp4, 64, 2, 12, 3, 128>(cand_words);
        }
    }
    return 0;
}

bool valid_fmt(idx_kv_format f)
{
    return f == IDX_KV_FP8_E4M3 || f == IDX_KV_MXFP4;
}

} // namespace
} // namespace idx

using namespace idx;

extern "C" idx_status idx_mqa_logits(const void *q, const void *q_scale, const float *weights,
                                     const void *k, const void *k_scale,
                                     const int32_t *row_ks, const int32_t *row_ke, int M,
                                     int N, int H, int D, idx_kv_format fmt, float *logits,
                                     int64_t ld_logits, void *ws, size_t ws_bytes,
                                     idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_mqa_logits");
    (void)ws;
    (void)ws_bytes;
    if (M < 0 || N < 0 || H <= 0 || D <= 0 || !valid_fmt(fmt))
        return IDX_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return IDX_OK;
    if (!q || !weights || !k || !k_scale || !row_ks || !row_ke || !logits || ld_logits < N)
        return IDX_ERR_INVALID_ARG;
    const int f = fmt == IDX_KV_FP8_E4M3 ? kFmtFp8 : kFmtMxfp4;
    if (f == kFmtMxfp4 && !q_scale)
        return IDX_ERR_INVALID_ARG;
    if (D != 128 || H != 64)
        return IDX_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(weights) ||
        (q_scale && !aligned16(q_scale)) || !aligned16(k_scale))
        return IDX_ERR_UNSUPPORTED;
    if (f == kFmtMxfp4 && N % 4 != 0)
        return IDX_ERR_UNSUPPORTED;
    const int nsm = sm_count();
    const int T = (N + kMmaM - 1) / kMmaM;  // 128-key tiles, for sizing only
    int G = 1;
    const int gmax = f == kFmtFp8 ? 4 : 2;
    for (int g = gmax; g > 1; g >>= 1)
        if (g <= M && (long long)((M + g - 1) / g) * T >= 2LL * nsm) {
            G = g;
            break;
        }
    const int rowb = f == kFmtFp8 ? D : D / 2;
    const CUtensorMapSwizzle swz =
        f == kFmtFp8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap tmK, tmQ, tmS;
    {
        // the key scales, 4 bytes per key (fp32 or four e8m0), 64 keys per box
        uint64_t dims[1] = {(uint64_t)N * 4};
        uint32_t box[1] = {(uint32_t)kHalfKeys * 4};
        if (!encode_tma_u8(&tmS, 1, k_scale, dims, nullptr, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return IDX_ERR_UNSUPPORTED;
    }
    {
        uint64_t dims[3] = {(uint64_t)rowb, (uint64_t)N, 1};
        uint64_t str[2] = {(uint64_t)rowb, (uint64_t)rowb * (uint64_t)N};
        uint32_t box[3] = {(uint32_t)rowb, (uint32_t)kHalfKeys, 1};
        if (!encode_tma_u8(&tmK, 3, k, dims, str, box, swz))
            return IDX_ERR_UNSUPPORTED;
    }
    {
        uint64_t dims[2] = {(uint64_t)rowb, (uint64_t)M * H};
        uint64_t str[1] = {(uint64_t)rowb};
        uint32_t box[2] = {(uint32_t)rowb, (uint32_t)(G * H)};
        if (!encode_tma_u8(&tmQ, 2, q, dims, str, box, swz))
            return IDX_ERR_UNSUPPORTED;
    }
    LogitsArgs a = {};
    a.paged = 0;
    a.page_shift = -1;
    a.page_size = 1;
    a.G = G;
    a.total_rows = M;
    a.num_groups = (M + G - 1) / G;
    a.H = H;
    a.q_scale = f == kFmtFp8 ? static_cast<const float *>(q_scale) : nullptr;
    a.q_sf = f == kFmtMxfp4 ? static_cast<const uint8_t *>(q_scale) : nullptr;
    a.weights = weights;
    a.kv = static_cast<const uint8_t *>(k);
    a.k_scale = f == kFmtFp8 ? static_cast<const float *>(k_scale) : nullptr;
    a.k_sf = f == kFmtMxfp4 ? static_cast<const uint8_t *>(k_scale) : nullptr;
    a.row_ks = row_ks;
    a.row_ke = row_ke;
    a.N = N;
    a.logits = logits;
    a.ld = ld_logits;
    a.width = N;
    a.status = device_status_ptr();
    if (!a.status)
        return IDX_ERR_CUDA;
    const long long units = (long long)a.num_groups * T;
    bool supported = false;
    cudaError_t e = launch_logits(f, H, G, a, tmK, tmQ, tmS, 0, units, (cudaStream_t)stream,
                                  &supported);
    if (!supported)
        return IDX_ERR_UNSUPPORTED;
    return launch_status(e);
}

// -inf over rows x [0, nb) of the block maxima, before the logits kernel
// raises them: grid (column blocks of 256, rows), both strided.
__global__ void __launch_bounds__(256) bmax_fill_kernel(float *bmax, int64_t ld, int rows, int nb)
{
    pdl_wait();
    pdl_launch_dependents();
    for (int r = blockIdx.y; r < rows; r += gridDim.y) {
        float *row = bmax + (size_t)r * ld;
        for (int j = blockIdx.x * 256 + threadIdx.x; j < nb; j += gridDim.x * 256)
            row[j] = -INFINITY;
    }
}

// Extra epilogue outputs requested with the logits: block maxima (nullable
// out) and the digit-1 histograms of a chunked top-k (nullable hist).
struct BlockMaxOut {
    float *out = nullptr;
    int64_t ld = 0;
    int block = 0;
    uint32_t *hist = nullptr, *hvalid = nullptr, *cvalid = nullptr;
    int hist_P = 0;
};

static idx_status paged_logits(bool cand_only,
    const void *q, const void *q_scale, const float *weights, const uint8_t *kv_pages,
    int64_t page_stride_bytes, int num_pages, const int32_t *block_table, int64_t bt_stride,
    const int32_t *context_lens, int ctx_per_row, const int32_t *row_ks, int B, int next_n,
    int H, int D, int page_size, idx_kv_format fmt, const int32_t *candidate_blocks,
    int64_t cand_stride, int num_cand, int cand_block, float *logits, int64_t ld_logits,
    int max_model_len, int num_ctas, void *ws, size_t ws_bytes, idx_stream_t stream,
    BlockMaxOut bm = BlockMaxOut(), bool check_only = false)
{
    if (B < 0 || next_n <= 0 || H <= 0 || D <= 0 || page_size <= 0 || num_pages < 0 ||
        max_model_len < 0 || num_ctas < 0 || !valid_fmt(fmt))
        return IDX_ERR_INVALID_ARG;
    if (B == 0 || max_model_len == 0)
        return IDX_OK;
    const int f = fmt == IDX_KV_FP8_E4M3 ? kFmtFp8 : kFmtMxfp4;
    const int max_blocks = (max_model_len + page_size - 1) / page_size;
    if (!q || !weights || !kv_pages || !block_table || !context_lens || !logits ||
        ld_logits < max_model_len || bt_stride < max_blocks || num_pages <= 0)
        return IDX_ERR_INVALID_ARG;
    if (f == kFmtMxfp4 && !q_scale)
        return IDX_ERR_INVALID_ARG;
    if (candidate_blocks && (num_cand < 0 || cand_block <= 0 || cand_stride < num_cand))
        return IDX_ERR_INVALID_ARG;
    int bm_blocks = 0;
    if (bm.out) {
        if (bm.block <= 0)
            return IDX_ERR_INVALID_ARG;
        bm_blocks = (int)(((long long)max_model_len + bm.block - 1) / bm.block);
        if (bm.ld < bm_blocks)
            return IDX_ERR_INVALID_ARG;
        if (bm.block < 32 || next_n > 2)
            return IDX_ERR_UNSUPPORTED;  // a warp's 32 keys span at most two blocks;
                                         // one- and two-row groups only
    }
    const int64_t page_bytes =
        (int64_t)page_size * (f == kFmtFp8 ? (D + 4) : (D / 2 + D / 32));
    if (page_stride_bytes < page_bytes)
        return IDX_ERR_INVALID_ARG;
    if (D != 128 || H != 64 || page_size % kHalfKeys != 0 || page_stride_bytes % 16 != 0)
        return IDX_ERR_UNSUPPORTED;
    const int G = next_n;
    if (!aligned16(q) || !aligned16(kv_pages) || !aligned16(weights) ||
        (q_scale && !aligned16(q_scale)))
        return IDX_ERR_UNSUPPORTED;
    const int rowb = f == kFmtFp8 ? D : D / 2;
    const CUtensorMapSwizzle swz =
        f == kFmtFp8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    int cand_words = 0;
    if (candidate_blocks && num_cand > 0) {
        const int nblk = (max_model_len + cand_block - 1) / cand_block;
        cand_words = (nblk + 31) / 32;
    }
    const size_t smem = logits_smem(f, H, G, cand_words);
    if (smem == 0 || smem > kMaxSmem)
        return IDX_ERR_UNSUPPORTED;
    CUtensorMap tmK, tmQ, tmS;
    {
        // each page's scale block: page_size x 4 bytes after the values
        uint64_t dims[2] = {(uint64_t)page_size * 4, (uint64_t)num_pages};
        uint64_t str[1] = {(uint64_t)page_stride_bytes};
        uint32_t box[2] = {(uint32_t)kHalfKeys * 4, 1};
        if (!encode_tma_u8(&tmS, 2, kv_pages + (size_t)page_size * rowb, dims, str, box,
                           CU_TENSOR_MAP_SWIZZLE_NONE))
            return IDX_ERR_UNSUPPORTED;
    }
    {
        uint64_t dims[3] = {(uint64_t)rowb, (uint64_t)page_size, (uint64_t)num_pages};
        uint64_t str[2] = {(uint64_t)rowb, (uint64_t)page_stride_bytes};
        uint32_t box[3] = {(uint32_t)rowb, (uint32_t)kHalfKeys, 1};
        if (!encode_tma_u8(&tmK, 3, kv_pages, dims, str, box, swz))
            return IDX_ERR_UNSUPPORTED;
    }
    {
        uint64_t dims[2] = {(uint64_t)rowb, (uint64_t)B * next_n * H};
        uint64_t str[1] = {(uint64_t)rowb};
        uint32_t box[2] = {(uint32_t)rowb, (uint32_t)(G * H)};
        if (!encode_tma_u8(&tmQ, 2, q, dims, str, box, swz))
            return IDX_ERR_UNSUPPORTED;
    }
    LogitsArgs a = {};
    a.paged = 1;
    a.G = G;
    a.total_rows = B * next_n;
    a.num_groups = B;
    a.H = H;
    a.q_scale = f == kFmtFp8 ? static_cast<const float *>(q_scale) : nullptr;
    a.q_sf = f == kFmtMxfp4 ? static_cast<const uint8_t *>(q_scale) : nullptr;
    a.weights = weights;
    a.kv = kv_pages;
    a.page_stride = page_stride_bytes;
    a.num_pages = num_pages;
    a.page_size = page_size;
    a.page_shift = -1;
    if ((page_size & (page_size - 1)) == 0)
        for (int b = 0; b < 31; ++b)
            if ((1 << b) == page_size)
                a.page_shift = b;
    a.scale_off = (int64_t)page_size * rowb;
    a.bt = block_table;
    a.bt_stride = bt_stride;
    a.max_blocks = max_blocks;
    a.ctx = context_lens;
    a.ctx_per_row = ctx_per_row ? 1 : 0;
    a.row_ks = row_ks;
    a.cand = cand_words ? candidate_blocks : nullptr;
    a.cand_stride = cand_stride;
    a.num_cand = num_cand;
    a.cand_block = cand_block;
    a.cand_shift = -1;
    for (int b = 0; b < 31; ++b)
        if ((1 << b) == cand_block)
            a.cand_shift = b;
    a.cand_words = cand_words;
    a.logits = logits;
    a.ld = ld_logits;
    a.width = max_model_len;
    a.status = device_status_ptr();
    if (!a.status)
        return IDX_ERR_CUDA;
    if (check_only)  // every host check passed; nothing is launched
        return IDX_OK;
    const int nctas = num_ctas;  // 0: from the occupancy of the kernel launched
    // gather path: with a fused candidate mask and scratch for the plan, only
    // tiles and 64-key boxes that hold a candidate key are loaded and scored
    const size_t plan_need =
        idx_paged_mqa_logits_workspace_size(B, next_n, max_model_len, a.cand ? num_cand : 0);
    const bool planned = plan_need > 0 && ws && ws_bytes >= plan_need && aligned16(ws);
    if (cand_only && !planned)
        return plan_need == 0 ? IDX_ERR_INVALID_ARG : IDX_ERR_WORKSPACE;
    a.hist = bm.hist;
    a.hvalid = bm.hvalid;
    a.cvalid = bm.cvalid;
    a.hist_P = bm.hist_P;
    if (bm.out) {
        a.bmax = bm.out;
        a.ld_bmax = bm.ld;
        a.bmax_block = bm.block;
        a.bmax_shift = -1;
        for (int b = 0; b < 31; ++b)
            if ((1 << b) == bm.block)
                a.bmax_shift = b;
        const dim3 grid(std::min((bm_blocks + 255) / 256, 64), std::min(B * next_n, 65535));
        if (launch_pdl(bmax_fill_kernel, grid, dim3(256), 0, (cudaStream_t)stream, bm.out, bm.ld,
                       B * next_n, bm_blocks) != cudaSuccess)
            return IDX_ERR_CUDA;
    }
    if (planned) {
        int tile_words = 0;
        a.plan = static_cast<uint32_t *>(ws);
        a.plan_fill = cand_only ? 0 : 1;
        plan_geom(max_model_len, &a.box_words, &a.plan_words, &tile_words);
        a.tile_shift = logits_tile_shift(f, G, true);
        if (launch_plan(a, B, tile_words, (cudaStream_t)stream) != cudaSuccess)
            return IDX_ERR_CUDA;
    }
    bool supported = false;
    cudaError_t e = launch_logits(f, H, G, a, tmK, tmQ, tmS, nctas, LLONG_MAX, (cudaStream_t)stream,
                                  &supported);
    if (!supported || e == cudaErrorNotSupported)
        return IDX_ERR_UNSUPPORTED;
    return launch_status(e);
}

extern "C" idx_status idx_paged_mqa_logits(
    const void *q, const void *q_scale, const float *weights, const uint8_t *kv_pages,
    int64_t page_stride_bytes, int num_pages, const int32_t *block_table, int64_t bt_stride,
    const int32_t *context_lens, int ctx_per_row, const int32_t *row_ks, int B, int next_n, int H,
    int D, int page_size, idx_kv_format fmt, const int32_t *candidate_blocks, int64_t cand_stride,
    int num_cand, int cand_block, float *logits, int64_t ld_logits, int max_model_len,
    int num_ctas, void *ws, size_t ws_bytes, idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_paged_mqa_logits");
    return paged_logits(false, q, q_scale, weights, kv_pages, page_stride_bytes, num_pages,
                        block_table, bt_stride, context_lens, ctx_per_row, row_ks, B, next_n, H, D,
                        page_size, fmt, candidate_blocks, cand_stride, num_cand, cand_block, logits,
                        ld_logits, max_model_len, num_ctas, ws, ws_bytes, stream);
}

extern "C" idx_status idx_paged_mqa_logits_candidates(
    const void *q, const void *q_scale, const float *weights, const uint8_t *kv_pages,
    int64_t page_stride_bytes, int num_pages, const int32_t *block_table, int64_t bt_stride,
    const int32_t *context_lens, int ctx_per_row, const int32_t *row_ks, int B, int next_n, int H,
    int D, int page_size, idx_kv_format fmt, const int32_t *candidate_blocks, int64_t cand_stride,
    int num_cand, int cand_block, float *logits, int64_t ld_logits, int max_model_len,
    int num_ctas, void *ws, size_t ws_bytes, idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_paged_mqa_logits_candidates");
    if (!candidate_blocks || num_cand <= 0)
        return IDX_ERR_INVALID_ARG;
    return paged_logits(true, q, q_scale, weights, kv_pages, page_stride_bytes, num_pages,
                        block_table, bt_stride, context_lens, ctx_per_row, row_ks, B, next_n, H, D,
                        page_size, fmt, candidate_blocks, cand_stride, num_cand, cand_block, logits,
                        ld_logits, max_model_len, num_ctas, ws, ws_bytes, stream);
}

extern "C" idx_status idx_paged_mqa_logits_block_max(
    const void *q, const void *q_scale, const float *weights, const uint8_t *kv_pages,
    int64_t page_stride_bytes, int num_pages, const int32_t *block_table, int64_t bt_stride,
    const int32_t *context_lens, int ctx_per_row, const int32_t *row_ks, int B, int next_n, int H,
    int D, int page_size, idx_kv_format fmt, float *logits, int64_t ld_logits, int max_model_len,
    float *block_max, int64_t ld_block_max, int block_size, int num_ctas, idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_paged_mqa_logits_block_max");
    if (!block_max)
        return IDX_ERR_INVALID_ARG;
    BlockMaxOut bm;
    bm.out = block_max;
    bm.ld = ld_block_max;
    bm.block = block_size;
    return paged_logits(false, q, q_scale, weights, kv_pages, page_stride_bytes, num_pages,
                        block_table, bt_stride, context_lens, ctx_per_row, row_ks, B, next_n, H, D,
                        page_size, fmt, nullptr, 0, 0, 0, logits, ld_logits, max_model_len,
                        num_ctas, nullptr, 0, stream, bm);
}

extern "C" idx_status idx_paged_mqa_logits_topk(
    const void *q, const void *q_scale, const float *weights, const uint8_t *kv_pages,
    int64_t page_stride_bytes, int num_pages, const int32_t *block_table, int64_t bt_stride,
    const int32_t *context_lens, int ctx_per_row, const int32_t *row_ks, int B, int next_n, int H,
    int D, int page_size, idx_kv_format fmt, float *logits, int64_t ld_logits, int max_model_len,
    float *block_max, int64_t ld_block_max, int block_size, const int32_t *lengths, int k,
    int32_t *out_idx, int64_t ld_out, int num_ctas, void *ws, size_t ws_bytes,
    idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_paged_mqa_logits_topk");
    if (B < 0 || next_n <= 0 || k < 0 || ld_out < k || ld_logits <= 0 || ld_logits > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    if (B == 0 || max_model_len == 0)
        return IDX_OK;
    if (!lengths || (k > 0 && !out_idx))
        return IDX_ERR_INVALID_ARG;
    const int rows = B * next_n;
    BlockMaxOut bm;
    bm.out = block_max;
    bm.ld = ld_block_max;
    bm.block = block_size;
    cudaStream_t s = (cudaStream_t)stream;
    // the fused path: the logits kernel counts the top-k's digit-1 histograms
    // (one- and two-row groups; the chunked top-k must apply)
    const bool fused = k > 0 && next_n <= 2 &&
                       topk_takes_chunked(logits, ld_logits, rows, k, ws, ws_bytes);
    if (fused) {
        // the logits call's own checks run before the top-k's plan is
        // launched, so a rejected call launches nothing
        const idx_status chk = paged_logits(false, q, q_scale, weights, kv_pages,
                                            page_stride_bytes, num_pages, block_table, bt_stride,
                                            context_lens, ctx_per_row, row_ks, B, next_n, H, D,
                                            page_size, fmt, nullptr, 0, 0, 0, logits, ld_logits,
                                            max_model_len, num_ctas, nullptr, 0, stream, bm,
                                            /*check_only=*/true);
        if (chk != IDX_OK)
            return chk;
        idx_status st = topk_chunked_plan(lengths, ld_logits, rows, ws, 1, s);
        if (st != IDX_OK)
            return st;
        bm.hist_P = topk_chunked_counts(ws, rows, ld_logits, &bm.hist, &bm.hvalid, &bm.cvalid);
        st = paged_logits(false, q, q_scale, weights, kv_pages, page_stride_bytes, num_pages,
                          block_table, bt_stride, context_lens, ctx_per_row, row_ks, B, next_n,
                          H, D, page_size, fmt, nullptr, 0, 0, 0, logits, ld_logits,
                          max_model_len, num_ctas, nullptr, 0, stream, bm);
        if (st != IDX_OK)
            return st;
        const int vec_ok = (ld_logits % 4 == 0) && aligned16(logits);
        return topk_chunked_phases(logits, ld_logits, rows, lengths, k, out_idx, ld_out, ws,
                                   vec_ok, 1, s);
    }
    const idx_status st = paged_logits(false, q, q_scale, weights, kv_pages, page_stride_bytes,
                                       num_pages, block_table, bt_stride, context_lens,
                                       ctx_per_row, row_ks, B, next_n, H, D, page_size, fmt,
                                       nullptr, 0, 0, 0, logits, ld_logits, max_model_len,
                                       num_ctas, nullptr, 0, stream, bm);
    if (st != IDX_OK || k == 0)
        return st;
    return idx_topk(logits, ld_logits, rows, lengths, k, out_idx, ld_out, ws, ws_bytes, stream);
}

extern "C" size_t idx_paged_mqa_logits_workspace_size(int B, int next_n, int max_model_len,
                                                      int num_cand)
{
    (void)next_n;
    if (B <= 0 || max_model_len <= 0 || num_cand <= 0)
        return 0;
    int bw, pw, tw;
    plan_geom(max_model_len, &bw, &pw, &tw);
    return (size_t)B * pw * 4;
}

extern "C" idx_status idx_get_device_status(idx_stream_t stream, uint32_t *out)
{
    IDX_NVTX_RANGE("idx_get_device_status");
    if (!out)
        return IDX_ERR_INVALID_ARG;
    unsigned int *p = device_status_ptr();
    if (!p)
        return IDX_ERR_CUDA;
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(p, 0, sizeof(unsigned int), (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize((cudaStream_t)stream);
    *out = v;
    return launch_status(e);
}

extern "C" const char *idx_version(void)
{
    return "idx 0.1 sm_103a";
}
