// idx_produce.cu -- the K and Q producers of the indexer cache.
//
// Passages: vllm/models/deepseek_v41/amd/rocm.py, rocm_mxfp4_indexer_k_store
// (the key is RMS-normalised, rotated at its position and written quantised
// into its cache slot) and rocm_mxfp4_indexer_q_quant (the query heads are
// rotated and quantised; the weights are multiplied by the softmax scale
// times the head scale).  RoPE: GPT-J pairs on the trailing rope_dim of a
// head, the cos/sin row laid out cos | sin (rocm_aiter_mla_sparse,
// _inverse_rope_gptj_kernel, whose rotation this inverts).  Quantiser:
// rocm_aiter_mla_sparse, _mxfp8_scale_bits: the biased E8M0 exponent that
// puts a block's amax at the top of the element range (448 for e4m3, 6 for
// e2m1), values multiplied by 2^(127 - bits) and rounded to the nearest code,
// ties to the even code.
//
// One warp per token (K) or per (token, head) (Q); lane l holds elements
// 4l .. 4l + 3 of the 128, so a GPT-J pair never leaves a lane, an MXFP4
// block of 32 is eight lanes and the token's amax is a warp reduction.  The
// work is a few hundred bytes per token: the kernels are bound by memory
// latency and bandwidth, not arithmetic.
#include <cstdint>
#include <cuda_fp8.h>

#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

constexpr int kProdThreads = 256;
constexpr unsigned kDevBadPosition = 8u;
constexpr int kProdFp8 = 0;
constexpr int kProdMxfp4 = 1;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b)
{
    return __uint_as_float(b << 16);
}

// Biased E8M0 exponent putting amax at the top of the element range,
// top = 1.f_top * 2^e_top, read off the bit fields: with amax = 1.f * 2^e
// (amax floored at 2^-126, so normal), the smallest k with amax <= top * 2^k
// is e - e_top, plus one when f > f_top; then 127 + k, clamped to [0, 254].
__device__ __forceinline__ int scale_bits(float amax, uint32_t f_top, int e_top)
{
    const uint32_t u = __float_as_uint(fmaxf(amax, 1.17549435e-38f));
    const int e = (int)(u >> 23) - 127;
    const int bits = 127 + e - e_top + ((u & 0x7fffffu) > f_top ? 1 : 0);
    return min(max(bits, 0), 254);
}

// 2^(127 - bits) for bits in [0, 254], built from its bit pattern (2^-127
// is the one subnormal value).
__device__ __forceinline__ float inv_scale(int bits)
{
    return bits < 254 ? __uint_as_float((uint32_t)(254 - bits) << 23) : __uint_as_float(0x400000u);
}

// 2^(bits - 127) for bits in [0, 254] (2^-127 subnormal, 2^127 normal).
__device__ __forceinline__ float scale_of(int bits)
{
    return bits > 0 ? __uint_as_float((uint32_t)bits << 23) : __uint_as_float(0x400000u);
}

// Four values (|y| <= 6 after scaling) to four e2m1 codes in the low 16
// bits, element 2j in the low nibble of byte j: the hardware conversion of
// a pair of f32 to a packed e2m1 pair, round to nearest even (its second
// source lands in the low nibble).
__device__ __forceinline__ uint32_t e2m1_pack4(float y0, float y1, float y2, float y3)
{
    uint32_t out;
    asm("{\n"
        ".reg .b8 lo, hi;\n"
        "cvt.rn.satfinite.e2m1x2.f32 lo, %2, %1;\n"
        "cvt.rn.satfinite.e2m1x2.f32 hi, %4, %3;\n"
        "mov.b32 %0, {lo, hi, 0, 0};\n"
        "}"
        : "=r"(out)
        : "f"(y0), "f"(y1), "f"(y2), "f"(y3));
    return out;
}

// GPT-J rotation of the lane's pairs (y[0], y[1]) and (y[2], y[3]) that lie
// in the trailing rope_dim of the head: even' = a cos - b sin,
// odd' = b cos + a sin.
__device__ __forceinline__ void rope_lane(float y[4], int lane, int rope_dim, const float *cs)
{
    const int n = 128 - rope_dim, half = rope_dim / 2;
    #pragma unroll
    for (int i = 0; i < 4; i += 2) {
        const int e = 4 * lane + i;
        if (e >= n) {
            const int p = (e - n) >> 1;
            const float c = cs[p], s = cs[half + p];
            const float a = y[i], b = y[i + 1];
            y[i] = a * c - b * s;
            y[i + 1] = b * c + a * s;
        }
    }
}

__device__ __forceinline__ float warp_max(float v)
{
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Quantise the lane's four values.  FP8: one exponent for the whole head
// (warp amax); the four e4m3 codes come back in one word.  MXFP4: one
// exponent per eight lanes; the four nibbles come back in the low 16 bits.
__device__ __forceinline__ uint32_t quantise_lane(const float y[4], int fmt, int *bits_out)
{
    float amax = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
    if (fmt == kProdFp8) {
        amax = warp_max(amax);
        const int bits = scale_bits(amax, 0x600000u, 8);  // 448 = 1.75 * 2^8
        const float inv = inv_scale(bits);
        uint32_t word = 0;
        #pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(y[i] * inv, __NV_SATFINITE, __NV_E4M3);
            word |= (uint32_t)c << (8 * i);
        }
        *bits_out = bits;
        return word;
    }
    #pragma unroll
    for (int o = 1; o < 8; o <<= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int bits = scale_bits(amax, 0x400000u, 2);  // 6 = 1.5 * 2^2
    const float inv = inv_scale(bits);
    *bits_out = bits;
    return e2m1_pack4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv);
}

__global__ void __launch_bounds__(kProdThreads)
    k_store_kernel(const uint16_t *__restrict__ k_pre, int64_t ld_k,
                   const int32_t *__restrict__ positions, const float *__restrict__ cos_sin,
                   int64_t ld_cs, int num_pos, int rope_dim, const float *__restrict__ norm_w,
                   float eps, uint8_t *__restrict__ pages, int64_t page_stride, int num_pages,
                   int page_size, const int64_t *__restrict__ slots, int T, int fmt,
                   unsigned int *status)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (kProdThreads / 32);
    for (int t = blockIdx.x * (kProdThreads / 32) + (threadIdx.x >> 5); t < T; t += warps) {
        const int64_t slot = slots[t];
        if (slot < 0)
            continue;
        const int64_t page = slot / page_size, off = slot - page * page_size;
        const int pos = positions[t];
        if (page >= num_pages || pos < 0 || pos >= num_pos) {
            if (lane == 0)
                atomicOr(status, page >= num_pages ? kDevBadPage : kDevBadPosition);
            continue;
        }
        const uint2 raw = *reinterpret_cast<const uint2 *>(k_pre + (size_t)t * ld_k + 4 * lane);
        float y[4] = {bf16_bits_to_float(raw.x & 0xffffu), bf16_bits_to_float(raw.x >> 16),
                      bf16_bits_to_float(raw.y & 0xffffu), bf16_bits_to_float(raw.y >> 16)};
        float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
        #pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = 1.0f / sqrtf(ss / 128.0f + eps);
        const float4 w = *reinterpret_cast<const float4 *>(norm_w + 4 * lane);
        y[0] = y[0] * r * w.x;
        y[1] = y[1] * r * w.y;
        y[2] = y[2] * r * w.z;
        y[3] = y[3] * r * w.w;
        rope_lane(y, lane, rope_dim, cos_sin + (size_t)pos * ld_cs);
        int bits;
        const uint32_t q = quantise_lane(y, fmt, &bits);
        uint8_t *pg = pages + page * page_stride;
        if (fmt == kProdFp8) {
            *reinterpret_cast<uint32_t *>(pg + off * 128 + 4 * lane) = q;
            if (lane == 0)
                *reinterpret_cast<float *>(pg + (int64_t)page_size * 128 + off * 4) =
                    scale_of(bits);
        } else {
            *reinterpret_cast<uint16_t *>(pg + off * 64 + 2 * lane) = (uint16_t)q;
            if ((lane & 7) == 0)
                pg[(int64_t)page_size * 64 + off * 4 + (lane >> 3)] = (uint8_t)bits;
        }
    }
}

// Each warp takes kQHeads heads of one token at a time: the token's
// position and cos/sin row are loaded once for them, and all the heads'
// loads are issued before any is computed (a head is only 256 bytes, so one
// head per warp leaves too little in flight to cover the memory latency).
constexpr int kQHeads = 8;

__global__ void __launch_bounds__(kProdThreads)
    q_quant_kernel(const uint16_t *__restrict__ q, const int32_t *__restrict__ positions,
                   const float *__restrict__ cos_sin, int64_t ld_cs, int num_pos, int rope_dim,
                   const float *__restrict__ w_in, float w_scale, int T, int H, int fmt,
                   uint8_t *__restrict__ q_out, uint8_t *__restrict__ q_sf,
                   float *__restrict__ w_out, unsigned int *status)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int groups = (H + kQHeads - 1) / kQHeads;  // head groups of a token
    const long long items = (long long)T * groups;
    const long long warps = (long long)gridDim.x * (kProdThreads / 32);
    const int n = 128 - rope_dim, half = rope_dim / 2;
    for (long long it = (long long)blockIdx.x * (kProdThreads / 32) + (threadIdx.x >> 5);
         it < items; it += warps) {
        const int t = (int)(it / groups);
        const int h0 = (int)(it - (long long)t * groups) * kQHeads;
        const int pos = positions[t];
        uint2 raw[kQHeads];
        #pragma unroll
        for (int u = 0; u < kQHeads; ++u) {
            const long long th = (long long)t * H + h0 + u;
            raw[u] = h0 + u < H ? *reinterpret_cast<const uint2 *>(q + th * 128 + 4 * lane)
                                : make_uint2(0u, 0u);
        }
        if (pos < 0 || pos >= num_pos) {
            if (lane == 0)
                atomicOr(status, kDevBadPosition);
            continue;
        }
        float cs[4] = {1.0f, 0.0f, 1.0f, 0.0f};  // cos, sin of the lane's two pairs
        #pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int e = 4 * lane + 2 * i;
            if (e >= n) {
                const float *row = cos_sin + (size_t)pos * ld_cs;
                cs[2 * i] = row[(e - n) >> 1];
                cs[2 * i + 1] = row[half + ((e - n) >> 1)];
            }
        }
        #pragma unroll
        for (int u = 0; u < kQHeads; ++u) {
            if (h0 + u >= H)
                break;
            const long long th = (long long)t * H + h0 + u;
            float y[4] = {bf16_bits_to_float(raw[u].x & 0xffffu), bf16_bits_to_float(raw[u].x >> 16),
                          bf16_bits_to_float(raw[u].y & 0xffffu), bf16_bits_to_float(raw[u].y >> 16)};
            #pragma unroll
            for (int i = 0; i < 2; ++i) {
                if (4 * lane + 2 * i >= n) {  // GPT-J pair of the trailing rope_dim
                    const float a = y[2 * i], b = y[2 * i + 1];
                    y[2 * i] = a * cs[2 * i] - b * cs[2 * i + 1];
                    y[2 * i + 1] = b * cs[2 * i] + a * cs[2 * i + 1];
                }
            }
            int bits;
            const uint32_t qq = quantise_lane(y, fmt, &bits);
            if (fmt == kProdFp8) {
                *reinterpret_cast<uint32_t *>(q_out + th * 128 + 4 * lane) = qq;
                if (lane == 0)
                    w_out[th] = w_in[th] * w_scale * scale_of(bits);
            } else {
                *reinterpret_cast<uint16_t *>(q_out + th * 64 + 2 * lane) = (uint16_t)qq;
                if ((lane & 7) == 0)
                    q_sf[th * 4 + (lane >> 3)] = (uint8_t)bits;
                if (lane == 0)
                    w_out[th] = w_in[th] * w_scale;
            }
        }
    }
}

int prod_grid(long long warps_needed)
{
    const long long ctas = (warps_needed + kProdThreads / 32 - 1) / (kProdThreads / 32);
    const long long cap = (long long)sm_count() * 16;
    return (int)(ctas < cap ? (ctas > 0 ? ctas : 1) : cap);
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

} // namespace
} // namespace idx

using namespace idx;

extern "C" idx_status idx_k_norm_rope_store(const uint16_t *k_pre, int64_t ld_k,
                                            const int32_t *positions, const float *cos_sin,
                                            int64_t ld_cos_sin, int num_positions, int rope_dim,
                                            const float *norm_weight, float eps, int T, int D,
                                            idx_kv_format fmt, uint8_t *kv_pages,
                                            int64_t page_stride_bytes, int num_pages,
                                            int page_size, const int64_t *slot_mapping,
                                            idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_k_norm_rope_store");
    if (T < 0 || D <= 0 || rope_dim < 0 || rope_dim % 2 != 0 || rope_dim > D ||
        num_positions < 0 || ld_cos_sin < rope_dim || page_size <= 0 || num_pages < 0 ||
        ld_k < D || !(eps >= 0.0f) ||
        (fmt != IDX_KV_FP8_E4M3 && fmt != IDX_KV_MXFP4))
        return IDX_ERR_INVALID_ARG;
    if (T == 0)
        return IDX_OK;
    if (!k_pre || !positions || !norm_weight || !kv_pages || !slot_mapping ||
        (rope_dim > 0 && !cos_sin))
        return IDX_ERR_INVALID_ARG;
    const int f = fmt == IDX_KV_FP8_E4M3 ? kProdFp8 : kProdMxfp4;
    const int64_t page_bytes = (int64_t)page_size * (f == kProdFp8 ? D + 4 : D / 2 + D / 32);
    if (page_stride_bytes < page_bytes)
        return IDX_ERR_INVALID_ARG;
    if (D != 128 || ld_k % 4 != 0 || !aligned(k_pre, 8) || !aligned(norm_weight, 16) ||
        !aligned(kv_pages, 4) || page_stride_bytes % 4 != 0)
        return IDX_ERR_UNSUPPORTED;
    unsigned int *status = device_status_ptr();
    if (!status)
        return IDX_ERR_CUDA;
    return launch_status(launch_pdl(k_store_kernel, dim3(prod_grid(T)), dim3(kProdThreads), 0,
                                    (cudaStream_t)stream, k_pre, ld_k, positions, cos_sin,
                                    ld_cos_sin, num_positions, rope_dim, norm_weight, eps,
                                    kv_pages, page_stride_bytes, num_pages, page_size,
                                    slot_mapping, T, f, status));
}

extern "C" idx_status idx_q_rope_quant(const uint16_t *q, const int32_t *positions,
                                       const float *cos_sin, int64_t ld_cos_sin,
                                       int num_positions, int rope_dim, const float *weights,
                                       float weight_scale, int T, int H, int D, idx_kv_format fmt,
                                       uint8_t *q_out, void *q_scale_out, float *weights_out,
                                       idx_stream_t stream)
{
    IDX_NVTX_RANGE("idx_q_rope_quant");
    if (T < 0 || H <= 0 || D <= 0 || rope_dim < 0 || rope_dim % 2 != 0 || rope_dim > D ||
        num_positions < 0 || ld_cos_sin < rope_dim ||
        (fmt != IDX_KV_FP8_E4M3 && fmt != IDX_KV_MXFP4))
        return IDX_ERR_INVALID_ARG;
    if (T == 0)
        return IDX_OK;
    const int f = fmt == IDX_KV_FP8_E4M3 ? kProdFp8 : kProdMxfp4;
    if (!q || !positions || !weights || !q_out || !weights_out ||
        (f == kProdMxfp4 && !q_scale_out) || (rope_dim > 0 && !cos_sin))
        return IDX_ERR_INVALID_ARG;
    if (D != 128 || !aligned(q, 8) || !aligned(q_out, 4))
        return IDX_ERR_UNSUPPORTED;
    unsigned int *status = device_status_ptr();
    if (!status)
        return IDX_ERR_CUDA;
    return launch_status(launch_pdl(q_quant_kernel,
                                    dim3(prod_grid((long long)T * ((H + kQHeads - 1) / kQHeads))),
                                    dim3(kProdThreads), 0, (cudaStream_t)stream, q, positions,
                                    cos_sin, ld_cos_sin, num_positions, rope_dim, weights,
                                    weight_scale, T, H, f,
                                    q_out, static_cast<uint8_t *>(q_scale_out), weights_out,
                                    status));
}
