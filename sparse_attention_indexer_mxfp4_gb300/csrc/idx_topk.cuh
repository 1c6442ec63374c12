// idx_topk.cuh -- per-row top-k by radix select, one CTA per row.
//
// Passage: vLLM page rocm_paged_mxfp4_indexer, _topk -- top-k over each
// row's [0, lengths[row]), -1 padding.  The design is our own.
//
// Each warp of the CTA takes a contiguous sub-slice of [0, len), so
// (warp, position) is index order.  Values become order-preserving 32-bit
// keys; non-finite values become key 0 and are never selected.  Every
// streaming pass keeps four float4 loads per thread in flight.
//   pass 1 (stream): histogram of the top 11 key bits and the valid count;
//          the bin b1 holding the k-th largest key follows from a block scan.
//   pass 2 (stream): keys in bin b1 are appended, with their index, to a
//          shared-memory candidate list; keys above b1 are counted per warp.
//   digits 2 and 3 (11 and 10 bits) are then resolved on the candidates
//          (or, if the list overflowed, by streaming the row again), which
//          gives the k-th largest key T and how many keys equal to T to take.
//   pass 3 (stream): every warp writes its selected indices in index order
//          at offsets from a block prefix sum.  Keys equal to T are taken
//          lowest index first, so the selected set is unique.
#pragma once

#include <cstdint>

#include "idx_common.cuh"

namespace idx {
// Slot counting in a top-k kernel that writes a row's indices (the fused
// top-k -> ragged slots call): the slot of position p of sequence b is valid
// when its logical page p / P is below max_blocks and bt[b, p / P] lies in
// [0, num_pages).  bt == nullptr: no counting.  lens[row] receives the
// row's valid slots; an invalid one sets kDevBadPage in *status.
struct SlotCount {
    const int32_t *bt;
    int64_t bt_stride;
    int max_blocks, P, shift, num_pages;  // shift = log2(P) when P is a power of two, else -1
    const int32_t *row_to_seq;            // nullptr: row / next_n
    int next_n;
    int32_t *lens;
    unsigned int *status;
};

// Whether the slot of position p of sequence b is valid (see SlotCount).
__device__ __forceinline__ bool slot_valid(const SlotCount &sc, int b, int p)
{
    const int lp = sc.shift >= 0 ? p >> sc.shift : p / sc.P;
    if (lp >= sc.max_blocks)
        return false;
    const int pg = __ldg(sc.bt + (size_t)b * sc.bt_stride + lp);
    return pg >= 0 && pg < sc.num_pages;
}

namespace topk_detail {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;             // float4 loads in flight per thread
constexpr int kChunk = 128 * kUnroll;  // elements a warp handles per step
constexpr int kCandCap = 6144;         // candidate keys kept in shared memory

struct Shared {
    uint32_t hist[2][2048];
    uint32_t cand_key[kCandCap];
    int32_t cand_idx[kCandCap];
    uint32_t wsum[kWarps + 1];
    uint32_t wgt[kWarps];  // per warp: keys > T
    uint32_t weq[kWarps];  // per warp: keys == T
    uint32_t sel[2];       // digit found, remaining rank
    uint32_t ncand;
};

__device__ __forceinline__ uint32_t float_key(float v)
{
    return order_key(v);
}

// Keys of elements i0..i0+3 of a row (0 past `end`).
__device__ __forceinline__ void load4(const float *row, int i0, int end, bool vec, uint32_t (&k)[4])
{
    if (vec && i0 + 3 < end) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(row + i0));
        k[0] = float_key(v.x);
        k[1] = float_key(v.y);
        k[2] = float_key(v.z);
        k[3] = float_key(v.w);
    } else {
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            k[e] = i0 + e < end ? float_key(__ldg(row + i0 + e)) : 0u;
    }
}

// Keys of U runs of four elements, run u starting at base + u * stride (0
// past `end`).  Every load is issued before any key is formed, so the U
// memory round trips overlap: float4 loads where the whole run is in range
// and the row allows them, scalar loads for the rest.
template <int U>
__device__ __forceinline__ void load_keys(const float *row, int base, int stride, int end, bool vec,
                                          uint32_t (&k)[U][4], int nrun = U)
{
    // runs u >= nrun (the same in every thread of the caller) hold no key and
    // issue no load
    float4 v[U];
    #pragma unroll
    for (int u = 0; u < U; ++u) {
        const int i0 = base + u * stride;
        v[u] = make_float4(NAN, NAN, NAN, NAN);
        if (u < nrun && vec && i0 + 3 < end)
            v[u] = __ldg(reinterpret_cast<const float4 *>(row + i0));
    }
    #pragma unroll
    for (int u = 0; u < U; ++u) {
        const int i0 = base + u * stride;
        if (u >= nrun)
            break;
        if (!(vec && i0 + 3 < end)) {
            if (i0 < end)
                v[u].x = __ldg(row + i0);
            if (i0 + 1 < end)
                v[u].y = __ldg(row + i0 + 1);
            if (i0 + 2 < end)
                v[u].z = __ldg(row + i0 + 2);
            if (i0 + 3 < end)
                v[u].w = __ldg(row + i0 + 3);
        }
    }
    #pragma unroll
    for (int u = 0; u < U; ++u) {
        k[u][0] = float_key(v[u].x);
        k[u][1] = float_key(v[u].y);
        k[u][2] = float_key(v[u].z);
        k[u][3] = float_key(v[u].w);
    }
}

// One warp step: the keys of elements cb + 128u + 4*lane + e (u < kUnroll,
// e < 4), all loads issued before any is used.  Element order within the
// step is (u, lane, e).
__device__ __forceinline__ void load_step(const float *row, int cb, int end, bool vec, int lane,
                                          uint32_t (&k)[kUnroll][4])
{
    load_keys<kUnroll>(row, cb + 4 * lane, 128, end, vec, k);
}

// Sum of a value over the warp.
__device__ __forceinline__ uint32_t warp_sum(uint32_t v)
{
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exclusive prefix of v over the lanes; *tot gets the warp total.
__device__ __forceinline__ uint32_t warp_excl(uint32_t v, int lane, uint32_t *tot)
{
    uint32_t x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += n;
    }
    *tot = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
}

// Find the bin (of nb, scanned from the top) where the descending
// cumulative count reaches krem; writes (bin, krem - count above it) to
// sh.sel.  All threads call it; it starts and ends with a barrier.
__device__ __forceinline__ void find_bin(Shared &sh, const uint32_t *h, int nb, uint32_t krem)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    uint32_t loc[4];
    uint32_t lsum = 0;
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int b = nb - 1 - (tid * 4 + j);  // descending bins
        loc[j] = b >= 0 ? h[b] : 0u;
        lsum += loc[j];
    }
    uint32_t wt;
    const uint32_t ex = warp_excl(lsum, lane, &wt);
    __syncthreads();  // earlier readers of wsum are done
    if (lane == 0)
        sh.wsum[w] = wt;
    __syncthreads();
    uint32_t before = ex;
    for (int i = 0; i < w; ++i)
        before += sh.wsum[i];
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int b = nb - 1 - (tid * 4 + j);
        if (b >= 0 && before < krem && before + loc[j] >= krem) {
            sh.sel[0] = (uint32_t)b;
            sh.sel[1] = krem - before;
        }
        before += loc[j];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 2)
    topk_kernel(const float *__restrict__ logits, int64_t ld, int rows,
                const int32_t *__restrict__ lengths, int k, int32_t *__restrict__ out,
                int64_t ld_out, int vec_ok)
{
    const int row = blockIdx.x;
    extern __shared__ __align__(16) uint8_t dsm[];
    Shared &sh = *reinterpret_cast<Shared *>(dsm);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (row >= rows) {
        pdl_launch_dependents();
        return;
    }
    for (int i = tid; i < 2 * 2048; i += kThreads)
        (&sh.hist[0][0])[i] = 0u;
    if (tid == 0)
        sh.ncand = 0;
    pdl_wait();  // the logits and lengths may come from the kernel before this one
    pdl_launch_dependents();
    const int len = max(0, min(lengths[row], (int)ld));
    // warp sub-slices, starts aligned to 4 elements
    const int wper = ((len + kWarps - 1) / kWarps + 3) & ~3;
    const int ws = min(len, warp * wper);
    const int we = min(len, ws + wper);
    const float *rowp = logits + (size_t)row * ld;
    const bool vec = vec_ok != 0;
    __syncthreads();

    // ---- pass 1: histogram of digit 1, count of valid keys
    uint32_t nvalid = 0;
    for (int cb = ws; cb < we; cb += kChunk) {
        uint32_t key[kUnroll][4];
        load_step(rowp, cb, we, vec, lane, key);
        #pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (key[u][e]) {
                    ++nvalid;
                    atomicAdd(&sh.hist[0][key[u][e] >> 21], 1u);
                }
    }
    nvalid = warp_sum(nvalid);
    if (lane == 0)
        sh.wsum[warp] = nvalid;
    __syncthreads();
    uint32_t total_valid = 0;
    for (int i = 0; i < kWarps; ++i)
        total_valid += sh.wsum[i];
    const bool take_all = total_valid <= (uint32_t)k;

    uint32_t T = 0, ties = 0;
    uint32_t my_gt = 0;  // this lane's keys above bin b1
    bool overflow = false;
    if (!take_all) {
        find_bin(sh, sh.hist[0], 2048, (uint32_t)k);
        const uint32_t b1 = sh.sel[0];
        uint32_t krem = sh.sel[1];
        // ---- pass 2: candidates of bin b1, count keys above it
        for (int cb = ws; cb < we; cb += kChunk) {
            uint32_t key[kUnroll][4];
            load_step(rowp, cb, we, vec, lane, key);
            #pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t d = key[u][e] >> 21;
                    my_gt += key[u][e] && d > b1;
                    const bool is_c = key[u][e] && d == b1;
                    const uint32_t ball = __ballot_sync(0xffffffffu, is_c);
                    if (ball) {
                        uint32_t base = 0;
                        if (lane == 0)
                            base = atomicAdd(&sh.ncand, (uint32_t)__popc(ball));
                        base = __shfl_sync(0xffffffffu, base, 0);
                        const uint32_t pos = base + __popc(ball & ((1u << lane) - 1u));
                        if (is_c && pos < (uint32_t)kCandCap) {
                            sh.cand_key[pos] = key[u][e];
                            sh.cand_idx[pos] = cb + 128 * u + 4 * lane + e;
                        }
                    }
                }
        }
        __syncthreads();
        const uint32_t ncand = sh.ncand;
        overflow = ncand > (uint32_t)kCandCap;
        // ---- digits 2 and 3
        uint32_t prefix = b1 << 21, pmask = 0xFFE00000u;
        for (int pass = 1; pass < 3; ++pass) {
            const int shift = pass == 1 ? 10 : 0;
            const int nb = pass == 1 ? 2048 : 1024;
            uint32_t *h = sh.hist[pass & 1];
            for (int i = tid; i < 2048; i += kThreads)
                h[i] = 0u;
            __syncthreads();
            if (!overflow) {
                for (uint32_t i = tid; i < ncand; i += kThreads) {
                    const uint32_t kk = sh.cand_key[i];
                    if ((kk & pmask) == prefix)
                        atomicAdd(&h[(kk >> shift) & (uint32_t)(nb - 1)], 1u);
                }
            } else {
                for (int cb = ws; cb < we; cb += kChunk) {
                    uint32_t key[kUnroll][4];
                    load_step(rowp, cb, we, vec, lane, key);
                    #pragma unroll
                    for (int u = 0; u < kUnroll; ++u)
                        #pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (key[u][e] && (key[u][e] & pmask) == prefix)
                                atomicAdd(&h[(key[u][e] >> shift) & (uint32_t)(nb - 1)], 1u);
                }
            }
            __syncthreads();
            find_bin(sh, h, nb, krem);
            prefix |= sh.sel[0] << shift;
            pmask |= (uint32_t)(nb - 1) << shift;
            krem = sh.sel[1];
        }
        T = prefix;
        ties = krem;
    }

    // ---- per-warp counts of keys > T and == T (T = 0 when every valid key fits)
    if (take_all || overflow) {
        uint32_t gt = 0, eq = 0;
        for (int cb = ws; cb < we; cb += kChunk) {
            uint32_t key[kUnroll][4];
            load_step(rowp, cb, we, vec, lane, key);
            #pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    gt += key[u][e] > T;
                    eq += key[u][e] == T && key[u][e];
                }
        }
        gt = warp_sum(gt);
        eq = warp_sum(eq);
        if (lane == 0) {
            sh.wgt[warp] = gt;
            sh.weq[warp] = eq;
        }
        __syncthreads();
    } else {
        my_gt = warp_sum(my_gt);
        if (lane == 0) {
            sh.wgt[warp] = my_gt;
            sh.weq[warp] = 0;
        }
        __syncthreads();
        const uint32_t ncand = sh.ncand;
        for (uint32_t i = tid; i < ncand; i += kThreads) {
            const uint32_t kk = sh.cand_key[i];
            const int wi = sh.cand_idx[i] / wper;
            if (kk > T)
                atomicAdd(&sh.wgt[wi], 1u);
            else if (kk == T)
                atomicAdd(&sh.weq[wi], 1u);
        }
        __syncthreads();
    }
    // this warp's tie quota and output base (warps in index order)
    uint32_t eq_run = 0, base = 0, total_sel = 0, quota = 0;
    for (int i = 0; i < kWarps; ++i) {
        const uint32_t e = sh.weq[i];
        const uint32_t take = eq_run >= ties ? 0u : min(e, ties - eq_run);
        if (i < warp)
            base += sh.wgt[i] + take;
        if (i == warp)
            quota = take;
        total_sel += sh.wgt[i] + take;
        eq_run += e;
    }

    // ---- pass 3: ordered write of the selection
    int32_t *orow = out + (size_t)row * ld_out;
    uint32_t written = 0, eq_seen = 0;
    for (int cb = ws; cb < we; cb += kChunk) {
        uint32_t key[kUnroll][4];
        load_step(rowp, cb, we, vec, lane, key);
        #pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            uint32_t neq = 0;
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                neq += key[u][e] == T && key[u][e];
            uint32_t eq_tot;
            uint32_t er = eq_seen + warp_excl(neq, lane, &eq_tot);
            uint32_t take[4], nt = 0;
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                bool t = key[u][e] > T;
                if (key[u][e] == T && key[u][e]) {
                    t = er < quota;
                    ++er;
                }
                take[e] = t;
                nt += t;
            }
            uint32_t tot;
            uint32_t pos = base + written + warp_excl(nt, lane, &tot);
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (take[e])
                    orow[pos++] = cb + 128 * u + 4 * lane + e;
            written += tot;
            eq_seen += eq_tot;
        }
    }
    for (int j = (int)total_sel + tid; j < k; j += kThreads)
        orow[j] = -1;
}

} // namespace topk_detail
} // namespace idx
