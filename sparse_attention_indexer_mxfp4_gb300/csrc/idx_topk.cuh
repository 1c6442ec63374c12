// idx_topk.cuh -- per-row top-k by cluster radix select.
//
// Passage: vLLM page rocm_paged_mxfp4_indexer, _topk -- top-k over each
// row's [0, lengths[row]), -1 padding.  The design is our own.
//
// One thread-block cluster of C CTAs handles one row; CTA c takes a
// contiguous slice of [0, len) and each of its warps a contiguous sub-slice,
// so (CTA, warp, position) is index order.  Values become order-preserving
// 32-bit keys; non-finite values become key 0 and are never selected.
//   pass 1 (stream): histogram of the top 11 key bits; the C histograms are
//          summed through distributed shared memory and every CTA finds the
//          same bin b1 holding the k-th largest key.
//   pass 2 (stream): keys in bin b1 are appended, with their index, to a
//          shared-memory candidate list; keys above b1 are counted per warp.
//   digits 2 and 3 (11 and 10 bits) are then resolved on the candidates
//          (or, if the list overflowed, by streaming the slice again), which
//          gives the k-th largest key T and how many keys equal to T to take.
//   pass 3 (stream): every warp writes its selected indices in index order
//          at offsets from block and cluster prefix sums.  Keys equal to T
//          are taken lowest index first, so the selected set is unique.
// All cross-CTA waits are hardware cluster barriers on a path every CTA of
// the cluster takes the same number of times.
#pragma once

#include <cooperative_groups.h>
#include <cstdint>

namespace idx {
namespace topk_detail {

namespace cg = cooperative_groups;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCandCap = 6144;  // candidate keys kept in shared memory per CTA
constexpr int kMaxCluster = 8;

struct Shared {
    uint32_t hist[2][2048];
    uint32_t cand_key[kCandCap];
    int32_t cand_idx[kCandCap];
    uint32_t wsum[kWarps + 1];
    uint32_t wgt[kWarps];     // per warp: keys > T
    uint32_t weq[kWarps];     // per warp: keys == T
    uint32_t cta[4];          // exported to the cluster: valid, selected, equal
    uint32_t sel[2];          // digit found, remaining rank
    uint32_t ncand;
};

__device__ __forceinline__ uint32_t float_key(float v)
{
    const uint32_t b = __float_as_uint(v);
    if (!isfinite(v))
        return 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
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

// Exclusive scan over the kWarps per-warp values v[w] (one thread per warp
// slot, executed by warp 0); returns nothing, rewrites v in place and puts
// the total in *tot.  Caller syncs.
__device__ __forceinline__ void warp0_excl_scan(uint32_t *v, uint32_t *tot)
{
    const int lane = threadIdx.x & 31;
    uint32_t x = lane < kWarps ? v[lane] : 0u;
    uint32_t incl = x;
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += n;
    }
    if (lane < kWarps)
        v[lane] = incl - x;
    if (lane == 31)
        *tot = incl;
}

// Sum the C histograms of `h` (nb bins) through distributed shared memory,
// find the bin where the descending cumulative count reaches krem; returns
// (bin, krem - count above the bin) via sh.sel.  Every CTA computes the same.
__device__ __forceinline__ void find_bin(cg::cluster_group &cluster, Shared &sh, uint32_t *h,
                                         int nb, uint32_t krem)
{
    const int C = (int)cluster.num_blocks();
    const int tid = threadIdx.x;
    uint32_t loc[4];
    uint32_t lsum = 0;
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int b = nb - 1 - (tid * 4 + j);  // descending bins
        uint32_t v = 0;
        if (b >= 0) {
            if (C == 1)
                v = h[b];
            else
                for (int r = 0; r < C; ++r)
                    v += cluster.map_shared_rank(h, r)[b];
        }
        loc[j] = v;
        lsum += v;
    }
    // block exclusive scan of lsum
    const int lane = tid & 31, w = tid >> 5;
    uint32_t x = lsum;
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t n = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += n;
    }
    if (lane == 31)
        sh.wsum[w] = x;
    __syncthreads();
    if (w == 0)
        warp0_excl_scan(sh.wsum, &sh.wsum[kWarps]);
    __syncthreads();
    uint32_t before = sh.wsum[w] + x - lsum;
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

__global__ void __launch_bounds__(kThreads)
    topk_kernel(const float *__restrict__ logits, int64_t ld, int rows,
                const int32_t *__restrict__ lengths, int k, int32_t *__restrict__ out,
                int64_t ld_out, int vec_ok)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int row = blockIdx.x / C;
    extern __shared__ __align__(16) uint8_t dsm[];
    Shared &sh = *reinterpret_cast<Shared *>(dsm);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const bool row_ok = row < rows;
    int len = row_ok ? lengths[row] : 0;
    len = max(0, min(len, (int)ld));
    // CTA slice and warp sub-slices, starts aligned to 4 elements
    const int per = ((len + C - 1) / C + 3) & ~3;
    const int lo = min(len, crank * per);
    const int hi = min(len, lo + per);
    const int wper = ((hi - lo + kWarps - 1) / kWarps + 3) & ~3;
    const int ws = min(hi, lo + warp * wper);
    const int we = min(hi, ws + wper);
    const float *rowp = logits + (size_t)(row_ok ? row : 0) * ld;
    const bool vec = vec_ok != 0;

    for (int i = tid; i < 2 * 2048; i += kThreads)
        (&sh.hist[0][0])[i] = 0u;
    if (tid == 0)
        sh.ncand = 0;
    __syncthreads();

    // ---- pass 1: histogram of digit 1, count of valid keys
    uint32_t nvalid = 0;
    for (int cb = ws; cb < we; cb += 128) {
        uint32_t key[4];
        load4(rowp, cb + 4 * lane, we, vec, key);
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if (key[e]) {
                ++nvalid;
                atomicAdd(&sh.hist[0][key[e] >> 21], 1u);
            }
    }
    for (int o = 16; o > 0; o >>= 1)
        nvalid += __shfl_xor_sync(0xffffffffu, nvalid, o);
    if (lane == 0)
        sh.wsum[warp] = nvalid;
    __syncthreads();
    if (tid == 0) {
        uint32_t t = 0;
        for (int i = 0; i < kWarps; ++i)
            t += sh.wsum[i];
        sh.cta[0] = t;
    }
    cluster.sync();
    uint32_t total_valid = 0;
    for (int r = 0; r < C; ++r)
        total_valid += C == 1 ? sh.cta[0] : cluster.map_shared_rank(&sh, r)->cta[0];
    const bool take_all = total_valid <= (uint32_t)k;

    uint32_t T = 0, ties = 0;
    uint32_t my_gt = 0;  // this lane's share of its warp's keys above bin b1
    bool overflow = false;
    if (!take_all) {
        find_bin(cluster, sh, sh.hist[0], 2048, (uint32_t)k);
        const uint32_t b1 = sh.sel[0];
        uint32_t krem = sh.sel[1];
        // ---- pass 2: candidates of bin b1, count keys above it
        for (int cb = ws; cb < we; cb += 128) {
            uint32_t key[4];
            load4(rowp, cb + 4 * lane, we, vec, key);
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t d = key[e] >> 21;
                my_gt += key[e] && d > b1;
                const bool is_c = key[e] && d == b1;
                const uint32_t ball = __ballot_sync(0xffffffffu, is_c);
                if (ball) {
                    uint32_t base = 0;
                    if (lane == 0)
                        base = atomicAdd(&sh.ncand, (uint32_t)__popc(ball));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    const uint32_t pos = base + __popc(ball & ((1u << lane) - 1u));
                    if (is_c && pos < (uint32_t)kCandCap) {
                        sh.cand_key[pos] = key[e];
                        sh.cand_idx[pos] = cb + 4 * lane + e;
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
                for (int cb = ws; cb < we; cb += 128) {
                    uint32_t key[4];
                    load4(rowp, cb + 4 * lane, we, vec, key);
                    #pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (key[e] && (key[e] & pmask) == prefix)
                            atomicAdd(&h[(key[e] >> shift) & (uint32_t)(nb - 1)], 1u);
                }
            }
            cluster.sync();
            find_bin(cluster, sh, h, nb, krem);
            prefix |= sh.sel[0] << shift;
            pmask |= (uint32_t)(nb - 1) << shift;
            krem = sh.sel[1];
        }
        T = prefix;
        ties = krem;
    }

    // ---- per-warp counts of keys > T and == T (T = 0 when every valid key fits)
    uint32_t gt = 0, eq = 0;
    if (take_all || overflow) {
        for (int cb = ws; cb < we; cb += 128) {
            uint32_t key[4];
            load4(rowp, cb + 4 * lane, we, vec, key);
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                gt += key[e] > T;
                eq += key[e] == T && key[e];
            }
        }
        for (int o = 16; o > 0; o >>= 1) {
            gt += __shfl_xor_sync(0xffffffffu, gt, o);
            eq += __shfl_xor_sync(0xffffffffu, eq, o);
        }
        if (lane == 0) {
            sh.wgt[warp] = gt;
            sh.weq[warp] = eq;
        }
        __syncthreads();
    } else {
        for (int o = 16; o > 0; o >>= 1)
            my_gt += __shfl_xor_sync(0xffffffffu, my_gt, o);
        if (lane == 0) {
            sh.wgt[warp] = my_gt;
            sh.weq[warp] = 0;
        }
        __syncthreads();
        const uint32_t ncand = sh.ncand;
        for (uint32_t i = tid; i < ncand; i += kThreads) {
            const uint32_t kk = sh.cand_key[i];
            const int wi = wper > 0 ? (sh.cand_idx[i] - lo) / wper : 0;
            if (kk > T)
                atomicAdd(&sh.wgt[wi], 1u);
            else if (kk == T)
                atomicAdd(&sh.weq[wi], 1u);
        }
        __syncthreads();
    }
    // block prefix over warps (index order), then cluster prefix over CTAs
    if (tid == 0) {
        uint32_t g = 0, e = 0;
        for (int i = 0; i < kWarps; ++i) {
            g += sh.wgt[i];
            e += sh.weq[i];
        }
        sh.cta[1] = g;
        sh.cta[2] = e;
    }
    cluster.sync();
    uint32_t eq_before_cta = 0, sel_before_cta = 0, total_sel = 0, eq_run = 0;
    for (int r = 0; r < C; ++r) {
        const Shared *o = C == 1 ? &sh : cluster.map_shared_rank(&sh, r);
        const uint32_t g = o->cta[1], e = o->cta[2];
        const uint32_t take = eq_run >= ties ? 0u : min(e, ties - eq_run);
        if (r < crank) {
            sel_before_cta += g + take;
            eq_before_cta += e;
        }
        total_sel += g + take;
        eq_run += e;
    }
    // this warp's tie quota and output base
    uint32_t eq_before = eq_before_cta, base = sel_before_cta;
    for (int i = 0; i < warp; ++i) {
        const uint32_t e = sh.weq[i];
        const uint32_t take = eq_before >= ties ? 0u : min(e, ties - eq_before);
        base += sh.wgt[i] + take;
        eq_before += e;
    }
    const uint32_t quota = eq_before >= ties ? 0u : min(sh.weq[warp], ties - eq_before);

    // ---- pass 3: ordered write of the selection
    if (row_ok) {
        int32_t *orow = out + (size_t)row * ld_out;
        uint32_t written = 0, eq_seen = 0;
        for (int cb = ws; cb < we; cb += 128) {
            uint32_t key[4];
            load4(rowp, cb + 4 * lane, we, vec, key);
            uint32_t neq = 0;
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                neq += key[e] == T && key[e];
            uint32_t eq_pre = neq;  // exclusive prefix of ties over lanes
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t n = __shfl_up_sync(0xffffffffu, eq_pre, o);
                if (lane >= o)
                    eq_pre += n;
            }
            const uint32_t eq_tot = __shfl_sync(0xffffffffu, eq_pre, 31);
            eq_pre -= neq;
            uint32_t take[4], nt = 0, er = eq_seen + eq_pre;
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                bool t = key[e] > T;
                if (key[e] == T && key[e]) {
                    t = er < quota;
                    ++er;
                }
                take[e] = t;
                nt += t;
            }
            uint32_t pre = nt;
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t n = __shfl_up_sync(0xffffffffu, pre, o);
                if (lane >= o)
                    pre += n;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, pre, 31);
            pre -= nt;
            uint32_t pos = base + written + pre;
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (take[e])
                    orow[pos++] = cb + 4 * lane + e;
            written += tot;
            eq_seen += eq_tot;
        }
        for (int j = (int)total_sel + crank * kThreads + tid; j < k; j += C * kThreads)
            orow[j] = -1;
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

} // namespace topk_detail
} // namespace idx
