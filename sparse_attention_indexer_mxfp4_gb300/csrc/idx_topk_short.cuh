// idx_topk_short.cuh -- top-k over keys held in registers: the per-row
// top-k for rows of at most 8192 keys, and the selection core that the
// candidate top-k (idx_topk_cand.cuh) shares.
//
// Passage: vLLM page rocm_paged_mxfp4_indexer, _topk -- top-k over each
// row's [0, lengths[row]), -1 padding.  The design is our own.
//
// One CTA per row.  Thread t of NT holds KS runs of four keys, run s at
// order positions 4 NT s + 4 t + e (e < 4), so (s, warp, lane, e) is the
// order in which ties are broken and indices are written.  Radix select
// over the order-preserving keys with 11/11/10-bit digits: a shared
// histogram per digit (digits 2 and 3 count only the keys matching the
// digits found so far), each followed by a descending bin search.  One
// counting pass then fills (step, warp) tables of the keys above the k-th
// largest key T and of the keys equal to it; two warps scan them, and the
// ordered write ranks each key inside its warp and step by ballots.  Keys
// equal to T are taken first in order.  When every key equal to T is taken
// (the usual case) one table of the keys at or above T serves instead.  Phases are separated by CTA
// barriers only.
#pragma once

#include <cstdint>

#include "idx_topk.cuh"

namespace idx {
namespace regsel {

template <int NT, int KS>
struct Shared {
    static constexpr int kWarps = NT / 32;
    static constexpr int kTab = KS * kWarps;  // (step, warp) entries
    uint32_t hist[2][2048];
    uint32_t wvalid[kWarps];
    uint32_t wbin[3][kWarps];
    uint32_t sel[3][3];
    uint32_t gt[kTab];  // keys above T per (step, warp), then exclusive offsets
    uint32_t eq[kTab];  // keys equal to T per (step, warp), then exclusive offsets
};

// Descending-bin search over nb bins (nb = 2048 or 1024) whose counts
// count(b) returns: the bin where the count from the top reaches krem, the
// rank left inside it and the bin's count go to sel[0..2].  Writes wbin and
// sel only; two barriers.
template <int NT, class Count>
__device__ __forceinline__ void find_bin_of(Count count, int nb, uint32_t krem, uint32_t *wbin,
                                            uint32_t *sel)
{
    constexpr int MAXPER = 2048 / NT;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = nb / NT;
    uint32_t loc[MAXPER], lsum = 0;
    #pragma unroll
    for (int j = 0; j < MAXPER; ++j) {
        loc[j] = j < per ? count(nb - 1 - (tid * per + j)) : 0u;
        lsum += loc[j];
    }
    uint32_t wt;
    uint32_t before = topk_detail::warp_excl(lsum, lane, &wt);
    if (lane == 0)
        wbin[w] = wt;
    __syncthreads();
    {
        // the counts of the warps before this one: a scan of the per-warp
        // totals across the lanes (NT / 32 <= 32 of them)
        const uint32_t wv = lane < NT / 32 ? wbin[lane] : 0u;
        uint32_t unused;
        const uint32_t wex = topk_detail::warp_excl(wv, lane, &unused);
        before += __shfl_sync(0xffffffffu, wex, w);
    }
    #pragma unroll
    for (int j = 0; j < MAXPER; ++j) {
        if (j < per && before < krem && before + loc[j] >= krem) {
            sel[0] = (uint32_t)(nb - 1 - (tid * per + j));
            sel[1] = krem - before;
            sel[2] = loc[j];  // the bin's count
        }
        before += loc[j];
    }
    __syncthreads();
}

// find_bin_of over the histogram h[nb] in this CTA's shared memory.
template <int NT>
__device__ __forceinline__ void find_bin(const uint32_t *h, int nb, uint32_t krem,
                                         uint32_t *wbin, uint32_t *sel)
{
    find_bin_of<NT>([h](int b) -> uint32_t { return h[b]; }, nb, krem, wbin, sel);
}

// In-place exclusive scan of an N-entry table (N a multiple of 32) by one
// warp; returns the table's total.
template <int N>
__device__ __forceinline__ uint32_t scan_tab(uint32_t *tab, int lane)
{
    constexpr int E = N / 32;
    uint32_t v[E], sum = 0;
    #pragma unroll
    for (int e = 0; e < E; ++e) {
        v[e] = tab[E * lane + e];
        sum += v[e];
    }
    uint32_t tot;
    uint32_t run = topk_detail::warp_excl(sum, lane, &tot);
    #pragma unroll
    for (int e = 0; e < E; ++e) {
        tab[E * lane + e] = run;
        run += v[e];
    }
    return tot;
}

// Selects the k largest nonzero keys of the CTA (ties first in order) and
// writes index_of(s, e) of each at its rank in order to orow[0, k), -1
// after the last.  key[s][e] is the thread's key at order position
// 4 NT s + 4 tid + e; 0 marks an empty or non-finite entry, and every key of
// the steps s >= ns (the same in every thread) is empty, so the passes stop
// there.  Uses every thread of the CTA; begins by clearing the histograms.
template <int NT, int KS, class IndexOf>
__device__ __forceinline__ void select_write(Shared<NT, KS> &sh, const uint32_t (&key)[KS][4],
                                             int k, int32_t *orow, IndexOf index_of,
                                             int ns = KS)
{
    using S = Shared<NT, KS>;
    static_assert(S::kTab % 32 == 0, "tables are scanned 32 lanes wide");
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    for (int i = tid; i < 2 * 2048 / 4; i += NT)
        reinterpret_cast<uint4 *>(&sh.hist[0][0])[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    // digit 1 (top 11 bits) and the number of finite keys
    uint32_t nvalid = 0;
    #pragma unroll
    for (int s = 0; s < KS; ++s) {
        if (s >= ns)
            break;
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if (key[s][e]) {
                ++nvalid;
                atomicAdd(&sh.hist[0][key[s][e] >> 21], 1u);
            }
    }
    nvalid = __reduce_add_sync(0xffffffffu, nvalid);
    if (lane == 0)
        sh.wvalid[w] = nvalid;
    __syncthreads();
    uint32_t total = 0;
    #pragma unroll
    for (int i = 0; i < S::kWarps; ++i)
        total += sh.wvalid[i];

    // T: the k-th largest key (0 when every finite key is taken); ties: how
    // many keys equal to T are taken
    uint32_t T = 0u, ties = 0u;
    bool all_ties = true;  // every key equal to T is taken
    if (total > (uint32_t)k) {
        find_bin<NT>(sh.hist[0], 2048, (uint32_t)k, sh.wbin[0], sh.sel[0]);
        const uint32_t b1 = sh.sel[0][0];
        uint32_t krem = sh.sel[0][1];
        // A digit's threshold bin whose keys are all taken ends the search:
        // T is then the bin's lowest key and every key at or above it is
        // taken (the k-th largest key is alone in its 22-bit bin for most
        // rows of distinct values, so digit 3 is usually skipped).
        if (krem == sh.sel[0][2]) {
            T = b1 << 21;
            goto found;
        }
        // digit 2 (next 11 bits) of the keys in bin b1; digit 1's histogram
        // is cleared meanwhile for digit 3
        for (int i = tid; i < 1024 / 4; i += NT)
            reinterpret_cast<uint4 *>(sh.hist[0])[i] = make_uint4(0u, 0u, 0u, 0u);
        #pragma unroll
        for (int s = 0; s < KS; ++s) {
            if (s >= ns)
                break;
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (key[s][e] >> 21 == b1)
                    atomicAdd(&sh.hist[1][(key[s][e] >> 10) & 2047u], 1u);
        }
        __syncthreads();
        find_bin<NT>(sh.hist[1], 2048, krem, sh.wbin[1], sh.sel[1]);
        const uint32_t p2 = (b1 << 11) | sh.sel[1][0];  // the top 22 bits of T
        krem = sh.sel[1][1];
        if (krem == sh.sel[1][2]) {
            T = p2 << 10;
            goto found;
        }
        // digit 3 (low 10 bits) of the keys matching the top 22 bits
        #pragma unroll
        for (int s = 0; s < KS; ++s) {
            if (s >= ns)
                break;
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (key[s][e] >> 10 == p2)
                    atomicAdd(&sh.hist[0][key[s][e] & 1023u], 1u);
        }
        __syncthreads();
        find_bin<NT>(sh.hist[0], 1024, krem, sh.wbin[2], sh.sel[2]);
        T = (p2 << 10) | sh.sel[2][0];
        ties = sh.sel[2][1];
        all_ties = ties == sh.hist[0][T & 1023u];  // the keys equal to T
    }
found:
    const uint32_t lt = (1u << lane) - 1u;

    if (all_ties) {
        // every key at or above tmin is taken (tmin = 1 when every finite
        // key is): one table of taken counts per (step, warp)
        const uint32_t tmin = T == 0u ? 1u : T;
        #pragma unroll
        for (int s = 0; s < KS; ++s) {
            uint32_t n = 0;
            if (s < ns) {
                #pragma unroll
                for (int e = 0; e < 4; ++e)
                    n += key[s][e] >= tmin;
                n = __reduce_add_sync(0xffffffffu, n);
            }
            if (lane == 0)
                sh.gt[s * S::kWarps + w] = n;
        }
        __syncthreads();
        if (w == 0)
            scan_tab<S::kTab>(sh.gt, lane);
        __syncthreads();
        #pragma unroll
        for (int s = 0; s < KS; ++s) {
            if (s >= ns)
                break;
            bool tk[4];
            uint32_t tk_below = 0;
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                tk[e] = key[s][e] >= tmin;
                tk_below += __popc(__ballot_sync(0xffffffffu, tk[e]) & lt);
            }
            uint32_t pos = sh.gt[s * S::kWarps + w] + tk_below;
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (tk[e])
                    orow[pos++] = index_of(s, e);
        }
        const int nsel = (int)min(total, (uint32_t)k);
        for (int j = nsel + tid; j < k; j += NT)
            orow[j] = -1;
        return;
    }

    // counts of keys above and equal to T per (step, warp)
    #pragma unroll
    for (int s = 0; s < KS; ++s) {
        uint32_t ngt = 0, neq = 0;
        if (s < ns) {
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                ngt += key[s][e] > T;
                neq += key[s][e] == T;
            }
            ngt = __reduce_add_sync(0xffffffffu, ngt);
            neq = __reduce_add_sync(0xffffffffu, neq);
        }
        if (lane == 0) {
            sh.gt[s * S::kWarps + w] = ngt;
            sh.eq[s * S::kWarps + w] = neq;
        }
    }
    __syncthreads();
    if (w == 0)
        scan_tab<S::kTab>(sh.gt, lane);
    else if (w == 1)
        scan_tab<S::kTab>(sh.eq, lane);
    __syncthreads();

    // ordered write: the keys of (step, warp) start after the keys above T
    // before it and the keys equal to T taken before it
    #pragma unroll
    for (int s = 0; s < KS; ++s) {
        if (s >= ns)
            break;
        const uint32_t eq0 = sh.eq[s * S::kWarps + w];
        uint32_t eq_below = 0;
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            eq_below += __popc(__ballot_sync(0xffffffffu, key[s][e] == T) & lt);
        bool tk[4];
        uint32_t mine_eq = 0;
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool is_eq = key[s][e] == T;
            tk[e] = key[s][e] > T || (is_eq && eq0 + eq_below + mine_eq < ties);
            mine_eq += is_eq;
        }
        uint32_t tk_below = 0;
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            tk_below += __popc(__ballot_sync(0xffffffffu, tk[e]) & lt);
        uint32_t pos = sh.gt[s * S::kWarps + w] + min(eq0, ties) + tk_below;
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if (tk[e])
                orow[pos++] = index_of(s, e);
    }
    const int nsel = (int)min(total, (uint32_t)k);
    for (int j = nsel + tid; j < k; j += NT)
        orow[j] = -1;
}

} // namespace regsel

namespace topk_short {

constexpr int kThreads = 256;
constexpr int kSteps = 8;                       // runs of four keys per thread
constexpr int kMaxLen = kSteps * kThreads * 4;  // 8192

// Rows of at most 8192 keys; thread t holds elements 1024 s + 4 t + e.
__global__ void __launch_bounds__(kThreads, 3)
    topk_short_kernel(const float *__restrict__ logits, int64_t ld, int rows,
                      const int32_t *__restrict__ lengths, int k, int32_t *__restrict__ out,
                      int64_t ld_out, int vec_ok)
{
    __shared__ __align__(16) regsel::Shared<kThreads, kSteps> sh;
    const int row = blockIdx.x, tid = threadIdx.x;
    pdl_wait();  // the logits and lengths may come from the kernel before this one
    pdl_launch_dependents();
    if (row >= rows)
        return;
    const int len = max(0, min(lengths[row], (int)ld));
    const int nrun = (len + 4 * kThreads - 1) / (4 * kThreads);  // runs holding keys
    uint32_t key[kSteps][4];
    topk_detail::load_keys<kSteps>(logits + (size_t)row * ld, 4 * tid, 4 * kThreads, len,
                                   vec_ok != 0, key, nrun);
    regsel::select_write<kThreads, kSteps>(
        sh, key, k, out + (size_t)row * ld_out,
        [&](int s, int e) -> int32_t { return s * 4 * kThreads + 4 * tid + e; }, nrun);
}

} // namespace topk_short
} // namespace idx
