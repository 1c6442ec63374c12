// idx_topk_cand.cuh -- per-row top-k restricted to a row's candidate blocks.
//
// Passage: vLLM page rocm_paged_mxfp4_indexer, _topk (top-k over a row's
// live keys, -1 padding) applied after the candidate mask of page
// rocm_aiter_mla_sparse, _apply_candidate_mask_strided: only keys of the
// row's candidate blocks [ks + id * blk, ks + (id + 1) * blk) within
// [ks, ke) can be selected, so only those are read.  The design is our own.
//
// One CTA per row.  The row's candidate ids are sorted and deduplicated in
// shared memory, the keys of the candidate blocks are gathered into shared
// memory in ascending id order (so that order is ascending token order), and
// the 11/11/10-bit radix select of idx_topk.cuh runs there: a histogram per
// digit over the shared keys, then an ordered write ranked by warp ballots.  Keys outside [ks, ke), non-finite values and
// duplicate ids read as key 0 and are never selected; ties at the k-th value
// go to the lowest token index.
#pragma once

#include <cstdint>

#include "idx_topk.cuh"

namespace idx {
namespace topk_cand {

constexpr int kThreads = 512;
constexpr int kMaxIds = 512;        // candidate ids per row
constexpr int kMaxKeys = 16384;     // num_cand * block_size
constexpr int kWarps = kThreads / 32;
constexpr int kSteps = kMaxKeys / kThreads;

struct Shared {
    uint32_t keys[kMaxKeys];
    int32_t ids[kMaxIds];    // sorted, -1 for duplicates and invalid ids
    uint32_t hist[2048];
    uint32_t wsum[kThreads / 32];
    uint32_t sel[2];
    uint32_t tab[(kMaxKeys / kThreads) * (kThreads / 32)];    // (step, warp) taken counts
    uint32_t eqtab[(kMaxKeys / kThreads) * (kThreads / 32)];  // (step, warp) counts of T
};

// Descending-bin search over hist[nb] (nb <= 2048, kThreads threads, 4 bins
// each): the bin where the count from the top reaches krem and the rank left
// in it go to sel[0..1].  Barriers on both sides.
__device__ __forceinline__ void find_bin(Shared &sh, int nb, uint32_t krem)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    uint32_t loc[4], lsum = 0;
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int b = nb - 1 - (tid * 4 + j);
        loc[j] = b >= 0 ? sh.hist[b] : 0u;
        lsum += loc[j];
    }
    uint32_t wt;
    const uint32_t ex = topk_detail::warp_excl(lsum, lane, &wt);
    __syncthreads();
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

// Exclusive prefix of v over the CTA; *tot gets the total.
__device__ __forceinline__ uint32_t block_excl(Shared &sh, uint32_t v, uint32_t *tot)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t wt;
    const uint32_t ex = topk_detail::warp_excl(v, lane, &wt);
    __syncthreads();
    if (lane == 0)
        sh.wsum[w] = wt;
    __syncthreads();
    uint32_t off = ex, t = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
        if (i < w)
            off += sh.wsum[i];
        t += sh.wsum[i];
    }
    __syncthreads();
    *tot = t;
    return off;
}

// Exclusive scan, in place, of the first nsteps * kWarps entries of a
// (step, warp) table by warp 0; returns the total.  Barriers on both sides.
__device__ __forceinline__ uint32_t scan_table(Shared &sh, uint32_t *tab, int nsteps)
{
    constexpr int E = kSteps * kWarps / 32;  // entries per lane
    __syncthreads();
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        const int n = nsteps * kWarps;
        uint32_t v[E], sum = 0;
        #pragma unroll
        for (int e = 0; e < E; ++e) {
            const int idx = lane * E + e;
            v[e] = idx < n ? tab[idx] : 0u;
            sum += v[e];
        }
        uint32_t tot;
        uint32_t run = topk_detail::warp_excl(sum, lane, &tot);
        #pragma unroll
        for (int e = 0; e < E; ++e) {
            const int idx = lane * E + e;
            if (idx < n)
                tab[idx] = run;
            run += v[e];
        }
        if (lane == 0)
            sh.sel[0] = tot;
    }
    __syncthreads();
    const uint32_t t = sh.sel[0];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(kThreads, 2)
    topk_cand_kernel(const float *__restrict__ logits, int64_t ld, int rows,
                     const int32_t *__restrict__ lengths, const int32_t *__restrict__ row_ks,
                     const int32_t *__restrict__ cand, int64_t cand_stride, int num_cand,
                     int blk, int row_repeat, int k, int32_t *__restrict__ out, int64_t ld_out,
                     int vec4)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    Shared &sh = *reinterpret_cast<Shared *>(dsm);
    const int r = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    const int ke = max(0, min(lengths[r], (int)ld));
    const int ks = row_ks ? max(0, min(row_ks[r], ke)) : 0;
    const int32_t *crow = cand + (size_t)(r / row_repeat) * cand_stride;
    const int n = num_cand;
    const int nkeys = n * blk;
    // block of compact position q: a shift for power-of-two blocks
    const int bsh = (blk & (blk - 1)) == 0 ? __ffs(blk) - 1 : -1;
    auto blk_of = [&](int q) -> int { return bsh >= 0 ? q >> bsh : q / blk; };

    // sort the ids (rank = ids before it in (id, position) order); a
    // repeated id keeps its first copy, invalid ids (negative, or a block
    // starting at or past ke) become -1 at the end of the order
    int32_t *raw = reinterpret_cast<int32_t *>(sh.keys);  // the ids as given, until the gather
    for (int i = tid; i < n; i += kThreads)
        raw[i] = crow[i];
    __syncthreads();
    const int id_end = (ke - ks + blk - 1) / blk;  // ids [0, id_end) start below ke
    for (int i = tid; i < n; i += kThreads) {
        const int id = raw[i];
        const bool valid = id >= 0 && id < id_end;
        const unsigned key_i = valid ? (unsigned)id : 0xFFFFFFFFu;
        int rank = 0;
        bool dup = false;
        for (int j = 0; j < n; ++j) {
            const int idj = raw[j];
            const unsigned key_j = idj >= 0 && idj < id_end ? (unsigned)idj : 0xFFFFFFFFu;
            rank += key_j < key_i || (key_j == key_i && j < i);
            dup = dup || (key_j == key_i && j < i);
        }
        sh.ids[rank] = valid && !dup ? id : -1;
    }
    __syncthreads();

    // gather the candidate blocks' keys in sorted order; every load of the
    // thread is issued before any key is formed
    const float *rowp = logits + (size_t)r * ld;
    if (vec4 && (ks & 3) == 0) {
        // four keys per load: blocks and the row start are 16-byte aligned
        constexpr int NV = kMaxKeys / 4 / kThreads;
        float4 v[NV];
        #pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int q = 4 * (tid + i * kThreads);
            v[i] = make_float4(NAN, NAN, NAN, NAN);
            if (q < nkeys) {
                const int e = blk_of(q), o = q - e * blk;
                const int id = sh.ids[e];
                const long long t = (long long)ks + (long long)id * blk + o;
                if (id >= 0 && t + 3 < ke)
                    v[i] = __ldg(reinterpret_cast<const float4 *>(rowp + t));
            }
        }
        #pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int q = 4 * (tid + i * kThreads);
            if (q < nkeys) {
                const int e = blk_of(q), o = q - e * blk;
                const int id = sh.ids[e];
                const long long t = (long long)ks + (long long)id * blk + o;
                float x[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                if (id >= 0 && t < ke && t + 3 >= ke)  // the row ends inside this group
                    for (int c = 0; c < 4; ++c)
                        x[c] = t + c < ke ? __ldg(rowp + t + c) : NAN;
                #pragma unroll
                for (int c = 0; c < 4; ++c)
                    sh.keys[q + c] = topk_detail::float_key(x[c]);
            }
        }
    } else {
        constexpr int NS = kMaxKeys / kThreads;
        float x[NS];
        #pragma unroll
        for (int i = 0; i < NS; ++i) {
            const int q = tid + i * kThreads;
            x[i] = NAN;
            if (q < nkeys) {
                const int e = blk_of(q), o = q - e * blk;
                const int id = sh.ids[e];
                const long long t = (long long)ks + (long long)id * blk + o;
                if (id >= 0 && t < ke)
                    x[i] = __ldg(rowp + t);
            }
        }
        #pragma unroll
        for (int i = 0; i < NS; ++i) {
            const int q = tid + i * kThreads;
            if (q < nkeys)
                sh.keys[q] = topk_detail::float_key(x[i]);
        }
    }
    for (int i = tid; i < 2048; i += kThreads)
        sh.hist[i] = 0u;
    __syncthreads();

    // digit 1 and the number of finite keys
    uint32_t nvalid = 0;
    for (int q = tid; q < nkeys; q += kThreads) {
        const uint32_t key = sh.keys[q];
        if (key) {
            ++nvalid;
            atomicAdd(&sh.hist[key >> 21], 1u);
        }
    }
    uint32_t total;
    block_excl(sh, nvalid, &total);  // its barriers also publish hist
    uint32_t T = 0u, ties = 0u;      // T = 0: every finite key is taken
    bool all_ties = true;
    if (total > (uint32_t)k) {
        find_bin(sh, 2048, (uint32_t)k);
        uint32_t prefix = sh.sel[0] << 21, pmask = 0xFFE00000u, krem = sh.sel[1];
        for (int pass = 1; pass < 3; ++pass) {
            const int shift = pass == 1 ? 10 : 0;
            const int nb = pass == 1 ? 2048 : 1024;
            for (int i = tid; i < 2048; i += kThreads)
                sh.hist[i] = 0u;
            __syncthreads();
            for (int q = tid; q < nkeys; q += kThreads) {
                const uint32_t key = sh.keys[q];
                if (key && (key & pmask) == prefix)
                    atomicAdd(&sh.hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
            }
            __syncthreads();
            find_bin(sh, nb, krem);
            prefix |= sh.sel[0] << shift;
            pmask |= (uint32_t)(nb - 1) << shift;
            krem = sh.sel[1];
        }
        T = prefix;
        ties = krem;
        all_ties = ties == sh.hist[T & 1023u];  // every key equal to T is taken
    }

    // Ordered write.  Step i covers keys [i * kThreads, (i + 1) * kThreads),
    // thread t key i * kThreads + t, so order is (step, warp, lane): a ballot
    // ranks a key inside its warp and step, and warp 0 scans the (step,
    // warp) counts.  Three light passes over the shared keys, ballots
    // recomputed rather than kept: count the keys equal to T, then the taken
    // keys (ties in index order up to the quota), then write.
    const int lane = tid & 31, w = tid >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    const int nsteps = (nkeys + kThreads - 1) / kThreads;
    auto key_at = [&](int i) -> uint32_t {
        const int q = i * kThreads + tid;
        return q < nkeys ? sh.keys[q] : 0u;
    };
    // pass 0 (only when some key equal to T is left out): keys equal to T
    if (!all_ties) {
        for (int i = 0; i < nsteps; ++i) {
            const uint32_t b = __ballot_sync(0xffffffffu, key_at(i) == T);
            if (lane == 0)
                sh.eqtab[i * kWarps + w] = __popc(b);
        }
        scan_table(sh, sh.eqtab, nsteps);
    }
    // every lane reaches the ballot: all_ties and T are the same CTA-wide
    const uint32_t tmin = T == 0u ? 1u : T;  // T = 0: every finite (nonzero) key
    auto taken = [&](int i, uint32_t key) -> bool {
        if (all_ties)
            return key >= tmin;
        const uint32_t eb = __ballot_sync(0xffffffffu, key == T);
        return key > T || (key == T && sh.eqtab[i * kWarps + w] + __popc(eb & lt) < ties);
    };
    // pass 1: taken keys
    for (int i = 0; i < nsteps; ++i) {
        const uint32_t b = __ballot_sync(0xffffffffu, taken(i, key_at(i)));
        if (lane == 0)
            sh.tab[i * kWarps + w] = __popc(b);
    }
    const uint32_t sel_tot = scan_table(sh, sh.tab, nsteps);
    // pass 2: write
    for (int i = 0; i < nsteps; ++i) {
        const uint32_t key = key_at(i);
        const bool t = taken(i, key);
        const uint32_t b = __ballot_sync(0xffffffffu, t);
        if (t) {
            const int q = i * kThreads + tid;
            const int e = blk_of(q), o = q - e * blk;
            out[(size_t)r * ld_out + sh.tab[i * kWarps + w] + __popc(b & lt)] =
                ks + sh.ids[e] * blk + o;
        }
    }
    int32_t *orow = out + (size_t)r * ld_out;
    for (int j = (int)sel_tot + tid; j < k; j += kThreads)
        orow[j] = -1;
}

} // namespace topk_cand
} // namespace idx
