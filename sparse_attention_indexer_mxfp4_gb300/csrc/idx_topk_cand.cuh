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
// digit over the shared keys, then one ordered write in which thread t owns
// a contiguous run of keys.  Keys outside [ks, ke), non-finite values and
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
constexpr int kPer = kMaxKeys / kThreads;  // keys a thread owns in the ordered write

struct Shared {
    uint32_t keys[kMaxKeys];
    int32_t ids[kMaxIds];    // sorted, -1 for duplicates and invalid ids
    uint32_t hist[2048];
    uint32_t wsum[kThreads / 32];
    uint32_t sel[2];
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

__global__ void __launch_bounds__(kThreads, 1)
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

    // sort the ids (rank = ids before it in (id, position) order); a
    // repeated id keeps its first copy, invalid ids (negative, or a block
    // starting at or past ke) become -1 at the end of the order
    int32_t *raw = reinterpret_cast<int32_t *>(sh.keys);  // the ids as given, until the gather
    for (int i = tid; i < n; i += kThreads)
        raw[i] = crow[i];
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
        int id = raw[i];
        const bool valid = id >= 0 && (long long)ks + (long long)id * blk < ke;
        const long long key_i = valid ? (long long)id : (1LL << 40);
        int rank = 0;
        bool dup = false;
        for (int j = 0; j < n; ++j) {
            const int idj = raw[j];
            const bool vj = idj >= 0 && (long long)ks + (long long)idj * blk < ke;
            const long long key_j = vj ? (long long)idj : (1LL << 40);
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
                const int e = q / blk, o = q - e * blk;
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
                const int e = q / blk, o = q - e * blk;
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
                const int e = q / blk, o = q - e * blk;
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
    }

    // ordered write: thread t owns keys [t * per, (t + 1) * per)
    const int per = (nkeys + kThreads - 1) / kThreads;
    const int q0 = min(nkeys, tid * per), q1 = min(nkeys, q0 + per);
    uint32_t neq = 0;
    for (int q = q0; q < q1; ++q)
        neq += T != 0u && sh.keys[q] == T;
    uint32_t eq_tot;
    uint32_t eq_rank = block_excl(sh, neq, &eq_tot);
    uint32_t nsel = 0;
    for (int q = q0; q < q1; ++q) {
        const uint32_t key = sh.keys[q];
        if (T == 0u) {
            nsel += key != 0u;
        } else if (key > T) {
            ++nsel;
        } else if (key == T) {
            nsel += eq_rank < ties;
            ++eq_rank;
        }
    }
    uint32_t sel_tot;
    uint32_t pos = block_excl(sh, nsel, &sel_tot);
    eq_rank -= neq;  // back to this thread's first tie rank
    int32_t *orow = out + (size_t)r * ld_out;
    for (int q = q0; q < q1; ++q) {
        const uint32_t key = sh.keys[q];
        bool take;
        if (T == 0u) {
            take = key != 0u;
        } else if (key > T) {
            take = true;
        } else if (key == T) {
            take = eq_rank < ties;
            ++eq_rank;
        } else {
            take = false;
        }
        if (take) {
            const int e = q / blk, o = q - e * blk;
            orow[pos++] = ks + sh.ids[e] * blk + o;
        }
    }
    for (int j = (int)sel_tot + tid; j < k; j += kThreads)
        orow[j] = -1;
}

} // namespace topk_cand
} // namespace idx
