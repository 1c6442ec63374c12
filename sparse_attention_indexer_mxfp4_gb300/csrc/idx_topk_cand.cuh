// idx_topk_cand.cuh -- per-row top-k restricted to a row's candidate blocks.
//
// Passage: vLLM page rocm_paged_mxfp4_indexer, _topk (top-k over a row's
// live keys, -1 padding) applied after the candidate mask of page
// rocm_aiter_mla_sparse, _apply_candidate_mask_strided: only keys of the
// row's candidate blocks [ks + id * blk, ks + (id + 1) * blk) within
// [ks, ke) can be selected, so only those are read.  The design is our own.
//
// One CTA of 512 threads per row.  The row's candidate ids are sorted and
// deduplicated in shared memory; the keys of the candidate blocks, in
// ascending id order (so compact position order is ascending token order),
// are loaded straight into registers, four consecutive compact positions
// per run, and the register selection of idx_topk_short.cuh picks the k
// largest and writes their token indices in order.  Keys outside [ks, ke),
// non-finite values and duplicate ids read as key 0 and are never selected;
// ties at the k-th value go to the lowest token index.
#pragma once

#include <cstdint>

#include "idx_topk_short.cuh"

namespace idx {
namespace topk_cand {

constexpr int kThreads = 512;
constexpr int kMaxIds = 512;     // candidate ids per row
constexpr int kMaxKeys = 16384;  // num_cand * block_size
constexpr int kStepsSmall = 4;   // runs per thread up to 8192 keys
constexpr int kStepsLarge = 8;   // up to 16384 keys

template <int KS>
struct Shared {
    int32_t raw[kMaxIds];  // the ids as given
    int32_t ids[kMaxIds];  // sorted, -1 for duplicates and invalid ids
    regsel::Shared<kThreads, KS> sel;
};

template <int KS>
__global__ void __launch_bounds__(kThreads, KS == kStepsSmall ? 2 : 1)
    topk_cand_kernel(const float *__restrict__ logits, int64_t ld, int rows,
                     const int32_t *__restrict__ lengths, const int32_t *__restrict__ row_ks,
                     const int32_t *__restrict__ cand, int64_t cand_stride, int num_cand,
                     int blk, int row_repeat, int k, int32_t *__restrict__ out, int64_t ld_out,
                     int vec4)
{
    __shared__ __align__(16) Shared<KS> sh;
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
    for (int i = tid; i < n; i += kThreads)
        sh.raw[i] = crow[i];
    __syncthreads();
    const int id_end = (ke - ks + blk - 1) / blk;  // ids [0, id_end) start below ke
    auto sort_key = [&](int id) -> unsigned {
        return id >= 0 && id < id_end ? (unsigned)id : 0xFFFFFFFFu;
    };
    if (n <= kThreads / 8) {
        // eight lanes per id, each comparing it with every eighth id, their
        // counts added across the eight lanes (which share a warp)
        const int i = tid >> 3, sub = tid & 7;
        int rank = 0, dup = 0, id = -1;
        if (i < n) {
            id = sh.raw[i];
            const unsigned key_i = sort_key(id);
            for (int j = sub; j < n; j += 8) {
                const unsigned key_j = sort_key(sh.raw[j]);
                rank += key_j < key_i || (key_j == key_i && j < i);
                dup |= key_j == key_i && j < i;
            }
        }
        #pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            rank += __shfl_xor_sync(0xffffffffu, rank, o);
            dup |= __shfl_xor_sync(0xffffffffu, dup, o);
        }
        if (i < n && sub == 0)
            sh.ids[rank] = sort_key(id) != 0xFFFFFFFFu && !dup ? id : -1;
    } else {
        for (int i = tid; i < n; i += kThreads) {
            const int id = sh.raw[i];
            const unsigned key_i = sort_key(id);
            int rank = 0;
            bool dup = false;
            for (int j = 0; j < n; ++j) {
                const unsigned key_j = sort_key(sh.raw[j]);
                rank += key_j < key_i || (key_j == key_i && j < i);
                dup = dup || (key_j == key_i && j < i);
            }
            sh.ids[rank] = key_i != 0xFFFFFFFFu && !dup ? id : -1;
        }
    }
    __syncthreads();

    // token of compact position q (-1: no key there)
    auto token_of = [&](int q) -> int {
        if (q >= nkeys)
            return -1;
        const int e = blk_of(q), id = sh.ids[e];
        return id >= 0 ? ks + id * blk + (q - e * blk) : -1;
    };

    // the keys of compact positions 4 (kThreads s + tid) + c, every load of
    // the thread issued before any key is formed
    const float *rowp = logits + (size_t)r * ld;
    uint32_t key[KS][4];
    {
        float4 v[KS];
        const bool vec = vec4 && (ks & 3) == 0;  // blocks and the row start are 16-byte aligned
        #pragma unroll
        for (int s = 0; s < KS; ++s) {
            const int q = 4 * (kThreads * s + tid);
            v[s] = make_float4(NAN, NAN, NAN, NAN);
            const int t = token_of(q);
            if (vec) {
                if (t >= 0 && t + 3 < ke)
                    v[s] = __ldg(reinterpret_cast<const float4 *>(rowp + t));
            } else if (t >= 0 && t < ke) {
                v[s].x = __ldg(rowp + t);
            }
        }
        #pragma unroll
        for (int s = 0; s < KS; ++s) {
            const int q = 4 * (kThreads * s + tid);
            float x[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
            const int t = token_of(q);
            if (vec) {
                if (t >= 0 && t < ke && t + 3 >= ke)  // the row ends inside this run
                    for (int c = 0; c < 4; ++c)
                        x[c] = t + c < ke ? __ldg(rowp + t + c) : NAN;
            } else {
                for (int c = 1; c < 4; ++c) {
                    const int tc = token_of(q + c);
                    x[c] = tc >= 0 && tc < ke ? __ldg(rowp + tc) : NAN;
                }
            }
            #pragma unroll
            for (int c = 0; c < 4; ++c)
                key[s][c] = topk_detail::float_key(x[c]);
        }
    }

    regsel::select_write<kThreads, KS>(
        sh.sel, key, k, out + (size_t)r * ld_out,
        [&](int s, int e) -> int32_t { return token_of(4 * (kThreads * s + tid) + e); });
}

} // namespace topk_cand
} // namespace idx
