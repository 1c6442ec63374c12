// idx_topk_cluster.cuh -- per-row top-k for rows of up to 262144 keys, one
// thread-block cluster per row, the row's keys in the cluster's shared
// memory.
//
// Passage: vLLM page rocm_paged_mxfp4_indexer, _topk -- top-k over each
// row's [0, lengths[row]), -1 padding.  The design is our own.
//
// A row's keys [0, len) are cut into C equal chunks (a multiple of four keys
// each, at most 32768); chunk c goes to the cluster's CTA of rank c
// (clusters of C = ceil(ld / 32768) <= 8 CTAs of 1024 threads, one CTA per
// SM by its shared memory), so a row shorter than the width still spreads
// over the whole cluster.  Every CTA keeps its chunk as order-preserving keys
// in shared memory, thread t holding positions 4 (1024 s + t) + e of the
// chunk (s < 8, e < 4), so (rank, s, warp, lane, e) is index order; every
// pass visits only the runs s that hold keys of the CTA's chunk.  The
// 11/11/10-bit radix select runs on histograms each CTA builds over its own
// keys; after a cluster barrier every CTA's bin search adds up the C
// histograms of the digit through distributed shared memory, bin by bin as
// it scans, and finds the same bin itself, so no reduction step or second
// barrier is needed per digit.  The write ranks
// keys by (step, warp) tables inside the CTA, offset by the counts of the
// lower-ranked CTAs (read remotely after one more barrier); keys equal to
// the k-th largest are taken lowest index first across the whole row.
// Every barrier is reached by every thread of every CTA of the cluster
// (the branches around them depend only on cluster-wide values), and the
// last one keeps each CTA's shared memory alive until the others have read
// it.
#pragma once

#include <cooperative_groups.h>
#include <cstdint>

#include "idx_topk_short.cuh"

namespace idx {
namespace topk_cluster {

namespace cg = cooperative_groups;

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSteps = 8;                        // runs of four keys per thread
constexpr int kChunk = kSteps * kThreads * 4;    // 32768 keys per CTA
constexpr int kMaxCluster = 8;                   // portable cluster size
constexpr int kMaxLen = kChunk * kMaxCluster;    // 262144
constexpr int kTab = kSteps * kWarps;            // (step, warp) entries
constexpr int kBtStage = 2048;                   // block-table entries staged per CTA

struct Shared {
    uint4 keys[kChunk / 4];
    uint32_t h1[2048];  // this CTA's digit histograms, read by the cluster
    uint32_t h2[2048];
    uint32_t h3[1024];
    uint32_t wbin[3][kWarps];
    uint32_t sel[3][3];
    uint32_t wred[kWarps];
    uint32_t cta[3];    // this CTA's finite keys, keys above T, keys equal to T
    uint32_t gt[kTab];  // keys above T (or taken) per (step, warp), then offsets
    uint32_t eq[kTab];  // keys equal to T per (step, warp), then offsets
    int32_t bts[kBtStage];  // (slot count) the chunk's pages' block-table entries
};

// Sum over the CTA of one value per thread (every thread gets it); one
// barrier.  Called once per launch, so its scratch is never reused.
__device__ __forceinline__ uint32_t cta_sum(Shared &sh, uint32_t v)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = __reduce_add_sync(0xffffffffu, v);
    if (lane == 0)
        sh.wred[w] = v;
    __syncthreads();
    static_assert(kWarps == 32, "one warp total per lane");
    return __reduce_add_sync(0xffffffffu, sh.wred[lane]);
}

// The bin search over the sum of every cluster CTA's histogram h (read
// through distributed shared memory; each thread sums only the bins it
// scans, so no merged copy and no barrier before the search).
__device__ __forceinline__ void find_bin_cluster(cg::cluster_group &cl, Shared &sh, uint32_t *h,
                                                 int nb, uint32_t krem, int C, int digit)
{
    regsel::find_bin_of<kThreads>(
        [&](int b) -> uint32_t {
            uint32_t v = 0;
            for (int r = 0; r < C; ++r)
                v += cl.map_shared_rank(h, r)[b];
            return v;
        },
        nb, krem, sh.wbin[digit], sh.sel[digit]);
}

__global__ void __launch_bounds__(kThreads, 1)
    topk_cluster_kernel(const float *__restrict__ logits, int64_t ld, int rows,
                        const int32_t *__restrict__ lengths, int k, int32_t *__restrict__ out,
                        int64_t ld_out, int vec_ok, const SlotCount sc)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    Shared &sh = *reinterpret_cast<Shared *>(dsm);
    cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks();
    const int rank = (int)cl.block_rank();
    const int row = blockIdx.x / C;  // the grid holds whole clusters: uniform per cluster
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const bool live = row < rows;
    for (int i = tid; i < 2048 + 2048 + 1024; i += kThreads)
        (i < 2048 ? sh.h1[i] : i < 4096 ? sh.h2[i - 2048] : sh.h3[i - 4096]) = 0u;
    pdl_wait();  // the logits and lengths may come from the kernel before this one
    pdl_launch_dependents();
    // the row's slot count starts at 0 (ordered before every CTA's addition
    // by the cluster barriers between)
    if (sc.bt && live && rank == 0 && tid == 0)
        sc.lens[row] = 0;
    const int len = live ? max(0, min(lengths[row], (int)ld)) : 0;
    // the row's keys spread evenly over the cluster, whole quads per CTA (the
    // chunk starts stay 16-byte aligned for vector loads)
    const int per = min(kChunk, ((len + C - 1) / C + 3) & ~3);
    const int base = rank * per;
    const int end = max(0, min(len - base, per));        // keys of this CTA's chunk
    const int nrun = (end + 4 * kThreads - 1) / (4 * kThreads);  // runs holding them
    const float *rowp = logits + (size_t)(live ? row : 0) * ld + base;
    // (slot count) the block-table entries of the chunk's pages go to shared
    // memory while the keys load, when they fit (-1 past max_blocks)
    const int seq = sc.bt && live ? (sc.row_to_seq ? __ldg(sc.row_to_seq + row) : row / sc.next_n)
                                  : 0;
    int bt_lo = 0;
    bool bt_staged = false;
    if (sc.bt && live && end > 0) {
        const int lo = sc.shift >= 0 ? base >> sc.shift : base / sc.P;
        const int hi = sc.shift >= 0 ? (base + end - 1) >> sc.shift : (base + end - 1) / sc.P;
        if (hi - lo < kBtStage) {
            bt_staged = true;
            bt_lo = lo;
            const int32_t *btrow = sc.bt + (size_t)seq * sc.bt_stride;
            for (int i = tid; i <= hi - lo; i += kThreads)
                sh.bts[i] = lo + i < sc.max_blocks ? __ldg(btrow + lo + i) : -1;
        }
    }

    // keys of this chunk into shared memory, the local digit-1 histogram
    // from them as they are formed (the histograms were cleared above)
    uint32_t nvalid = 0;
    {
        uint32_t key[kSteps][4];
        topk_detail::load_keys<kSteps>(rowp, 4 * tid, 4 * kThreads, end, vec_ok != 0, key, nrun);
        __syncthreads();
        #pragma unroll
        for (int s = 0; s < kSteps; ++s) {
            if (s >= nrun)
                break;
            sh.keys[s * kThreads + tid] = make_uint4(key[s][0], key[s][1], key[s][2], key[s][3]);
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (key[s][e]) {
                    ++nvalid;
                    atomicAdd(&sh.h1[key[s][e] >> 21], 1u);
                }
        }
    }
    // the thread's run s of keys, from shared memory (only this thread writes it)
    auto run = [&](int s) -> uint4 { return sh.keys[s * kThreads + tid]; };
    nvalid = cta_sum(sh, nvalid);
    if (tid == 0)
        sh.cta[0] = nvalid;
    cl.sync();  // histograms and counts of digit 1 complete in every CTA

    uint32_t total = 0;
    for (int r = 0; r < C; ++r)
        total += cl.map_shared_rank(sh.cta, r)[0];

    // T: the k-th largest key; every key at or above it is taken unless
    // some_ties (then keys equal to T are taken lowest index first, ties of
    // eq_total of them).  A digit's threshold bin whose keys are all taken
    // ends the search with T its lowest key (the usual case after digit 2
    // for rows of distinct values).  Every branch is cluster-uniform.
    uint32_t T = 0u, ties = 0u, eq_total = 0u;
    bool some_ties = false;
    if (total > (uint32_t)k) {
        find_bin_cluster(cl, sh, sh.h1, 2048, (uint32_t)k, C, 0);
        const uint32_t b1 = sh.sel[0][0];
        uint32_t krem = sh.sel[0][1];
        if (krem == sh.sel[0][2]) {
            T = b1 << 21;
            goto found;
        }
        #pragma unroll
        for (int s = 0; s < kSteps; ++s) {
            if (s >= nrun)
                break;
            const uint4 v = run(s);
            const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (kk[e] >> 21 == b1)
                    atomicAdd(&sh.h2[(kk[e] >> 10) & 2047u], 1u);
        }
        cl.sync();  // digit-2 histograms complete
        find_bin_cluster(cl, sh, sh.h2, 2048, krem, C, 1);
        const uint32_t p2 = (b1 << 11) | sh.sel[1][0];
        krem = sh.sel[1][1];
        if (krem == sh.sel[1][2]) {
            T = p2 << 10;
            goto found;
        }
        #pragma unroll
        for (int s = 0; s < kSteps; ++s) {
            if (s >= nrun)
                break;
            const uint4 v = run(s);
            const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (kk[e] >> 10 == p2)
                    atomicAdd(&sh.h3[kk[e] & 1023u], 1u);
        }
        cl.sync();  // digit-3 histograms complete
        find_bin_cluster(cl, sh, sh.h3, 1024, krem, C, 2);
        T = (p2 << 10) | sh.sel[2][0];
        ties = sh.sel[2][1];
        eq_total = sh.sel[2][2];
        some_ties = ties != eq_total;
    }
found:
    const bool all_ties = !some_ties;  // every key at or above tmin is taken
    const uint32_t tmin = T == 0u ? 1u : T;

    // per (step, warp): keys taken outright (above T, or at or above tmin
    // when every key equal to T is taken) and keys equal to T
    #pragma unroll
    for (int s = 0; s < kSteps; ++s) {
        if (s >= nrun) {  // runs without keys count nothing
            if (lane == 0) {
                sh.gt[s * kWarps + w] = 0u;
                sh.eq[s * kWarps + w] = 0u;
            }
            continue;
        }
        const uint4 v = run(s);
        const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
        uint32_t ngt = 0, neq = 0;
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
            ngt += all_ties ? kk[e] >= tmin : kk[e] > T;
            neq += kk[e] == T;
        }
        ngt = __reduce_add_sync(0xffffffffu, ngt);
        neq = __reduce_add_sync(0xffffffffu, neq);
        if (lane == 0) {
            sh.gt[s * kWarps + w] = ngt;
            sh.eq[s * kWarps + w] = neq;
        }
    }
    __syncthreads();
    if (w == 0) {
        const uint32_t a = regsel::scan_tab<kTab>(sh.gt, lane);
        if (lane == 0)
            sh.cta[1] = a;
    } else if (w == 1) {
        const uint32_t a = regsel::scan_tab<kTab>(sh.eq, lane);
        if (lane == 0)
            sh.cta[2] = a;
    }
    cl.sync();  // every CTA's counts are published

    // offsets of this CTA: the taken keys and the keys equal to T of the
    // lower-ranked CTAs
    uint32_t gt_before = 0, eq_before = 0;
    for (int r = 0; r < rank; ++r) {
        const uint32_t *c = cl.map_shared_rank(sh.cta, r);
        gt_before += c[1];
        eq_before += c[2];
    }
    // the last reads of other CTAs' shared memory are done: arrive at the
    // barrier that keeps each CTA's shared memory alive until then (waited
    // on at the end, so the writes below overlap it)
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    const uint32_t lt = (1u << lane) - 1u;
    int32_t *orow = out + (size_t)(live ? row : 0) * ld_out;
    uint32_t nslot = 0, nbad = 0;  // valid and invalid slots of this thread's taken keys
    if (live) {
        #pragma unroll
        for (int s = 0; s < kSteps; ++s) {
            if (s >= nrun)
                break;
            const uint4 v = run(s);
            const uint32_t key[4] = {v.x, v.y, v.z, v.w};
            const uint32_t eq0 = eq_before + sh.eq[s * kWarps + w];
            uint32_t eq_below = 0;
            if (!all_ties) {
                #pragma unroll
                for (int e = 0; e < 4; ++e)
                    eq_below += __popc(__ballot_sync(0xffffffffu, key[e] == T) & lt);
            }
            bool tk[4];
            uint32_t mine_eq = 0, tk_below = 0;
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool is_eq = key[e] == T;
                tk[e] = all_ties ? key[e] >= tmin
                                 : key[e] > T || (is_eq && eq0 + eq_below + mine_eq < ties);
                mine_eq += is_eq;
                tk_below += __popc(__ballot_sync(0xffffffffu, tk[e]) & lt);
            }
            uint32_t pos = gt_before + sh.gt[s * kWarps + w] +
                           (all_ties ? 0u : min(eq0, ties)) + tk_below;
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if (tk[e]) {
                    const int p = base + 4 * (s * kThreads + tid) + e;
                    orow[pos++] = p;
                    if (sc.bt) {
                        bool ok;
                        if (bt_staged) {
                            const int lp = sc.shift >= 0 ? p >> sc.shift : p / sc.P;
                            const int pg = sh.bts[lp - bt_lo];
                            ok = pg >= 0 && pg < sc.num_pages;
                        } else {
                            ok = slot_valid(sc, seq, p);
                        }
                        nslot += ok;
                        nbad += !ok;
                    }
                }
        }
        if (rank == 0) {
            const int nsel = (int)min(total, (uint32_t)k);
            for (int j = nsel + tid; j < k; j += kThreads)
                orow[j] = -1;
        }
        if (sc.bt) {
            nslot = __reduce_add_sync(0xffffffffu, nslot);
            nbad = __reduce_add_sync(0xffffffffu, nbad);
            if (lane == 0 && nslot)
                atomicAdd(sc.lens + row, (int32_t)nslot);
            if (lane == 0 && nbad)
                atomicOr(sc.status, kDevBadPage);
        }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

} // namespace topk_cluster
} // namespace idx
