// idx_logits_kernel.cuh -- the warp-specialised tcgen05 logits kernel.
//
// One persistent CTA per SM, warp-specialised:
//   producers (warps 0-1, even / odd tiles): TMA loads of each tile
//             (values and key scales, 64-key boxes page by page through the
//             block table) into a ring of shared-memory stages; warp 0 also
//             loads each row group's Q tile, weights and scales into one of
//             two group slots and builds the group's candidate bitmap.  The
//             32 lanes resolve the pages of 32 boxes at a time, one window
//             ahead, so a tile costs a barrier wait and a few TMA issues;
//   MMA issuers (warps 2-3): one elected lane issues the tcgen05 MMAs
//             S[t, (r,h)] = k[t,:] . q[r,h,:] with keys on M (128 TMEM lanes)
//             and the group's (row, head) pairs on N, into one of NA TMEM
//             accumulators, after the warp has copied the tile's key scales
//             out of the stage, which the MMA's commit then frees; warp 2 owns
//             the TMEM allocation;
//   epilogue  NA warpgroups, one per accumulator: thread i of a warpgroup
//             owns TMEM lane i, i.e. one key, and reduces
//             sum_h w[r,h] * relu(scale * S[t,(r,h)]) over the heads in
//             registers, applies the [ks, ke) and candidate masks and stores
//             the fp32 logit.  Per-head scores never leave TMEM and registers;
//             the key's scale comes from the accumulator's side copy.
// Stages, group slots and accumulators are handed over with mbarriers whose
// waits are all bounded (mbar_wait), so a broken pipeline ends the kernel
// with IDX_DEV_TIMEOUT instead of hanging.
#pragma once

#include "idx_common.cuh"
#include "idx_logits.cuh"

namespace idx {

constexpr int kFmtFp8 = 0;
constexpr int kFmtMxfp4 = 1;
// Warp roles: 0-1 producers (even / odd tiles), 2-3 MMA issuers, 4..
// epilogue (NA warpgroups).  Tile c goes to TMEM accumulator c % NA, which
// MMA warp (c % NA) & 1 fills and epilogue warpgroup c % NA drains, so every
// accumulator has one filler and one drainer.  Every SMSP (warp % 4) runs one
// control warp and NA epilogue warps, and the per-tile issue cost of each
// control role is split over two warps.
constexpr int kFirstEpiWarp = 4;

// Tile descriptor: {j, gq}, written by the MMA warp beside each tile it
// issues (and {kDescDone, -} after the last one where the epilogue cannot
// tell that it was the last), from which the accumulator's epilogue
// warpgroup takes the tile's place: only the control warps walk the CTA's
// unit range.  j: tile index within the group (keys [j TK, (j + 1) TK)); gq:
// the CTA's count of the group (Q slot gq & 1, its q_full phase (gq >> 1) & 1).
// Compute tiles go to the accumulators in turn (tile c to c % NA), so the
// epilogue's use u of accumulator a is the CTA's compute tile a + u NA.
constexpr int kDescDone = -1;

// Group block: 16 words beside each Q slot, written by producer 0 before the
// slot's q_full arrival: rows, ranges and the keys live in every row.
enum GroupBlock : int {
    kGrpNrows = 0,
    kGrpRow0 = 1,
    kGrpLo = 2,    // union of the rows' ranges [lo, hi)
    kGrpHi = 3,
    kGrpInLo = 4,  // keys live in every row: [in_lo, in_hi)
    kGrpInHi = 5,
    kGrpCEnd = 6,  // end of the group's compute tiles in the CTA's count
    kGrpLast = 7,  // 1: the CTA's range ends in this group
    kGrpRks = 8,   // rows' starts (four words), then ends (four words)
    kGrpRke = 12,
    kGrpWords = 16,
};
constexpr int kMmaWarp = 2;

template <int FMT, int H, int G, int S, int NA, int TK>
struct LogitsCfg {
    static_assert(TK == 128 || TK == 256, "a tile is one or two MMAs of 128 keys");
    static constexpr int NSUB = TK / kMmaM;               // MMAs (of 128 keys) per tile
    static constexpr int NH = TK / kHalfKeys;             // 64-key TMA boxes per tile
    static constexpr int WIN_TILES = 32 / NH;             // tiles of one producer page window
    static constexpr int NCOLS = G * H;                    // MMA N
    static constexpr int ACC_COLS = NSUB * NCOLS;          // TMEM columns of one tile
    static constexpr int ROWB = FMT == kFmtFp8 ? 128 : 64;  // value bytes per key / query row
    static constexpr int A_BYTES = TK * ROWB;
    static constexpr int SUB_BYTES = kMmaM * ROWB;         // one MMA's A operand
    // stage: K values | key scales as loaded (FP8 fp32, MXFP4 e8m0 words) |
    // (MXFP4) the scale words in MMA order | flags: which halves hold data
    static constexpr int SF_STAGE = TK * 4;
    static constexpr int SF_ATOM = FMT == kFmtFp8 ? 0 : NSUB * 512;
    static constexpr int OFF_FLAGS = A_BYTES + SF_STAGE + SF_ATOM;
    static constexpr int STAGE_BYTES = ((OFF_FLAGS + 16) + 1023) / 1024 * 1024;
    static constexpr int Q_BYTES = (NCOLS * ROWB + 1023) / 1024 * 1024;
    static constexpr int W_BYTES = G * H * 4;
    static constexpr int QS_BYTES = G * H * 4;  // FP8 q_scale or MXFP4 q scale words
    static constexpr int QATOMS = (NCOLS + 127) / 128;
    static constexpr int QATOM_BYTES = FMT == kFmtFp8 ? 0 : QATOMS * 512;  // per MMA warp
    // shared memory offsets
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_Q = OFF_STAGE + S * STAGE_BYTES;
    static constexpr int OFF_W = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_QS = OFF_W + 2 * W_BYTES;
    static constexpr int GRP_BYTES = 4 * kGrpWords;  // group block per Q slot
    static constexpr int OFF_GRP = OFF_QS + 2 * QS_BYTES;
    static constexpr int OFF_QATOM = OFF_GRP + 2 * GRP_BYTES;
    // per accumulator: the tile's key scales (FP8) and flags, copied out of
    // the stage by the MMA warp so that the stage is free once the MMA is done,
    // and the tile's descriptor (TileDesc words) for the epilogue
    static constexpr int SIDE_FLAGS = FMT == kFmtFp8 ? TK * 4 : 0;
    static constexpr int SIDE_DESC = SIDE_FLAGS + 16;
    static constexpr int SIDE_BYTES = SIDE_DESC + 16;  // descriptor: two words, padded
    static constexpr int OFF_SIDE = OFF_QATOM + 4 * QATOM_BYTES;
    static constexpr int OFF_BAR = (OFF_SIDE + NA * SIDE_BYTES + 7) / 8 * 8;
    // full[S], empty[S], acc_full[NA], acc_empty[NA], q_full[2], q_empty[2]
    // + hist[NA][2]: a warpgroup's histogram hand-over (histogram variant)
    // + drain[2]: each MMA warp's last commit after an abort
    // + acc_full2[NA], acc_empty2[NA]: the second column half of each
    //   accumulator (split accumulators)
    static constexpr int NUM_BARS = 2 * S + 2 * NA + 4 + 2 * NA + 2 + 2 * NA;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // tmem base, abort flag
    static constexpr int OFF_SCRATCH = (OFF_MISC + 16 + 7) / 8 * 8;  // 40 long longs
    static constexpr int OFF_BITMAP = OFF_SCRATCH + 40 * 8;
    static constexpr int fixed_bytes() { return OFF_BITMAP + 1024; }  // + alignment slack
    // TMEM columns: accumulators, then (MXFP4) scale factors of A per
    // accumulator and of B per group slot.
    static constexpr int TM_SFA = NA * ACC_COLS;
    static constexpr int TM_SFB = TM_SFA + (FMT == kFmtFp8 ? 0 : NA * NSUB * 4);
    static constexpr int TM_USED = TM_SFB + (FMT == kFmtFp8 ? 0 : 4 * QATOMS * 4);  // 2 slots x 2 MMA warps
    static constexpr int TM_COLS = TM_USED <= 32 ? 32 : TM_USED <= 64 ? 64 : TM_USED <= 128 ? 128
                                 : TM_USED <= 256 ? 256 : 512;
    static_assert(TM_USED <= 512, "accumulators do not fit in tensor memory");
    static_assert(NCOLS % 16 == 0 && NCOLS >= 16 && NCOLS <= 256, "MMA N out of range");
    static_assert(H % 32 == 0, "heads are read from TMEM 32 columns at a time");
    static_assert(NA == 2 || NA == 3, "two or three epilogue warpgroups");
    static_assert(G <= 4, "the group block holds four rows' ranges");
    static constexpr int EPI_WARPS = 4 * NA;
    static constexpr int THREADS = 32 * (kFirstEpiWarp + EPI_WARPS);
    // Tile c uses stage c % S.  S a multiple of 2 and of NA keeps every stage
    // with one producer and one MMA warp (and every accumulator with one MMA
    // warp and one epilogue warpgroup), each of which waits on every phase of
    // it in turn: a role that could skip a phase might wait one phase early,
    // and an mbarrier parity wait cannot tell phase n from phase n + 2.
    static_assert(S >= 2 && S % 2 == 0 && S % NA == 0, "stages must divide among the roles");
    __host__ __device__ static constexpr int stage(int c) { return c % S; }
    __host__ __device__ static constexpr uint32_t phase(int c) { return (uint32_t)(c / S) & 1u; }
    // instruction descriptor: fp32 accumulate, K-major A and B, M = 128, N = NCOLS
    __host__ __device__ static constexpr uint32_t idesc_f8()
    {
        return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(NCOLS >> 3) << 17) |
               ((uint32_t)(kMmaM >> 4) << 24);
    }
    // the same with N = NCOLS / 2 (one column half of a split accumulator)
    __host__ __device__ static constexpr uint32_t idesc_f8_half()
    {
        return (1u << 4) | ((uint32_t)(NCOLS >> 4) << 17) | ((uint32_t)(kMmaM >> 4) << 24);
    }
    // block-scaled e2m1 x e2m1 with ue8m0 scales; the scale-factor ids select
    // the byte of each 32-bit scale word the MMA starts from.
    __host__ __device__ static constexpr uint32_t idesc_mxf4(int sf_id)
    {
        return ((uint32_t)sf_id << 4) | (1u << 7) | (1u << 10) |
               ((uint32_t)(NCOLS >> 3) << 17) | (1u << 23) |
               ((uint32_t)(kMmaM >> 4) << 24) | ((uint32_t)sf_id << 29);
    }
};

// Whether the walk's current unit is scored (K loaded, MMA issued) rather
// than only written -inf: it overlaps the group's live keys and, under a
// gather plan, holds a candidate key.
template <bool PLAN>
__device__ __forceinline__ bool unit_compute(const UnitWalk &w, int shift)
{
    return PLAN || tile_is_compute(w.gi, w.j, shift);  // a plan lists compute tiles only
}

// Logical page of key position t (shift when the page size is a power of two).
__device__ __forceinline__ int page_of(const LogitsArgs &a, int t)
{
    return a.page_shift >= 0 ? (t >> a.page_shift) : t / a.page_size;
}

// One lane's 64-key box of a producer window of 32 / NH units starting at
// unit k0 of the walk's group (lane l: box l % NH of unit k0 + l / NH): does
// the group need it, which page and row it starts at.  The block-table load
// is issued here and only consumed when the window becomes current.
struct HalfInfo {
    int page, row;
    bool need;
};

template <int NH, bool PLAN>
__device__ __forceinline__ HalfInfo half_info(const LogitsArgs &a, const UnitWalk &w, int k0,
                                              int lane)
{
    HalfInfo h;
    const GroupInfo &gi = w.gi;
    const int g = w.g;
    int tok;
    if constexpr (PLAN) {
        const int kk = k0 + lane / NH;
        tok = kk < w.n ? (unit_tile<PLAN>(a, g, kk) * NH + lane % NH) * kHalfKeys : gi.hi;
    } else {
        tok = (k0 * NH + lane) * kHalfKeys;  // units are consecutive tiles
    }
    h.need = tok < gi.hi && tok + kHalfKeys > gi.lo && (!PLAN || plan_box(a, g, tok / kHalfKeys));
    h.page = 0;
    h.row = tok;
    if (a.paged) {
        const int lp = page_of(a, tok);
        h.row = tok - lp * a.page_size;
        h.page = h.need && lp < a.max_blocks ? __ldg(a.bt + (size_t)g * a.bt_stride + lp) : -1;
    }
    return h;
}

} // namespace idx

namespace idx {

// Shared-memory bytes of the digit-1 histograms of the histogram variant:
// one 2048-bin histogram per row of the group for each epilogue warpgroup,
// placed after the candidate bitmaps.
template <int G, int NA>
constexpr int hist_smem_bytes()
{
    return NA * G * 2048 * 4;
}

template <int FMT, int H, int G, int S, int NA, int TK, bool PLAN, bool BMAX = false,
          bool HIST = false>
__global__ void __launch_bounds__(LogitsCfg<FMT, H, G, S, NA, TK>::THREADS, 1)
    logits_kernel(const __grid_constant__ LogitsArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmS)
{
    using C = LogitsCfg<FMT, H, G, S, NA, TK>;
    constexpr int TSH = TK == 256 ? 8 : 7;  // equals a.tile_shift
    // Tile descriptors (only the control warps walk the units; the epilogue
    // takes each tile from its descriptor) where they measured faster: block
    // maxima, four-row groups, MXFP4.  On the FP8 decodes every warp walks
    // the units, which keeps the control warps' work per tile, there the
    // longer chain, at its least.
    constexpr bool DESC = BMAX || G == 4 || FMT == kFmtMxfp4;
    // Split accumulators (four-row FP8 groups, N = 256): each tile's MMA is
    // issued as two N = 128 halves (rows 0-1 and 2-3 of the group) with
    // their own full / empty barriers, so the next tile's first half runs
    // while the epilogue drains the second half of this one.
    constexpr bool SPLIT = DESC && FMT == kFmtFp8 && G == 4 && C::NSUB == 1;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // swizzled TMA tiles and MMA descriptors assume 1024-byte aligned tiles
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bars, *empty = bars + S;
    uint64_t *acc_full = bars + 2 * S, *acc_empty = acc_full + NA;
    uint64_t *q_full = acc_empty + NA, *q_empty = q_full + 2;
    uint64_t *hbar = q_empty + 2;  // [NA][2]: counts done, flush done
    uint64_t *drain = hbar + 2 * NA;  // [2]: MMA warps' commits after an abort
    uint64_t *acc_full2 = drain + 2, *acc_empty2 = acc_full2 + NA;  // split accumulators
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    long long *scratch = reinterpret_cast<long long *>(smem + C::OFF_SCRATCH);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem + C::OFF_BITMAP);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);  // the MMA's commit
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(&acc_full[i], 2);  // the MMA's commit + the MMA warp's side copy
            mbar_init(&acc_empty[i], 4);  // the owning warpgroup's warps
            mbar_init(&acc_full2[i], 1);  // the second half's commit
            mbar_init(&acc_empty2[i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 2 + C::EPI_WARPS);  // both MMA warps' commits + epilogue
        }
        for (int i = 0; i < 2 * NA; ++i) {
            mbar_init(&hbar[i], 4);  // the warpgroup's four warps
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmS);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, C::TM_COLS);
        tmem_relinquish();
    }
    // the schedule's first dependent loads (each row's context length and
    // start) go to L2 while the previous kernel on the stream finishes
    if (a.paged && warp == kMmaWarp + 1) {
        const int nctx = a.ctx_per_row ? a.total_rows : a.num_groups;
        for (int i = lane * 32; i < nctx; i += 32 * 32)
            prefetch_l2(a.ctx + i);
        if (a.row_ks)
            for (int i = lane * 32; i < a.total_rows; i += 32 * 32)
                prefetch_l2(a.row_ks + i);
    }
    // everything above touches only this CTA's own resources (and prefetches
    // into L2); inputs and the logits buffer may still be in use by the
    // previous kernel on the stream
    pdl_wait();
    pdl_launch_dependents();
    int g0, k0, n0;
    long long count;
    locate_units<PLAN>(a, scratch, g0, k0, n0, count);  // contains __syncthreads
    // histogram variant: one 2048-bin histogram per (warpgroup, row of the
    // group), after the candidate bitmaps, cleared before the barrier below
    uint32_t *hist_sm = nullptr;
    if constexpr (HIST) {
        hist_sm = reinterpret_cast<uint32_t *>(
            smem + ((C::OFF_BITMAP + 2 * G * a.cand_words * 4 + 15) & ~15));
        for (int b = threadIdx.x; b < NA * G * 2048; b += C::THREADS)
            hist_sm[b] = 0u;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    UnitWalk w;
    walk_begin<PLAN>(a, w, g0, k0, n0, count);

    if (warp < 2) {
        // ------------------------------------------------------------ producers
        // Producer pw issues the compute tiles with c % 2 == pw (stage parity
        // pw); producer 0 also loads each group's Q tile, weights and scales.
        const int pw = warp;
        int gq = 0;        // groups started by this CTA
        int c = 0;         // compute tiles of this CTA seen so far
        int win0 = 0;      // first tile of the current page window
        HalfInfo cur = {}, nxt = {};
        bool cur_ok = false;
        int nfill = 0;     // fill units seen (producer nfill & 1 writes each)
        int fke = 0;       // lane i < nrows: row i's end
        for (; w.left > 0; walk_next<PLAN>(a, w)) {
            int fks = 0;
            if (w.first_in_group) {
                // page window of this group: current and next, block-table
                // loads in flight before anything else
                win0 = w.k;
                cur = half_info<C::NH, PLAN>(a, w, win0, lane);
                nxt = half_info<C::NH, PLAN>(a, w, win0 + C::WIN_TILES, lane);
                cur_ok = false;
                // (descriptors) the rows' ranges, lane i holding row i's
                fke = 0;
                if (DESC && lane < w.gi.nrows)
                    row_range(a, w.gi.row0 + lane, fks, fke);
            }
            if (w.first_in_group && pw == 0) {
                const int slot = gq & 1;
                if (!mbar_wait(&q_empty[slot], ((gq >> 1) & 1) ^ 1, abort_flag, a.status))
                    break;
                const int nrows = w.gi.nrows;
                if (a.cand) {  // candidate bitmap of each row of the group
                    uint32_t *bm = bitmap + (size_t)slot * G * a.cand_words;
                    for (int i = lane; i < G * a.cand_words; i += 32)
                        bm[i] = 0u;
                    __syncwarp();
                    const int nbits = a.cand_words * 32;
                    for (int i = 0; i < nrows; ++i) {
                        const int32_t *cr = a.cand + (size_t)(w.gi.row0 + i) * a.cand_stride;
                        for (int e = lane; e < a.num_cand; e += 32) {
                            int id = cr[e];
                            if (id >= 0 && id < nbits)
                                atomicOr(&bm[i * a.cand_words + (id >> 5)], 1u << (id & 31));
                        }
                    }
                    __syncwarp();
                }
                if constexpr (DESC) {
                    // this CTA's compute tiles of the group: c .. cend - 1 (tile c to
                    // accumulator c % NA); an accumulator that gets none of them is
                    // done with the Q slot at once (its warpgroup's four arrivals)
                    const long long kend = min((long long)w.n, (long long)w.k + w.left);
                    long long ncomp;
                    if constexpr (PLAN) {
                        ncomp = kend - w.k;
                    } else {
                        const long long jlo = w.gi.hi > w.gi.lo ? (w.gi.lo >> TSH) : kend;
                        const long long jhi = w.gi.hi > w.gi.lo ? ((w.gi.hi - 1) >> TSH) + 1 : kend;
                        ncomp = max(0LL, min(kend, jhi) - max((long long)w.k, jlo));
                    }
                    const int cend = c + (int)ncomp;
                    const int glast = walk_group_is_last(a, w);
                    if (lane == 0)
                        for (int acc = 0; acc < NA; ++acc)
                            if (((acc - c % NA) + NA) % NA >= ncomp)
                                mbar_arrive_cnt(&q_empty[slot], 4);
                    {
                        // the group block, published by the q_full arrival below
                        const int in_lo = __reduce_max_sync(0xffffffffu, lane < nrows ? fks : 0);
                        const int in_hi =
                            __reduce_min_sync(0xffffffffu, lane < nrows ? fke : 0x7fffffff);
                        const int rk = __shfl_sync(0xffffffffu, fks, (lane - kGrpRks) & 31);
                        const int re = __shfl_sync(0xffffffffu, fke, (lane - kGrpRke) & 31);
                        if (lane < kGrpWords)
                            reinterpret_cast<int *>(smem + C::OFF_GRP + slot * C::GRP_BYTES)[lane] =
                                lane == kGrpNrows   ? nrows
                                : lane == kGrpRow0  ? w.gi.row0
                                : lane == kGrpLo    ? w.gi.lo
                                : lane == kGrpHi    ? w.gi.hi
                                : lane == kGrpInLo  ? in_lo
                                : lane == kGrpInHi  ? in_hi
                                : lane == kGrpCEnd  ? cend
                                : lane == kGrpLast  ? glast
                                : lane >= kGrpRks && lane < kGrpRks + G ? rk
                                : lane >= kGrpRke && lane < kGrpRke + G ? re
                                                                         : 0;
                        __syncwarp();
                    }
                }
                if (lane == 0) {
                    uint32_t bytes = (uint32_t)(C::NCOLS * C::ROWB) + nrows * H * 4;
                    const bool qs = FMT == kFmtFp8 ? a.q_scale != nullptr : true;
                    if (qs)
                        bytes += nrows * H * 4;
                    mbar_arrive_expect_tx(&q_full[slot], bytes);
                    tma_load_2d(smem + C::OFF_Q + slot * C::Q_BYTES, &tmQ, &q_full[slot], 0,
                                w.gi.row0 * H);
                    bulk_load(smem + C::OFF_W + slot * C::W_BYTES,
                              a.weights + (size_t)w.gi.row0 * H, nrows * H * 4, &q_full[slot]);
                    if (qs) {
                        const void *src = FMT == kFmtFp8
                                              ? (const void *)(a.q_scale + (size_t)w.gi.row0 * H)
                                              : (const void *)(a.q_sf + (size_t)w.gi.row0 * H * 4);
                        bulk_load(smem + C::OFF_QS + slot * C::QS_BYTES, src, nrows * H * 4,
                                  &q_full[slot]);
                    }
                }
                __syncwarp();
                ++gq;
            }
            if (!unit_compute<PLAN>(w, TSH)) {
                // (descriptors) a fill unit: -inf over the tile for each row,
                // up to its end; without descriptors the epilogue writes it
                if (DESC && (nfill++ & 1) == pw) {
                    const int t0 = w.j << TSH;
                    const int wend = a.paged ? w.gi.hi : a.N;
                    #pragma unroll 1
                    for (int i = 0; i < w.gi.nrows; ++i) {
                        const int ke = __shfl_sync(0xffffffffu, fke, i);
                        const int end = min(wend, a.paged ? ke : a.N);
                        float *orow = a.logits + (size_t)(w.gi.row0 + i) * a.ld;
                        #pragma unroll
                        for (int m = 0; m < TK / 32; ++m) {
                            const int t = t0 + m * 32 + lane;
                            if (t < end)
                                orow[t] = -INFINITY;
                        }
                    }
                }
                continue;
            }
            if ((c & 1) != pw) {  // the other producer's tile
                ++c;
                continue;
            }
            if (w.k >= win0 + C::WIN_TILES) {  // slide the window (warp-uniform)
                const int step = (w.k - win0) / C::WIN_TILES;
                if (step == 1) {
                    cur = nxt;
                } else {
                    cur = half_info<C::NH, PLAN>(a, w, win0 + step * C::WIN_TILES, lane);
                }
                win0 += step * C::WIN_TILES;
                nxt = half_info<C::NH, PLAN>(a, w, win0 + C::WIN_TILES, lane);
                cur_ok = false;
            }
            if (!cur_ok) {  // first use of this window: resolve validity
                if (a.paged && cur.need && (cur.page < 0 || cur.page >= a.num_pages)) {
                    atomicOr(a.status, kDevBadPage);
                    cur.need = false;
                }
                cur_ok = true;
            }
            const int s = C::stage(c);
            if (!mbar_wait(&empty[s], C::phase(c) ^ 1, abort_flag, a.status))
                break;
            const int h0 = C::NH * (w.k - win0);  // lanes h0 .. h0 + NH - 1 own this tile's boxes
            const uint32_t ball = __ballot_sync(0xffffffffu, cur.need);
            const uint32_t mine = (ball >> h0) & ((1u << C::NH) - 1u);
            uint8_t *st = smem + C::OFF_STAGE + s * C::STAGE_BYTES;
            if (lane == 0) {
                *reinterpret_cast<uint32_t *>(st + C::OFF_FLAGS) = mine;
                mbar_arrive_expect_tx(&full[s], (uint32_t)__popc(mine) *
                                                    (kHalfKeys * C::ROWB + kHalfKeys * 4));
            }
            __syncwarp();
            if (lane >= h0 && lane < h0 + C::NH && cur.need) {
                const int k = lane - h0;
                tma_load_3d(st + k * kHalfKeys * C::ROWB, &tmK, &full[s], 0, cur.row, cur.page);
                // the half's 64 key scales (FP8 fp32 / MXFP4 4 x e8m0), 256 bytes
                if (a.paged)
                    tma_load_2d(st + C::A_BYTES + k * 256, &tmS, &full[s], cur.row * 4, cur.page);
                else
                    tma_load_1d(st + C::A_BYTES + k * 256, &tmS, &full[s], cur.row * 4);
            }
            __syncwarp();
            ++c;
        }
        // Tail: wait until the MMA has released every stage and the epilogue
        // every group slot this CTA filled, so no copy or commit is still in
        // flight when the CTA exits.
        if (!*abort_flag) {
            for (int i = c > S ? c - S : 0; i < c; ++i)
                if ((i & 1) == pw &&
                    !mbar_wait(&empty[C::stage(i)], C::phase(i), abort_flag,
                               a.status))
                    break;
            for (int i = gq > 2 ? gq - 2 : 0; i < gq; ++i)
                if (!mbar_wait(&q_empty[i & 1], (i >> 1) & 1, abort_flag, a.status))
                    break;
        }
        if (*abort_flag) {
            // after an abort: the copies this warp issued (its last S tiles'
            // stages, the last two group slots) land before the CTA exits
            for (int i = c > S ? c - S : 0; i < c; ++i)
                if ((i & 1) == pw)
                    mbar_wait_drain(&full[C::stage(i)], C::phase(i));
            for (int i = gq > 2 ? gq - 2 : 0; i < gq; ++i)
                mbar_wait_drain(&q_full[i & 1], (i >> 1) & 1);
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // ------------------------------------------------------------ MMA issuers
        // MMA warp mw issues the tiles with (c % NA) & 1 == mw and writes
        // each one's descriptor for the accumulator's epilogue warpgroup.
        const int mw = warp - kMmaWarp;
        int gq = 0;
        int c = 0;
        int slot = 0;
        uint32_t in_group = 0;  // accumulators with a compute tile in the current group
        bool glast = false;     // the current group is the CTA's last
        for (; w.left > 0; walk_next<PLAN>(a, w)) {
            if (w.first_in_group) {
                slot = gq & 1;
                if (!mbar_wait(&q_full[slot], (gq >> 1) & 1, abort_flag, a.status))
                    break;
                if constexpr (FMT == kFmtMxfp4) {
                    // q scale words -> 32x16B atoms in MMA order, then into TMEM
                    const uint32_t *qsw =
                        reinterpret_cast<const uint32_t *>(smem + C::OFF_QS + slot * C::QS_BYTES);
                    uint8_t *atom = smem + C::OFF_QATOM + (mw * 2 + slot) * C::QATOM_BYTES;
                    const int nvalid = w.gi.nrows * H;
                    for (int at = 0; at < C::QATOMS; ++at) {
                        uint4 v;
                        int n0 = at * 128 + lane;
                        v.x = n0 < nvalid ? qsw[n0] : 0u;
                        v.y = n0 + 32 < nvalid ? qsw[n0 + 32] : 0u;
                        v.z = n0 + 64 < nvalid ? qsw[n0 + 64] : 0u;
                        v.w = n0 + 96 < nvalid ? qsw[n0 + 96] : 0u;
                        *reinterpret_cast<uint4 *>(atom + at * 512 + lane * 16) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tc_fence_after();
                        for (int at = 0; at < C::QATOMS; ++at) {
                            uint64_t d = make_smem_desc(smem_u32(atom + at * 512), 128, 128,
                                                        kLayoutNone);
                            tmem_cp_32x128b_warpx4(
                                tmem_base + C::TM_SFB + ((mw * 2 + slot) * C::QATOMS + at) * 4, d);
                        }
                    }
                    __syncwarp();
                }
                if constexpr (DESC) {
                    // which accumulators get a compute tile of the group (the
                    // epilogue ends on the last group's last tile of each)
                    const long long kend = min((long long)w.n, (long long)w.k + w.left);
                    long long ncomp;
                    if constexpr (PLAN) {
                        ncomp = kend - w.k;
                    } else {
                        const long long jlo = w.gi.hi > w.gi.lo ? (w.gi.lo >> TSH) : kend;
                        const long long jhi =
                            w.gi.hi > w.gi.lo ? ((w.gi.hi - 1) >> TSH) + 1 : kend;
                        ncomp = max(0LL, min(kend, jhi) - max((long long)w.k, jlo));
                    }
                    glast = walk_group_is_last(a, w);
                    in_group = 0;
                    for (int acc = 0; acc < NA; ++acc)
                        if (((acc - c % NA) + NA) % NA < ncomp)
                            in_group |= 1u << acc;
                }
                __syncwarp();
                ++gq;
            }
            const bool compute = unit_compute<PLAN>(w, TSH);
            if (!compute) {
                // a fill unit (the producers write it)
            } else if (((c % NA) & 1) != mw) {
                ++c;  // the other MMA warp's tile
            } else {
                const int acc = c % NA;
                const int s = C::stage(c);
                uint8_t *st = smem + C::OFF_STAGE + s * C::STAGE_BYTES;
                uint8_t *sd = smem + C::OFF_SIDE + acc * C::SIDE_BYTES;
                if (!mbar_wait(&full[s], C::phase(c), abort_flag, a.status))
                    break;
                if constexpr (FMT == kFmtMxfp4) {
                    // K scale words (key-major as loaded) -> one MMA-order atom
                    // per 128 keys, in the stage: built while the accumulator
                    // may still be draining
                    const uint32_t *sw = reinterpret_cast<const uint32_t *>(st + C::A_BYTES);
                    #pragma unroll
                    for (int sub = 0; sub < C::NSUB; ++sub) {
                        uint4 v;
                        v.x = sw[sub * kMmaM + lane];
                        v.y = sw[sub * kMmaM + lane + 32];
                        v.z = sw[sub * kMmaM + lane + 64];
                        v.w = sw[sub * kMmaM + lane + 96];
                        *reinterpret_cast<uint4 *>(st + C::A_BYTES + C::SF_STAGE + sub * 512 +
                                                   lane * 16) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (!mbar_wait(&acc_empty[acc], (uint32_t)((c / NA) & 1) ^ 1, abort_flag, a.status))
                    break;
                {
                    // the epilogue's key scales and flags, out of the stage
                    if constexpr (FMT == kFmtFp8) {
                        const float4 *src = reinterpret_cast<const float4 *>(st + C::A_BYTES);
                        #pragma unroll
                        for (int i = lane; i < TK / 4; i += 32)
                            reinterpret_cast<float4 *>(sd)[i] = src[i];
                    }
                    if (lane == 0)
                        *reinterpret_cast<uint32_t *>(sd + C::SIDE_FLAGS) =
                            *reinterpret_cast<const uint32_t *>(st + C::OFF_FLAGS);
                    __syncwarp();
                }
                if (SPLIT && lane == 0) {
                    // the first column half: rows 0-1 of the group
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(smem + C::OFF_Q + slot * C::Q_BYTES);
                    const uint32_t a_addr = smem_u32(st);
                    #pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        uint64_t ad = make_smem_desc(a_addr + kk * 32, 16, 1024, kLayoutSw128);
                        uint64_t bd = make_smem_desc(b_addr + kk * 32, 16, 1024, kLayoutSw128);
                        mma_f8f6f4(tmem_base + acc * C::ACC_COLS, ad, bd, C::idesc_f8_half(),
                                   kk > 0 ? 1u : 0u);
                    }
                    *reinterpret_cast<int2 *>(sd + C::SIDE_DESC) = make_int2(w.j, gq - 1);
                    mma_commit(&acc_full[acc]);
                    mbar_arrive(&acc_full[acc]);  // releases the side copy and descriptor
                } else if (!SPLIT && lane == 0) {
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(smem + C::OFF_Q + slot * C::Q_BYTES);
                    #pragma unroll
                    for (int sub = 0; sub < C::NSUB; ++sub) {
                        // keys 128 sub .. 128 sub + 127 of the tile -> columns
                        // [sub NCOLS, (sub + 1) NCOLS) of the accumulator
                        const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS + sub * C::NCOLS;
                        const uint32_t a_addr = smem_u32(st + sub * C::SUB_BYTES);
                        if constexpr (FMT == kFmtFp8) {
                            #pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                uint64_t ad = make_smem_desc(a_addr + kk * 32, 16, 1024, kLayoutSw128);
                                uint64_t bd = make_smem_desc(b_addr + kk * 32, 16, 1024, kLayoutSw128);
                                mma_f8f6f4(d_tmem, ad, bd, C::idesc_f8(), kk > 0 ? 1u : 0u);
                            }
                        } else {
                            const uint32_t sfa = tmem_base + C::TM_SFA + (acc * C::NSUB + sub) * 4;
                            const uint32_t sfb =
                                tmem_base + C::TM_SFB + (mw * 2 + slot) * C::QATOMS * 4;
                            uint64_t cd = make_smem_desc(
                                smem_u32(st + C::A_BYTES + C::SF_STAGE + sub * 512), 128, 128,
                                kLayoutNone);
                            tmem_cp_32x128b_warpx4(sfa, cd);
                            #pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                uint64_t ad = make_smem_desc(a_addr + kk * 32, 16, 512, kLayoutSw64);
                                uint64_t bd = make_smem_desc(b_addr + kk * 32, 16, 512, kLayoutSw64);
                                mma_mxf4(d_tmem, ad, bd, C::idesc_mxf4(2 * kk), sfa, sfb,
                                         kk > 0 ? 1u : 0u);
                            }
                        }
                    }
                    if (DESC)
                        *reinterpret_cast<int2 *>(sd + C::SIDE_DESC) = make_int2(w.j, gq - 1);
                    mma_commit(&empty[s]);
                    mma_commit(&acc_full[acc]);
                    mbar_arrive(&acc_full[acc]);  // releases the side copy and descriptor
                }
                __syncwarp();
                if constexpr (SPLIT) {
                    // the second column half (rows 2-3), once the epilogue
                    // has drained it of the accumulator's previous tile
                    if (!mbar_wait(&acc_empty2[acc], (uint32_t)((c / NA) & 1) ^ 1, abort_flag,
                                   a.status))
                        break;
                    if (lane == 0) {
                        tc_fence_after();
                        const uint32_t b_addr = smem_u32(smem + C::OFF_Q + slot * C::Q_BYTES) +
                                                (uint32_t)(C::NCOLS / 2 * C::ROWB);
                        const uint32_t a_addr = smem_u32(st);
                        #pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            uint64_t ad = make_smem_desc(a_addr + kk * 32, 16, 1024, kLayoutSw128);
                            uint64_t bd = make_smem_desc(b_addr + kk * 32, 16, 1024, kLayoutSw128);
                            mma_f8f6f4(tmem_base + acc * C::ACC_COLS + C::NCOLS / 2, ad, bd,
                                       C::idesc_f8_half(), kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&empty[s]);
                        mma_commit(&acc_full2[acc]);
                    }
                    __syncwarp();
                }
                ++c;
            }
            if (walk_last_in_group(w)) {
                if (lane == 0)
                    mma_commit(&q_empty[slot]);
                __syncwarp();
            }
        }
        if (DESC && !*abort_flag) {
            // each of this warp's accumulators whose last tile the epilogue
            // could not tell was the last (none in the CTA's last group): a
            // descriptor without a tile, once the epilogue has drained it
            for (int acc = mw; acc < NA; acc += 2) {
                if (glast && ((in_group >> acc) & 1u))
                    continue;
                const int uses = c > acc ? (c - acc + NA - 1) / NA : 0;
                if (!mbar_wait(&acc_empty[acc], (uint32_t)(uses & 1) ^ 1, abort_flag, a.status))
                    break;
                if (lane == 0) {
                    uint8_t *sd = smem + C::OFF_SIDE + acc * C::SIDE_BYTES;
                    reinterpret_cast<int *>(sd + C::SIDE_DESC)[0] = kDescDone;
                    mbar_arrive_cnt(&acc_full[acc], 2);
                }
                __syncwarp();
            }
        }
        if (*abort_flag) {
            // after an abort: this warp's MMAs and tensor-memory copies in
            // flight complete before the tensor memory is freed
            if (lane == 0) {
                mma_commit(&drain[mw]);
                mbar_wait_drain(&drain[mw], 0);
            }
            __syncwarp();
        }
    } else if (warp >= kFirstEpiWarp) {
        // ------------------------------------------------------------ epilogue
        // NA warpgroups; warpgroup wg drains accumulator wg.  With
        // descriptors, every tile the MMA warp issues into it comes with one
        // (the tile and its row group) and the group's rows, ranges and
        // compute-tile end come from the group block beside its Q slot.
        // Without, the warpgroup walks the units: it drains the compute
        // tiles with c % NA == wg and writes the fill units with u % NA == wg.
        const int ew = warp - kFirstEpiWarp;
        const int wg = ew >> 2;
        const int acc = wg;
        const int quad = warp & 3;            // TMEM lane quadrant of this warp
        const int kq = quad * 32 + lane;      // key of each 128-key MMA block this thread owns
        int gq = DESC ? -1 : 0;               // group of the last descriptor / groups started
        int c = 0;                            // (walk) compute tiles seen, all warpgroups'
        long long u = 0;                      // (walk) units seen
        int slot = 0, nrows = 0, row0 = 0, glo = 0, ghi = 0;
        int in_lo = 0, in_hi = 0;             // keys live in every row of the group
        int cend = 0, glast = 0;              // the group's compute-tile end, last-group flag
        int rks[G], rke[G];
        // one-row groups on 256-key tiles: the row's 64 head weights held in
        // registers for the whole group
        constexpr bool kWregs = G == 1 && C::NSUB == 2;
        float4 wreg[kWregs ? 16 : 1];
        constexpr int NSUB = C::NSUB;
        // histogram variant: this warpgroup's G x 2048 bins; the warp's
        // valid keys of each row in the 8192-key chunk it is in (flushed
        // when the chunk or the group changes) and in the group
        uint32_t *hs = HIST ? hist_sm + (size_t)wg * G * 2048 : nullptr;
        uint32_t hphase = 0;  // phase of this warpgroup's hand-over barriers
        uint32_t vchunk_n[G], vrow_n[G];
        int vchunk = -1;
        #pragma unroll
        for (int i = 0; i < G; ++i)
            vchunk_n[i] = vrow_n[i] = 0u;
        for (uint32_t use = 0;; ++use) {
            bool compute = true, mine = true, last;
            int j;
            uint32_t halves = 0;
            float ksc[NSUB];
            if constexpr (DESC) {
                if (!mbar_wait(&acc_full[acc], use & 1u, abort_flag, a.status))
                    break;
                tc_fence_after();
                const uint8_t *sd = smem + C::OFF_SIDE + acc * C::SIDE_BYTES;
                // the descriptor, box flags and key scales are read together,
                // before any branch on them
                const int2 d0 = *reinterpret_cast<const int2 *>(sd + C::SIDE_DESC);  // j, gq
                halves = *reinterpret_cast<const uint32_t *>(sd + C::SIDE_FLAGS);
                #pragma unroll
                for (int sub = 0; sub < NSUB; ++sub)
                    ksc[sub] = FMT == kFmtFp8
                                   ? reinterpret_cast<const float *>(sd)[sub * kMmaM + kq]
                                   : 1.0f;
                if (d0.x == kDescDone)
                    break;
                if (d0.y != gq) {  // a new row group: its weights, rows and ranges
                    gq = d0.y;
                    slot = gq & 1;
                    if (!mbar_wait(&q_full[slot], (gq >> 1) & 1, abort_flag, a.status))
                        break;
                    const int *gb =
                        reinterpret_cast<const int *>(smem + C::OFF_GRP + slot * C::GRP_BYTES);
                    const int4 g0v = *reinterpret_cast<const int4 *>(gb);
                    const int4 g1v = *reinterpret_cast<const int4 *>(gb + 4);
                    const int4 rs = *reinterpret_cast<const int4 *>(gb + kGrpRks);
                    const int4 re = *reinterpret_cast<const int4 *>(gb + kGrpRke);
                    nrows = g0v.x;
                    row0 = g0v.y;
                    glo = g0v.z;
                    ghi = g0v.w;
                    in_lo = g1v.x;
                    in_hi = g1v.y;
                    cend = g1v.z;
                    glast = g1v.w;
                    const int rsa[4] = {rs.x, rs.y, rs.z, rs.w};
                    const int rea[4] = {re.x, re.y, re.z, re.w};
                    #pragma unroll
                    for (int i = 0; i < G; ++i) {
                        rks[i] = rsa[i];
                        rke[i] = rea[i];
                    }
                    if constexpr (kWregs) {
                        const float4 *w4 =
                            reinterpret_cast<const float4 *>(smem + C::OFF_W + slot * C::W_BYTES);
                        #pragma unroll
                        for (int q = 0; q < 16; ++q)
                            wreg[q] = w4[q];
                    }
                }
                j = d0.x;
                // the group's last tile on this accumulator; in the CTA's last
                // group, the accumulator's last tile
                last = acc + (int)use * NA + NA >= cend;
            } else {
                if (w.left <= 0)
                    break;
                if (w.first_in_group) {
                    slot = gq & 1;
                    nrows = w.gi.nrows;
                    row0 = w.gi.row0;
                    glo = w.gi.lo;
                    ghi = w.gi.hi;
                    in_lo = 0;
                    in_hi = 0x7fffffff;
                    for (int i = 0; i < G; ++i) {
                        rks[i] = 0;
                        rke[i] = 0;
                        if (i < nrows) {
                            row_range(a, row0 + i, rks[i], rke[i]);
                            in_lo = max(in_lo, rks[i]);
                            in_hi = min(in_hi, rke[i]);
                        }
                    }
                    if (!mbar_wait(&q_full[slot], (gq >> 1) & 1, abort_flag, a.status))
                        break;
                    if constexpr (kWregs) {
                        const float4 *w4 =
                            reinterpret_cast<const float4 *>(smem + C::OFF_W + slot * C::W_BYTES);
                        #pragma unroll
                        for (int q = 0; q < 16; ++q)
                            wreg[q] = w4[q];
                    }
                    ++gq;
                }
                j = w.j;
                compute = unit_compute<PLAN>(w, TSH);
                if (compute) {
                    mine = c % NA == wg;
                    ++c;
                } else {
                    mine = (int)(u % NA) == wg;
                }
                last = walk_last_in_group(w);
            }
            // a tile whose every key is live in every row of the group (and
            // no candidate mask): no range tests, unconditional stores
            const bool interior = !a.cand && (j << TSH) >= in_lo && (j << TSH) + TK <= in_hi;
            const int t0 = (j << TSH) + kq;  // this thread's key in sub-tile 0
            const int wend = a.paged ? ghi : a.N;  // columns this group writes
            float val[NSUB][G];
            #pragma unroll
            for (int sub = 0; sub < NSUB; ++sub)
                #pragma unroll
                for (int i = 0; i < G; ++i)
                    val[sub][i] = -INFINITY;
            if (compute && mine) {
                if constexpr (!DESC) {
                    const int use_w = (c - 1) / NA;  // uses of this accumulator so far
                    if (!mbar_wait(&acc_full[acc], (uint32_t)(use_w & 1), abort_flag, a.status))
                        break;
                    tc_fence_after();
                    // key scales and box flags from the accumulator's side copy
                    const uint8_t *sd = smem + C::OFF_SIDE + acc * C::SIDE_BYTES;
                    halves = *reinterpret_cast<const uint32_t *>(sd + C::SIDE_FLAGS);
                    #pragma unroll
                    for (int sub = 0; sub < NSUB; ++sub)
                        ksc[sub] = FMT == kFmtFp8
                                       ? reinterpret_cast<const float *>(sd)[sub * kMmaM + kq]
                                       : 1.0f;
                }
                bool live[NSUB];
                bool pos = true;
                #pragma unroll
                for (int sub = 0; sub < NSUB; ++sub) {
                    const int key = sub * kMmaM + kq, t = t0 + sub * kMmaM;
                    live[sub] = (interior || (t < ghi && t >= glo)) &&
                                ((halves >> (key >> 6)) & 1u);
                    pos = pos && ksc[sub] >= 0.0f;
                }
                const float *wsm = reinterpret_cast<const float *>(smem + C::OFF_W + slot * C::W_BYTES);
                const float *qsm = reinterpret_cast<const float *>(smem + C::OFF_QS + slot * C::QS_BYTES);
                const bool use_qs = FMT == kFmtFp8 && a.q_scale != nullptr;
                // relu(ksc * x) = |ksc| * relu(sgn * x); the common all-positive
                // case skips the sign multiply.  Branches stay warp-uniform so
                // the warp is converged at every tcgen05.ld.
                const bool all_pos = __all_sync(0xffffffffu, pos);
                bool h0_back = false;  // (split) the first column half handed back
                const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * C::ACC_COLS;
                bool summed = false;
                if constexpr (NSUB == 2) {
                    if (!use_qs && all_pos) {
                        // Common path on 256-key tiles: for each row, both
                        // sub-tiles' blocks of a half of the heads are loaded
                        // together and summed side by side, so each weight is
                        // read once per tile (one-row groups hold them in
                        // registers) and the two sub-tiles' packed-FMA chains
                        // interleave.  Rows past the group's last are computed
                        // and discarded.
                        #pragma unroll
                        for (int i = 0; i < G; ++i) {
                            float2 cc[2][4];
                            #pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                uint32_t rb[2][32];
                                const uint32_t tcol = tbase + i * H + half * 32;
                                tmem_ld_32x32b_x32(tcol, rb[0]);
                                tmem_ld_32x32b_x32(tcol + C::NCOLS, rb[1]);
                                tmem_ld_wait();
                                if (half == 0) {
                                    #pragma unroll
                                    for (int jj = 0; jj < 4; ++jj)
                                        cc[0][jj] = cc[1][jj] = make_float2(0.0f, 0.0f);
                                }
                                const float4 *w4 =
                                    reinterpret_cast<const float4 *>(wsm + i * H + half * 32);
                                #pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const int h4 = half * 8 + q;
                                    const float4 wv = kWregs ? wreg[kWregs ? h4 : 0] : w4[q];
                                    const int jj = (h4 & 1) * 2;
                                    #pragma unroll
                                    for (int sb = 0; sb < 2; ++sb) {
                                        const float *x =
                                            reinterpret_cast<const float *>(&rb[sb][4 * q]);
                                        cc[sb][jj] = fma2(
                                            make_float2(wv.x, wv.y),
                                            make_float2(fmaxf(x[0], 0.0f), fmaxf(x[1], 0.0f)),
                                            cc[sb][jj]);
                                        cc[sb][jj + 1] = fma2(
                                            make_float2(wv.z, wv.w),
                                            make_float2(fmaxf(x[2], 0.0f), fmaxf(x[3], 0.0f)),
                                            cc[sb][jj + 1]);
                                    }
                                }
                            }
                            #pragma unroll
                            for (int sb = 0; sb < 2; ++sb) {
                                const float sum =
                                    ((cc[sb][0].x + cc[sb][2].x) + (cc[sb][0].y + cc[sb][2].y)) +
                                    ((cc[sb][1].x + cc[sb][3].x) + (cc[sb][1].y + cc[sb][3].y));
                                val[sb][i] = fabsf(ksc[sb]) * sum;
                            }
                        }
                        summed = true;
                    }
                }
                if (summed) {
                } else if (!use_qs && all_pos) {
                    // Common path.  The (sub-tile, row, half) blocks of 32 heads
                    // are loaded from TMEM into two register buffers in turn: the
                    // load of the next block is in flight while this one is
                    // summed (tcgen05.wait::ld then waits for it).  Each row sums
                    // its heads in eight partial sums, four packed-FMA chains.
                    // Rows past the group's last are computed and discarded.
                    constexpr int NU = NSUB * G * 2;
                    uint32_t rb[2][32];
                    float2 cc[4];
                    tmem_ld_32x32b_x32(tbase, rb[0]);
                    tmem_ld_wait();
                    #pragma unroll
                    for (int u = 0; u < NU; ++u) {
                        const int sub = u / (2 * G), i = (u / 2) % G, half = u & 1;
                        // (split) the second column half is loaded only once
                        // its MMA has landed, below
                        if (u + 1 < NU && !(SPLIT && u + 1 == NU / 2)) {
                            const int s1 = (u + 1) / (2 * G), i1 = ((u + 1) / 2) % G,
                                      h1 = (u + 1) & 1;
                            tmem_ld_32x32b_x32(tbase + s1 * C::NCOLS + i1 * H + h1 * 32,
                                               rb[(u + 1) & 1]);
                        }
                        if (half == 0) {
                            #pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                cc[jj] = make_float2(0.0f, 0.0f);
                        }
                        const float4 *w4 = reinterpret_cast<const float4 *>(wsm + i * H + half * 32);
                        #pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int h4 = half * 8 + q;
                            const float4 wv = w4[q];
                            const float *x = reinterpret_cast<const float *>(&rb[u & 1][4 * q]);
                            const int jj = (h4 & 1) * 2;
                            cc[jj] = fma2(make_float2(wv.x, wv.y),
                                          make_float2(fmaxf(x[0], 0.0f), fmaxf(x[1], 0.0f)), cc[jj]);
                            cc[jj + 1] = fma2(make_float2(wv.z, wv.w),
                                              make_float2(fmaxf(x[2], 0.0f), fmaxf(x[3], 0.0f)),
                                              cc[jj + 1]);
                        }
                        if (half == 1) {
                            const float sum = ((cc[0].x + cc[2].x) + (cc[0].y + cc[2].y)) +
                                              ((cc[1].x + cc[3].x) + (cc[1].y + cc[3].y));
                            val[sub][i] = fabsf(ksc[sub]) * sum;
                        }
                        if (SPLIT && u + 1 == NU / 2) {
                            // rows 0-1 done: their half goes back to the MMA
                            // warp, then rows 2-3 once their half has landed
                            // (after an abort the wait returns at once and the
                            // tile's values are discarded)
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(&acc_empty[acc]);
                            h0_back = true;
                            (void)mbar_wait(&acc_full2[acc], use & 1u, abort_flag, a.status);
                            tc_fence_after();
                            tmem_ld_32x32b_x32(tbase + C::NCOLS / 2, rb[(u + 1) & 1]);
                            tmem_ld_wait();
                        } else if (u + 1 < NU) {
                            tmem_ld_wait();
                        }
                    }
                } else {
                    if constexpr (SPLIT) {  // both column halves first
                        (void)mbar_wait(&acc_full2[acc], use & 1u, abort_flag, a.status);
                        tc_fence_after();
                    }
                    #pragma unroll
                    for (int sub = 0; sub < NSUB; ++sub) {
                        const float sgn = ksc[sub] >= 0.0f ? 1.0f : -1.0f;
                        #pragma unroll
                        for (int i = 0; i < G; ++i) {
                            if (i >= nrows)
                                break;
                            const uint32_t trow = tbase + sub * C::NCOLS + i * H;
                            const float4 *w4 = reinterpret_cast<const float4 *>(wsm + i * H);
                            float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // independent partial sums
                            {
                                // rare (per-head q scales, or a negative key scale):
                                // a rolled loop over four heads at a time keeps the
                                // code small
                                const float *qrow = qsm + i * H;
                                #pragma unroll 1
                                for (int h = 0; h < H; h += 4) {
                                    uint32_t x4[4];
                                    tmem_ld_32x32b_x4(trow + h, x4);
                                    tmem_ld_wait();
                                    const float4 wv = w4[h >> 2];
                                    const float wj[4] = {wv.x, wv.y, wv.z, wv.w};
                                    #pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float x = __uint_as_float(x4[e]);
                                        const float y = use_qs ? ksc[sub] * qrow[h + e] * x : sgn * x;
                                        s4[e] = fmaf(wj[e], fmaxf(y, 0.0f), s4[e]);
                                    }
                                }
                            }
                            const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
                            val[sub][i] = use_qs ? sum : fabsf(ksc[sub]) * sum;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (SPLIT && !h0_back)
                        mbar_arrive(&acc_empty[acc]);
                    mbar_arrive(SPLIT ? &acc_empty2[acc] : &acc_empty[acc]);
                }
                // masks
                #pragma unroll
                for (int sub = 0; sub < NSUB; ++sub) {
                    const int t = t0 + sub * kMmaM;
                    if (interior) {
                        if (!live[sub])
                            #pragma unroll
                            for (int i = 0; i < G; ++i)
                                val[sub][i] = -INFINITY;
                        continue;
                    }
                    #pragma unroll
                    for (int i = 0; i < G; ++i) {
                        bool keep = live[sub] && t >= rks[i] && t < rke[i];
                        if (keep && a.cand) {
                            const uint32_t *bm = bitmap + ((size_t)slot * G + i) * a.cand_words;
                            const int blk = a.cand_shift >= 0 ? (t - rks[i]) >> a.cand_shift
                                                              : (t - rks[i]) / a.cand_block;
                            keep = blk < a.cand_words * 32 && ((bm[blk >> 5] >> (blk & 31)) & 1u);
                        }
                        if (!keep)
                            val[sub][i] = -INFINITY;
                    }
                }
            }
            if (mine) {
                #pragma unroll
                for (int i = 0; i < G; ++i) {
                    if (i >= nrows)
                        break;
                    const int end = min(wend, a.paged ? rke[i] : a.N);
                    float *orow = a.logits + (size_t)(row0 + i) * a.ld;
                    #pragma unroll
                    for (int sub = 0; sub < NSUB; ++sub) {
                        const int t = t0 + sub * kMmaM;
                        if (interior || t < end)
                            orow[t] = val[sub][i];
                    }
                }
                if (HIST && compute) {
                    // digit-1 counts of the written logits into the
                    // warpgroup's shared histogram, one atomic per distinct
                    // bin of the warp; valid keys counted per warp (its 32
                    // keys lie in one 8192-key chunk)
                    #pragma unroll
                    for (int sub = 0; sub < NSUB; ++sub) {
                        const int chunk = (t0 - lane + sub * kMmaM) >> 13;  // the warp's first key
                        if (chunk != vchunk) {
                            if (vchunk >= 0 && lane == 0)
                                #pragma unroll
                                for (int i = 0; i < G; ++i)
                                    if (vchunk_n[i])
                                        atomicAdd(a.cvalid + (size_t)(row0 + i) * a.hist_P +
                                                      vchunk, vchunk_n[i]);
                            #pragma unroll
                            for (int i = 0; i < G; ++i)
                                vchunk_n[i] = 0u;
                            vchunk = chunk;
                        }
                        #pragma unroll
                        for (int i = 0; i < G; ++i) {
                            if (i >= nrows)
                                break;
                            const uint32_t key = order_key(val[sub][i]);
                            const uint32_t bin = key ? key >> 21 : 0xffffffffu;
                            const uint32_t peers = __match_any_sync(0xffffffffu, bin);
                            if (key && lane == __ffs(peers) - 1)
                                atomicAdd(&hs[i * 2048 + bin], (uint32_t)__popc(peers));
                            const uint32_t n = (uint32_t)__popc(__ballot_sync(0xffffffffu, key != 0u));
                            vchunk_n[i] += n;
                            vrow_n[i] += n;
                        }
                    }
                }
                if (BMAX && compute) {
                    // block maxima: a warp's 32 consecutive keys span at most
                    // two blocks (block >= 32 keys); each part's maximum goes
                    // to memory with one atomic
                    #pragma unroll
                    for (int i = 0; i < G; ++i) {
                        if (i >= nrows)
                            break;
                        float *brow = a.bmax + (size_t)(row0 + i) * a.ld_bmax;
                        #pragma unroll
                        for (int sub = 0; sub < NSUB; ++sub) {
                            const int t = t0 + sub * kMmaM;
                            const int d = t - rks[i];
                            const int b = d < 0 ? -1
                                          : a.bmax_shift >= 0 ? d >> a.bmax_shift
                                                              : d / a.bmax_block;
                            const int b0 = __shfl_sync(0xffffffffu, b, 0);
                            const bool first = b == b0;
                            // each part's maximum as an order-preserving key
                            // (-inf: 0), one warp reduction each
                            const uint32_t kv = order_key(val[sub][i]);
                            const uint32_t k0 = __reduce_max_sync(0xffffffffu, first ? kv : 0u);
                            const uint32_t k1 = __reduce_max_sync(0xffffffffu, first ? 0u : kv);
                            const uint32_t second = __ballot_sync(0xffffffffu, !first);
                            if (lane == 0 && b0 >= 0 && k0)
                                atomic_max_float(brow + b0, key_float(k0));
                            if (second && lane == __ffs(second) - 1 && b >= 0 && k1)
                                atomic_max_float(brow + b, key_float(k1));
                        }
                    }
                }
            }
            if (last) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&q_empty[slot]);
                if constexpr (HIST) {
                    // the warp's valid counts of the group go out; the
                    // group's bins of this warpgroup go to the rows'
                    // histograms once its four warps are done with the
                    // group; the bins are cleared before any warp counts the
                    // next group (bounded waits on two barriers)
                    if (lane == 0)
                        #pragma unroll
                        for (int i = 0; i < G; ++i) {
                            if (i < nrows && vchunk_n[i])
                                atomicAdd(a.cvalid + (size_t)(row0 + i) * a.hist_P + vchunk,
                                          vchunk_n[i]);
                            if (i < nrows && vrow_n[i])
                                atomicAdd(a.hvalid + row0 + i, vrow_n[i]);
                        }
                    #pragma unroll
                    for (int i = 0; i < G; ++i)
                        vchunk_n[i] = vrow_n[i] = 0u;
                    vchunk = -1;
                    if (lane == 0)
                        mbar_arrive(&hbar[2 * wg]);
                    if (!mbar_wait(&hbar[2 * wg], hphase, abort_flag, a.status))
                        break;
                    for (int b = quad * 32 + lane; b < G * 2048; b += 128) {
                        const uint32_t v = hs[b];
                        if (v) {
                            atomicAdd(a.hist + (size_t)(row0 + b / 2048) * 2048 + (b & 2047),
                                      v);
                            hs[b] = 0u;
                        }
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&hbar[2 * wg + 1]);
                    if (!mbar_wait(&hbar[2 * wg + 1], hphase, abort_flag, a.status))
                        break;
                    hphase ^= 1u;
                }
            }
            if constexpr (DESC) {
                if (last && glast)
                    break;
            } else {
                walk_next<PLAN>(a, w);
                ++u;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TM_COLS);
    }
}


// ----------------------------------------------------------------- gather plan
//
// Grid (row groups, kPlanSlices).  Each CTA finds, for its row group, the
// 64-key boxes that hold a candidate key of any of the group's rows
// (candidate blocks clipped to each row's [ks, ke)) and the tiles of 2^TSH
// keys that hold such a box (and overlap the group's live keys).  Slice 0
// writes the plan the logits kernel walks: the number of such tiles, the box
// bits and the tile list.  Every CTA writes -inf over the other tiles of its
// slice of the group, for each row up to the row's end: the logits the
// logits kernel will not write.  Dynamic shared memory: box_words +
// ceil(width / 128 / 32) words.
constexpr int kPlanSlices = 8;
constexpr int kPlanThreads = 256;

template <int TSH>
__global__ void __launch_bounds__(kPlanThreads) cand_plan_kernel(const __grid_constant__ LogitsArgs a)
{
    extern __shared__ uint32_t pbits[];
    uint32_t *box = pbits, *tb = pbits + a.box_words;
    __shared__ int rks[8], rke[8];
    pdl_wait();
    pdl_launch_dependents();
    const int g = blockIdx.x, slice = blockIdx.y, tid = threadIdx.x;
    const int tw = ((a.width + kMmaM - 1) / kMmaM + 31) / 32;
    // the group's candidate ids (row-major over its rows) are loaded before
    // the row ranges, so the two loads overlap; ids past the register batch
    // are read in the loop below
    const int row0 = g * a.G, nrows = min(a.G, a.total_rows - row0);
    const int nid = nrows * a.num_cand;
    constexpr int kIds = 4;
    int idv[kIds];
    #pragma unroll
    for (int q = 0; q < kIds; ++q) {
        const int e = tid + q * kPlanThreads;
        idv[q] = -1;
        if (e < nid)
            idv[q] = a.cand[(size_t)(row0 + e / a.num_cand) * a.cand_stride + e % a.num_cand];
    }
    const GroupInfo gi = group_info(a, g);
    for (int i = tid; i < a.box_words + tw; i += kPlanThreads)
        pbits[i] = 0u;
    if (tid < gi.nrows)
        row_range(a, gi.row0 + tid, rks[tid], rke[tid]);
    __syncthreads();
    for (int q = 0; q * kPlanThreads < nid; ++q) {
        const int e = tid + q * kPlanThreads;
        if (e >= nid)
            break;
        int id = -1;
        #pragma unroll
        for (int qq = 0; qq < kIds; ++qq)
            if (qq == q)
                id = idv[qq];
        if (q >= kIds)
            id = a.cand[(size_t)(row0 + e / a.num_cand) * a.cand_stride + e % a.num_cand];
        if (id < 0)
            continue;
        const int i = e / a.num_cand;
        const int ks = rks[i], ke = rke[i];
        const long long lo = (long long)ks + (long long)id * a.cand_block;
        if (lo >= ke)
            continue;
        const int t_lo = (int)lo;
        const int t_hi = (int)min((long long)ke, lo + a.cand_block);
        // the box bits, and the bits of the tiles holding those boxes (every
        // such tile overlaps the group's live keys: the box lies in a row's
        // [ks, ke))
        constexpr int BSH = TSH - 6;  // log2 of the 64-key boxes per tile
        for (int b = t_lo / kHalfKeys; b <= (t_hi - 1) / kHalfKeys; ++b) {
            atomicOr(&box[b >> 5], 1u << (b & 31));
            atomicOr(&tb[(b >> BSH) >> 5], 1u << ((b >> BSH) & 31));
        }
    }
    __syncthreads();
    if (slice == 0) {
        // the tile list in ascending order, by warp 0: each lane takes one
        // word of tile bits per round, and a shuffle scan of the words' bit
        // counts places its tiles
        uint32_t *dst = a.plan + (size_t)g * a.plan_words;
        uint32_t *list = dst + 1 + a.box_words;
        if (tid < 32) {
            uint32_t run = 0;
            for (int base = 0; base < tw; base += 32) {
                uint32_t bits = base + tid < tw ? tb[base + tid] : 0u;
                const uint32_t n = __popc(bits);
                uint32_t x = n;
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                    if (tid >= o)
                        x += y;
                }
                uint32_t pos = run + x - n;
                while (bits) {
                    const int bit = __ffs(bits) - 1;
                    list[pos++] = (uint32_t)((base + tid) * 32 + bit);
                    bits &= bits - 1u;
                }
                run += __shfl_sync(0xffffffffu, x, 31);
            }
            if (tid == 0)
                dst[0] = run;
        }
        for (int i = tid; i < a.box_words; i += kPlanThreads)
            dst[1 + i] = box[i];
    }
    if (!a.plan_fill)
        return;
    // -inf over the slice's tiles that are not scored, four keys per store
    // where the row allows it
    const int j0 = (int)((long long)gi.tiles * slice / kPlanSlices);
    const int j1 = (int)((long long)gi.tiles * (slice + 1) / kPlanSlices);
    constexpr int V = (1 << TSH) / 4;  // float4 per tile
    const bool vec = (a.ld & 3) == 0 && ((uintptr_t)a.logits & 15) == 0;
    for (int i = 0; i < gi.nrows; ++i) {
        float *orow = a.logits + (size_t)(gi.row0 + i) * a.ld;
        const int end = rke[i];
        for (int v = tid; v < (j1 - j0) * V; v += kPlanThreads) {
            const int j = j0 + v / V;
            if ((tb[j >> 5] >> (j & 31)) & 1u)
                continue;
            const int t = (j << TSH) + 4 * (v % V);
            if (t + 4 <= end && vec) {
                *reinterpret_cast<float4 *>(orow + t) =
                    make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            } else {
                for (int e = 0; e < 4 && t + e < end; ++e)
                    orow[t + e] = -INFINITY;
            }
        }
    }
}

} // namespace idx
