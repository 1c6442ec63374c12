// idx_logits.cuh -- argument block and work schedule of the logits kernel.
//
// Work is cut into units of (row group, key tile), a tile being 128 or 256
// keys (LogitsArgs::tile_shift; the kernel instantiation fixes it).  A row group is the
// set of query rows that share one key sequence and one MMA: the next_n rows
// of a sequence for paged decode / MTP, or G consecutive rows of a contiguous
// prefill chunk.  Each unit is either a "compute" tile (it overlaps the
// group's live key range: K is loaded and scored on the tensor cores) or a
// "fill" tile (it lies entirely below the group's first live key or, for the
// contiguous layout, past its last one, and is only written -inf).
//
// The grid is persistent: CTA i takes the contiguous unit range
// [i*U/G, (i+1)*U/G) of the global unit list (U units, G CTAs).  Ranges may
// cross group boundaries; logits columns of different units never overlap,
// so no reduction between CTAs is needed.  This is the flash-decode style
// context split of the vLLM page rocm_aiter_mla_sparse (_decode_num_splits,
// rocm_fp8_paged_mqa_logits_triton's N_SPLITS) done as an even split of
// key tiles over a machine-sized grid.
#pragma once

#include <cstdint>

namespace idx {

constexpr int kMmaM = 128;     // keys per MMA = TMEM lanes
constexpr int kHalfKeys = 64;  // keys per TMA box (one page of 64 or part of a larger page)

struct LogitsArgs {
    int paged;         // 1: K through a block table; 0: one contiguous K sequence
    int num_groups;    // paged: B; contiguous: ceil(M / G)
    int G;             // rows per group (paged: next_n)
    int total_rows;    // M (contiguous) or B * next_n (paged)
    int H;
    // query side
    const float *q_scale;  // FP8: nullable fp32 [rows, H]
    const uint8_t *q_sf;   // MXFP4: e8m0 [rows, H, D/32]
    const float *weights;  // [rows, H]
    // key side
    const uint8_t *kv;       // paged: page pool; contiguous: k
    int64_t page_stride;     // bytes between pages (paged)
    int num_pages;           // pages in the pool (paged)
    int page_size;           // tokens per page (paged)
    int page_shift;          // log2(page_size) if a power of two, else -1
    int64_t scale_off;       // byte offset of the scale block inside a page
    const float *k_scale;    // contiguous FP8: fp32 [N]
    const uint8_t *k_sf;     // contiguous MXFP4: e8m0 [N, D/32]
    const int32_t *bt;       // [B, bt_stride]
    int64_t bt_stride;
    int max_blocks;          // logical pages per sequence (columns of bt in use)
    // row ranges
    const int32_t *ctx;      // paged: context lengths
    int ctx_per_row;
    const int32_t *row_ks;   // nullable for paged
    const int32_t *row_ke;   // contiguous only
    int N;                   // contiguous: number of keys
    // fused candidate mask (paged; nullable)
    const int32_t *cand;
    int64_t cand_stride;
    int num_cand;
    int cand_block;
    int cand_shift;          // log2(cand_block) if a power of two, else -1
    int cand_words;          // 32-bit words of one row's candidate bitmap
    // output
    float *logits;
    int64_t ld;
    int width;               // paged: max_model_len; contiguous: N
    unsigned int *status;    // device status word (IDX_DEV_* bits)
    int tile_shift;          // log2 of the keys per tile (7 or 8)
    int group_cost;          // paged: units a CTA is charged for starting a row group
    // Block maxima of the candidate source (nullable): bmax[r, j] = max of the
    // row's logits over [ks + j * bmax_block, ks + (j + 1) * bmax_block),
    // prefilled with -inf and raised by atomics (bmax_block >= 32).
    float *bmax;
    int64_t ld_bmax;
    int bmax_block;
    int bmax_shift;          // log2(bmax_block) if a power of two, else -1
    // Digit-1 histograms for a chunked top-k that runs next (nullable):
    // hist[r][2048] counts the written finite logits of row r by their
    // order-preserving key's top 11 bits, hvalid[r] and cvalid[r][hist_P]
    // (per 8192-key chunk) count them; all cleared beforehand.
    uint32_t *hist;
    uint32_t *hvalid;
    uint32_t *cvalid;
    int hist_P;
    // Candidate gather plan (nullable), written by cand_plan_kernel: per row
    // group plan_words words: [0] the number n of compute tiles (tiles that
    // hold a candidate key of any of the group's rows), then box_words words
    // of per-64-key-box bits (boxes holding a candidate key), then the n
    // compute tile indices in ascending order.  Only those tiles are scored
    // and only those boxes loaded; every other key is -inf anyway.
    uint32_t *plan;
    int plan_words, box_words;
    int plan_fill;  // the plan kernel writes -inf over the tiles it does not list
};

// Plan bit of 64-key box b of group g (true without a plan).
__device__ __forceinline__ bool plan_box(const LogitsArgs &a, int g, int b)
{
    return !a.plan ||
           ((__ldg(a.plan + (size_t)g * a.plan_words + 1 + (b >> 5)) >> (b & 31)) & 1u);
}

// Key range [ks, ke) of row r, clamped as the oracle clamps it.
__device__ __forceinline__ void row_range(const LogitsArgs &a, int r, int &ks, int &ke)
{
    if (a.paged) {
        int e;
        if (a.ctx_per_row) {
            e = a.ctx[r];
        } else {
            int b = r / a.G, j = r - (r / a.G) * a.G;
            e = a.ctx[b] - a.G + j + 1;
        }
        ke = min(max(e, 0), a.width);
        ks = a.row_ks ? min(max(a.row_ks[r], 0), ke) : 0;
    } else {
        ke = min(max(a.row_ke[r], 0), a.N);
        ks = min(max(a.row_ks[r], 0), ke);
    }
}

struct GroupInfo {
    int row0, nrows;  // rows [row0, row0 + nrows)
    int lo, hi;       // union of the rows' live ranges: [min ks, max ke)
    int tiles;        // units of this group
};

__device__ __forceinline__ GroupInfo group_info_inline(const LogitsArgs &a, int g)
{
    GroupInfo gi;
    gi.row0 = g * a.G;
    gi.nrows = min(a.G, a.total_rows - gi.row0);
    int lo = 0x7fffffff, hi = 0;
    for (int i = 0; i < gi.nrows; ++i) {
        int ks, ke;
        row_range(a, gi.row0 + i, ks, ke);
        if (ke > ks) {
            lo = min(lo, ks);
            hi = max(hi, ke);
        }
    }
    if (hi <= 0)
        lo = 0;
    gi.lo = lo;
    gi.hi = hi;
    const int tk = 1 << a.tile_shift;
    if (a.paged)
        gi.tiles = (hi + tk - 1) >> a.tile_shift;  // columns [0, max ke) are written
    else
        gi.tiles = (a.N + tk - 1) >> a.tile_shift;  // every column of [0, N) is written
    return gi;
}

// Out of line on purpose: it runs once per group and inlining it into every
// role multiplies the kernel's code size several times over, which starves
// the instruction cache of the hot loops.
__device__ __noinline__ GroupInfo group_info(const LogitsArgs &a, int g)
{
    return group_info_inline(a, g);
}

__device__ __forceinline__ bool tile_is_compute(const GroupInfo &gi, int j, int shift)
{
    const int t0 = j << shift;
    return gi.hi > gi.lo && t0 < gi.hi && t0 + (1 << shift) > gi.lo;
}

// Walks this CTA's unit range in order.  Every role of the CTA runs its own
// copy and sees the same sequence.
struct UnitWalk {
    int g, j;          // current group and tile
    int k, n;          // unit index within the group, the group's units
    long long left;    // units still to visit (including the current one)
    GroupInfo gi;
    bool first_in_group;  // current unit is the first of its group in this range
};

} // namespace idx

namespace idx {

// Block-wide helpers for the schedule prologue (blockDim.x a multiple of 32).
__device__ __forceinline__ long long block_sum_ll(long long v, long long *scratch)
{
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        scratch[w] = v;
    __syncthreads();
    long long t = 0;
    for (int i = 0; i < nw; ++i)
        t += scratch[i];
    __syncthreads();
    return t;
}

// Inclusive block scan of v; *total gets the block total.
__device__ __forceinline__ long long block_incl_scan_ll(long long v, long long *scratch,
                                                        long long *total)
{
    int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int o = 1; o < 32; o <<= 1) {
        long long n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += n;
    }
    __syncthreads();
    if (lane == 31)
        scratch[w] = v;
    __syncthreads();
    long long off = 0, t = 0;
    for (int i = 0; i < nw; ++i) {
        if (i < w)
            off += scratch[i];
        t += scratch[i];
    }
    __syncthreads();
    *total = t;
    return v + off;
}

// Units of group g: all its tiles, or under a gather plan only its compute
// tiles (the plan kernel writes -inf over the others).
template <bool PLAN>
__device__ __forceinline__ long long group_units(const LogitsArgs &a, int g)
{
    if constexpr (PLAN)
        return (long long)__ldg(a.plan + (size_t)g * a.plan_words);
    else
        return group_info(a, g).tiles;
}

// Tile of unit k of group g: k itself, or under a gather plan the group's
// k-th compute tile.
template <bool PLAN>
__device__ __forceinline__ int unit_tile(const LogitsArgs &a, int g, int k)
{
    if constexpr (PLAN)
        return (int)__ldg(a.plan + (size_t)g * a.plan_words + 1 + a.box_words + k);
    else
        return k;
}

// Find this CTA's first unit: returns (g0, k0, n0) -- the group, the unit's
// index within it and the group's number of units -- and the CTA's number of
// units.  The CTAs split the units evenly.  Paged: every group with units
// also counts a.group_cost leading units that are never scored, so that a
// CTA whose range starts a group (new Q tile, row ranges and page window:
// a few microseconds of latency) gets that many fewer tiles; k0 and count
// include them and the walk skips them.  Thread t owns a contiguous range
// of groups, so one block scan of the per-thread unit counts places every
// range, and the one thread whose range holds the CTA's first unit walks it
// again (from L1) to find the group.
// scratch: >= blockDim.x/32 + 3 long longs of shared memory (at most 1024
// threads).
template <bool PLAN>
__device__ __forceinline__ void locate_units(const LogitsArgs &a, long long *scratch, int &g0,
                                             int &k0, int &n0, long long &count)
{
    if (!a.paged) {
        const int T = (a.N + (1 << a.tile_shift) - 1) >> a.tile_shift;
        const long long total = (long long)a.num_groups * T;
        const long long u0 = total * blockIdx.x / gridDim.x;
        count = total * (blockIdx.x + 1) / gridDim.x - u0;
        g0 = (int)(u0 / (T > 0 ? T : 1));
        k0 = (int)(u0 - (long long)g0 * T);
        n0 = T;
        if (count <= 0) {
            g0 = a.num_groups;
            k0 = 0;
            count = 0;
        }
        return;
    }
    const int m = (a.num_groups + (int)blockDim.x - 1) / (int)blockDim.x;
    const int gb = min((int)threadIdx.x * m, a.num_groups), ge = min(gb + m, a.num_groups);
    long long loc = 0;
    for (int g = gb; g < ge; ++g) {
        const long long v = group_units<PLAN>(a, g);
        loc += v > 0 ? v + a.group_cost : 0;
    }
    long long total;
    const long long start = block_incl_scan_ll(loc, scratch, &total) - loc;
    const long long u0 = total * blockIdx.x / gridDim.x;
    count = total * (blockIdx.x + 1) / gridDim.x - u0;
    if (count <= 0) {  // the same in every thread
        g0 = a.num_groups;
        k0 = 0;
        n0 = 0;
        count = 0;
        return;
    }
    volatile long long *found = scratch + 32;  // [0] = g0, [1] = unit within it, [2] = its units
    if (loc > 0 && u0 >= start && u0 < start + loc) {
        long long run = start;
        for (int g = gb; g < ge; ++g) {
            const long long v = group_units<PLAN>(a, g);
            const long long e = v > 0 ? v + a.group_cost : 0;
            if (u0 < run + e) {
                found[0] = g;
                found[1] = u0 - run;
                found[2] = v;
                break;
            }
            run += e;
        }
    }
    __syncthreads();
    g0 = (int)found[0];
    k0 = (int)found[1];
    n0 = (int)found[2];
    __syncthreads();
}

// The first unit's tile load and the group's row ranges are issued together
// (group_info inlined here: walk_begin runs once, before the roles split).
// k0 and count include the group's charged units (paged), which are skipped.
template <bool PLAN>
__device__ __forceinline__ void walk_begin(const LogitsArgs &a, UnitWalk &w, int g0, int k0,
                                           int n0, long long count)
{
    const int skip = a.paged ? max(a.group_cost - k0, 0) : 0;
    w.g = g0;
    w.k = a.paged ? max(k0 - a.group_cost, 0) : k0;
    w.n = n0;
    w.left = count - skip;
    w.first_in_group = true;
    if (w.left > 0) {
        w.j = unit_tile<PLAN>(a, g0, w.k);
        w.gi = group_info_inline(a, g0);
    }
}

__device__ __forceinline__ bool walk_last_in_group(const UnitWalk &w)
{
    return w.left == 1 || w.k + 1 >= w.n;
}

// At a group's first unit: whether the walk ends in this group.  It goes on
// to another group only if units are left after this group's beyond the
// next group's charged units (paged; walk_next charges them on entry).
__device__ __forceinline__ bool walk_group_is_last(const LogitsArgs &a, const UnitWalk &w)
{
    const long long after = (long long)w.k + w.left - w.n;
    return after <= (a.paged ? (long long)a.group_cost : 0LL);
}

// Next unit: the group's next one, else the first of the next group that
// has units (after its charged units, paged).
template <bool PLAN>
__device__ __forceinline__ void walk_next(const LogitsArgs &a, UnitWalk &w)
{
    ++w.k;
    --w.left;
    w.first_in_group = false;
    while (w.left > 0 && w.k >= w.n) {
        ++w.g;
        w.k = 0;
        w.first_in_group = true;
        w.gi = group_info(a, w.g);
        w.n = PLAN ? (int)group_units<PLAN>(a, w.g) : w.gi.tiles;
        if (w.n > 0 && a.paged)
            w.left -= a.group_cost;
    }
    if constexpr (PLAN) {
        if (w.left > 0)
            w.j = unit_tile<PLAN>(a, w.g, w.k);
    } else {
        w.j = w.k;
    }
}

} // namespace idx
