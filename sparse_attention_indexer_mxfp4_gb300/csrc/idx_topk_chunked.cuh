// idx_topk_chunked.cuh -- per-row top-k for long rows, spread over the
// whole GPU: every row is cut into chunks of kCh elements, so a 131072-key
// row is worked on by 16 CTAs at once and rows of different lengths balance
// out.
//
// Same selection as idx_topk.cuh (order-preserving keys, non-finite keys
// never selected, 11/11/10-bit radix digits, ties taken lowest index first,
// output in ascending index order).  Cross-CTA state lives in the caller's
// workspace.  Two launches:
//   plan     (grid):       clears the counters and lists the non-empty
//                          (row, chunk) pairs ("items")
//   phases   (one cooperative grid, every CTA resident; the phases are
//             separated by grid barriers whose waits are bounded):
//     hist     per item:   digit-1 histogram merged into the row's histogram
//     filter   per item:   threshold bin b1 from the row's histogram; keys
//                          in b1 appended to the row's candidate list (one
//                          reservation per warp), keys above b1 counted
//     resolve  per row:    digits 2-3 on the candidates -> threshold key T
//                          and ties; per-chunk output offsets and tie quotas
//     write    per item:   ordered write of the chunk's selected indices,
//                          ranks from warp scans of packed per-step counts
// A row with no more valid keys than k takes all of them: filter and resolve
// skip the search and write takes every valid key.  Workspace words that
// other CTAs wrote in an earlier phase are read with ld.global.cg (L2), never
// through the non-coherent L1.
#pragma once

#include <cstdint>

#include "idx_common.cuh"
#include "idx_topk.cuh"

namespace idx {
namespace topk_chunked {

constexpr int kCh = 8192;                 // elements per chunk
constexpr int kThreads = 256;             // chunk kernels
constexpr int kVec = kCh / kThreads / 4;  // 8 float4 loads per thread
constexpr int kCap = 8192;                // candidates kept per row
constexpr int kRowThreads = 256;          // resolve: one CTA per row
constexpr int kMaxChunks = 1024;          // chunks per row (ld <= 8M elements)
constexpr int kChunksPerThread = kMaxChunks / kRowThreads;
constexpr int kPlanThreads = 1024;
constexpr int kCandBatch = 8;             // candidate loads in flight per thread
constexpr int kResident = 3;              // chunks a phase CTA keeps in shared memory
constexpr int kSlotBytes = kCh * 4;       // one resident chunk
// Control words: [0] live chunks, [1] grid barrier arrivals of the call.
constexpr int kCtrlWords = 32;

// Workspace (rows R, chunks per row P).  hist, valid and ncand are
// contiguous and cleared by the plan kernel; everything else is written
// before it is read within one call.
struct Ws {
    uint32_t *hist;      // [R][2048]  row histograms of digit 1
    uint32_t *valid;     // [R]        valid (finite) keys per row
    uint32_t *ncand;     // [R]        candidates appended per row
    uint32_t *state;     // [R][4]     -, b1, rank left in b1 (rows with > k valid keys)
    uint32_t *nitems;    // [kCtrlWords] live chunks, grid barrier words (see grid_sync)
    int4 *items;         // [R * P]    live chunks: row, chunk, first, end
    uint32_t *cvalid;    // [R][P]     valid keys per live chunk
    uint32_t *cgt;       // [R][P]     keys with digit 1 > b1 per live chunk
    uint32_t *cbase;     // [R][P]     output offset of the chunk
    uint32_t *cquota;    // [R][P]     keys equal to T the chunk takes
    uint32_t *tkey;      // [R][2]     threshold key T
    uint32_t *cand_key;  // [R][kCap]
    int32_t *cand_idx;   // [R][kCap]
};

// Carves the workspace starting at base (16-byte aligned); returns the bytes
// used.  With base == nullptr it only measures.
__host__ __device__ inline size_t ws_layout(void *base, int R, int P, Ws *w)
{
    const size_t r = (size_t)R, rp = (size_t)R * P;
    // word offsets of the arrays, in the order of the struct
    const size_t o_hist = 0, o_valid = o_hist + r * 2048, o_ncand = o_valid + r;
    const size_t o_state = o_ncand + r, o_nitems = o_state + r * 4;
    const size_t o_items = (o_nitems + kCtrlWords + 3) & ~(size_t)3;  // 16-byte aligned
    const size_t o_cvalid = o_items + rp * 4, o_cgt = o_cvalid + rp, o_cbase = o_cgt + rp;
    const size_t o_cquota = o_cbase + rp, o_tkey = o_cquota + rp, o_ck = o_tkey + r * 2;
    const size_t o_ci = o_ck + r * kCap, off = o_ci + r * kCap;
    if (w) {
        uint32_t *p = static_cast<uint32_t *>(base);
        w->hist = p + o_hist;
        w->valid = p + o_valid;
        w->ncand = p + o_ncand;
        w->state = p + o_state;
        w->nitems = p + o_nitems;
        w->items = reinterpret_cast<int4 *>(p + o_items);
        w->cvalid = p + o_cvalid;
        w->cgt = p + o_cgt;
        w->cbase = p + o_cbase;
        w->cquota = p + o_cquota;
        w->tkey = p + o_tkey;
        w->cand_key = p + o_ck;
        w->cand_idx = reinterpret_cast<int32_t *>(p + o_ci);
    }
    return off * 4;
}

__host__ __device__ inline size_t ws_bytes(int R, int P)
{
    return ws_layout(nullptr, R, P, nullptr);
}

// The thread's 32 keys: elements c0 + 4 * (u * kThreads + tid) + e, u < 8,
// e < 4 (0 past c1).  Block-wide, step u covers a contiguous 1024-element run.
__device__ __forceinline__ void load_chunk(const float *rowp, int c0, int c1, bool vec,
                                           uint32_t (&k)[kVec][4])
{
    topk_detail::load_keys<kVec>(rowp, c0 + 4 * (int)threadIdx.x, 4 * kThreads, c1, vec, k);
}

// Keys of a chunk from its shared-memory copy (slot != nullptr; elements
// past the chunk's n keys read as key 0) or else from global memory, in the
// same thread / step layout as load_chunk.
__device__ __forceinline__ void chunk_keys(const float *slot, const float *logits, int64_t ld,
                                           int4 item, bool vec, uint32_t (&k)[kVec][4])
{
    if (slot) {
        const int n = item.w - item.z;
        #pragma unroll
        for (int u = 0; u < kVec; ++u) {
            const int i0 = 4 * (u * kThreads + (int)threadIdx.x);
            const float4 v = reinterpret_cast<const float4 *>(slot)[u * kThreads + threadIdx.x];
            k[u][0] = i0 < n ? topk_detail::float_key(v.x) : 0u;
            k[u][1] = i0 + 1 < n ? topk_detail::float_key(v.y) : 0u;
            k[u][2] = i0 + 2 < n ? topk_detail::float_key(v.z) : 0u;
            k[u][3] = i0 + 3 < n ? topk_detail::float_key(v.w) : 0u;
        }
    } else {
        load_chunk(logits + (size_t)item.x * ld, item.z, item.w, vec, k);
    }
}

// Exclusive prefix of v over the CTA in thread order; *tot gets the total.
__device__ __forceinline__ uint32_t block_excl(uint32_t v, uint32_t *red, uint32_t *tot)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t wt;
    const uint32_t ex = topk_detail::warp_excl(v, lane, &wt);
    __syncthreads();
    if (lane == 0)
        red[w] = wt;
    __syncthreads();
    uint32_t off = ex, t = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
        if (i < w)
            off += red[i];
        t += red[i];
    }
    __syncthreads();
    *tot = t;
    return off;
}


__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t ld_cg(const uint32_t *p)
{
    return __ldcg(reinterpret_cast<const unsigned int *>(p));
}

// Valid keys always have a digit 1 of at least 4 (the smallest finite value,
// -FLT_MAX, maps to 0x00800000); key 0 (non-finite) has digit 0, so tests of
// the form digit > b1 or digit == b1 never pick it.

// ------------------------------------------------------------------ plan
// Every CTA clears a slice of hist / valid / ncand; CTA 0 also lists the
// live chunks in (row, chunk) order, stores their number and clears the
// grid barrier's arrival count.
__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const int32_t *__restrict__ lengths, int64_t ld, int R, int P, Ws ws,
                int zero_cvalid)
{
    __shared__ uint32_t red[kPlanThreads / 32];
    pdl_wait();  // the workspace and lengths may belong to the previous kernel until here
    const int tid = threadIdx.x;
    const size_t nz = (size_t)R * (2048 + 2);  // hist, valid, ncand are contiguous
    const size_t stride = (size_t)gridDim.x * kPlanThreads;
    uint4 *z4 = reinterpret_cast<uint4 *>(ws.hist);
    for (size_t i = (size_t)blockIdx.x * kPlanThreads + tid; i < nz / 4; i += stride)
        z4[i] = make_uint4(0u, 0u, 0u, 0u);
    if (blockIdx.x == 0 && tid < (int)(nz & 3))
        ws.hist[(nz & ~(size_t)3) + tid] = 0u;
    if (zero_cvalid)  // a logits kernel will count the chunks' valid keys into it
        for (size_t i = (size_t)blockIdx.x * kPlanThreads + tid; i < (size_t)R * P; i += stride)
            ws.cvalid[i] = 0u;
    if (blockIdx.x != 0)
        return;
    uint32_t carry = 0;
    for (int r0 = 0; r0 < R; r0 += kPlanThreads) {
        const int r = r0 + tid;
        const int len = r < R ? max(0, min(lengths[r], (int)ld)) : 0;
        const uint32_t n = (uint32_t)((len + kCh - 1) / kCh);
        uint32_t tot;
        const uint32_t off = carry + block_excl(n, red, &tot);
        for (uint32_t c = 0; c < n; ++c) {
            const int c0 = (int)c * kCh;
            ws.items[off + c] = make_int4(r, (int)c, c0, min(len, c0 + kCh));
        }
        carry += tot;
    }
    if (tid == 0) {
        ws.nitems[0] = carry;
        ws.nitems[1] = 0u;  // grid barrier arrivals of this call
    }
}

// ------------------------------------------------------------- phase hist
struct HistShared {
    uint32_t h[2048];
    uint32_t nvalid;
};

__device__ __forceinline__ void hist_item(const float *logits, int64_t ld, int P, const Ws &ws,
                                          bool vec, int4 item, const float *slot, HistShared &sh)
{
    uint32_t k[kVec][4];
    chunk_keys(slot, logits, ld, item, vec, k);
    for (int i = threadIdx.x; i < 2048; i += kThreads)
        sh.h[i] = 0u;
    if (threadIdx.x == 0)
        sh.nvalid = 0u;
    __syncthreads();
    uint32_t n = 0;
    #pragma unroll
    for (int u = 0; u < kVec; ++u)
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if (k[u][e]) {
                ++n;
                atomicAdd(&sh.h[k[u][e] >> 21], 1u);
            }
    n = topk_detail::warp_sum(n);
    if ((threadIdx.x & 31) == 0 && n)
        atomicAdd(&sh.nvalid, n);
    __syncthreads();
    uint32_t *gh = ws.hist + (size_t)item.x * 2048;
    for (int i = threadIdx.x; i < 2048; i += kThreads)
        if (sh.h[i])
            atomicAdd(&gh[i], sh.h[i]);
    if (threadIdx.x == 0) {
        atomicAdd(&ws.valid[item.x], sh.nvalid);
        ws.cvalid[(size_t)item.x * P + item.y] = sh.nvalid;
    }
    __syncthreads();  // h and nvalid are cleared again for the next item
}

// ----------------------------------------------------------- phase filter
struct FilterShared {
    uint32_t red[kThreads / 32];
    uint32_t sel[2];
    uint32_t ngt;
};

__device__ __forceinline__ void filter_item(const float *logits, int64_t ld, int k, int P,
                                            const Ws &ws, bool vec, int4 item, const float *slot,
                                            FilterShared &sh)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int row = item.x;
    if (ld_cg(ws.valid + row) <= (uint32_t)k)
        return;  // the row takes all its valid keys (CTA-uniform)
    uint32_t key[kVec][4];
    chunk_keys(slot, logits, ld, item, vec, key);

    // threshold bin b1 of the row: thread t holds bins 2047 - 8t down to
    // 2040 - 8t; the count from the top reaches k in exactly one
    const uint4 *gh = reinterpret_cast<const uint4 *>(ws.hist + (size_t)row * 2048);
    const uint4 hi = __ldcg(gh + ((2044 - 8 * tid) >> 2)), lo = __ldcg(gh + ((2040 - 8 * tid) >> 2));
    const uint32_t loc[8] = {hi.w, hi.z, hi.y, hi.x, lo.w, lo.z, lo.y, lo.x};
    uint32_t lsum = 0;
    #pragma unroll
    for (int j = 0; j < 8; ++j)
        lsum += loc[j];
    uint32_t wt;
    uint32_t before = topk_detail::warp_excl(lsum, lane, &wt);
    __syncthreads();  // the previous item is done with red, sel and ngt
    if (lane == 0)
        sh.red[w] = wt;
    if (tid == 0)
        sh.ngt = 0u;
    __syncthreads();
    for (int i = 0; i < w; ++i)
        before += sh.red[i];
    #pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (before < (uint32_t)k && before + loc[j] >= (uint32_t)k) {
            sh.sel[0] = (uint32_t)(2047 - 8 * tid - j);
            sh.sel[1] = (uint32_t)k - before;
        }
        before += loc[j];
    }
    __syncthreads();
    const uint32_t b1 = sh.sel[0];
    if (item.y == 0 && tid == 0) {
        uint32_t *st = ws.state + (size_t)row * 4;
        st[1] = b1;
        st[2] = sh.sel[1];
    }

    uint32_t gt = 0, nc = 0;
    #pragma unroll
    for (int u = 0; u < kVec; ++u)
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t d = key[u][e] >> 21;
            gt += d > b1;
            nc += d == b1;
        }
    gt = topk_detail::warp_sum(gt);
    if (lane == 0 && gt)
        atomicAdd(&sh.ngt, gt);
    // candidates: one reservation in the row's list per warp
    uint32_t wtot;
    const uint32_t off = topk_detail::warp_excl(nc, lane, &wtot);
    uint32_t base = 0;
    if (lane == 0 && wtot)
        base = atomicAdd(&ws.ncand[row], wtot);
    uint32_t pos = __shfl_sync(0xffffffffu, base, 0) + off;
    uint32_t *ck = ws.cand_key + (size_t)row * kCap;
    int32_t *ci = ws.cand_idx + (size_t)row * kCap;
    #pragma unroll
    for (int u = 0; u < kVec; ++u)
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((key[u][e] >> 21) == b1) {
                if (pos < (uint32_t)kCap) {
                    ck[pos] = key[u][e];
                    ci[pos] = item.z + 4 * (u * kThreads + tid) + e;
                }
                ++pos;
            }
    __syncthreads();
    if (tid == 0)
        ws.cgt[(size_t)row * P + item.y] = sh.ngt;
}

// Descending-bin search over a shared histogram h[nb] (nb <= 2048) with
// kRowThreads threads, BPT bins each: the bin where the count from the top
// reaches krem, and the rank left inside it, go to sel[0..1].  Barriers on
// both sides.
__device__ __forceinline__ void row_find_bin(const uint32_t *h, int nb, uint32_t krem,
                                             uint32_t *wsum, uint32_t *sel)
{
    constexpr int BPT = 2048 / kRowThreads;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    uint32_t loc[BPT];
    uint32_t lsum = 0;
    #pragma unroll
    for (int j = 0; j < BPT; ++j) {
        const int b = nb - 1 - (tid * BPT + j);
        loc[j] = b >= 0 ? h[b] : 0u;
        lsum += loc[j];
    }
    uint32_t wt;
    const uint32_t ex = topk_detail::warp_excl(lsum, lane, &wt);
    __syncthreads();
    if (lane == 0)
        wsum[w] = wt;
    __syncthreads();
    uint32_t before = ex;
    for (int i = 0; i < w; ++i)
        before += wsum[i];
    #pragma unroll
    for (int j = 0; j < BPT; ++j) {
        const int b = nb - 1 - (tid * BPT + j);
        if (b >= 0 && before < krem && before + loc[j] >= krem) {
            sel[0] = (uint32_t)b;
            sel[1] = krem - before;
        }
        before += loc[j];
    }
    __syncthreads();
}

// ---------------------------------------------------------- phase resolve
struct ResolveShared {
    uint32_t h[2048];
    uint32_t wsum[kRowThreads / 32];
    uint32_t sel[2];
    uint32_t cgt[kMaxChunks];  // candidates > T per chunk (all keys > T when streaming)
    uint32_t ceq[kMaxChunks];  // keys == T per chunk
};

__device__ __forceinline__ void resolve_row(const float *logits, int64_t ld,
                                            const int32_t *lengths, int k, int P, const Ws &ws,
                                            bool vec, int row, ResolveShared &sh, int32_t *out,
                                            int64_t ld_out)
{
    const int tid = threadIdx.x;
    const int len = max(0, min(lengths[row], (int)ld));
    const int nch = (len + kCh - 1) / kCh;
    const bool take_all = ld_cg(ws.valid + row) <= (uint32_t)k;
    const float *rowp = logits + (size_t)row * ld;
    for (int i = tid; i < nch; i += kRowThreads) {
        sh.cgt[i] = 0;
        sh.ceq[i] = 0;
    }
    uint32_t T = 0, ties = 0;
    bool overflow = false;
    if (!take_all) {
        const uint32_t *st = ws.state + (size_t)row * 4;
        const uint32_t ncand = ld_cg(ws.ncand + row);
        overflow = ncand > (uint32_t)kCap;
        const uint32_t *ck = ws.cand_key + (size_t)row * kCap;
        const int32_t *ci = ws.cand_idx + (size_t)row * kCap;
        uint32_t prefix = ld_cg(st + 1) << 21, pmask = 0xFFE00000u, krem = ld_cg(st + 2);
        for (int pass = 1; pass < 3; ++pass) {
            const int shift = pass == 1 ? 10 : 0;
            const int nb = pass == 1 ? 2048 : 1024;
            __syncthreads();
            for (int i = tid; i < 2048; i += kRowThreads)
                sh.h[i] = 0u;
            __syncthreads();
            if (!overflow) {
                // kCandBatch loads in flight per thread (keys past ncand read 0,
                // which matches no prefix)
                for (uint32_t i0 = tid; i0 < ncand; i0 += kCandBatch * kRowThreads) {
                    uint32_t kk[kCandBatch];
                    #pragma unroll
                    for (int j = 0; j < kCandBatch; ++j) {
                        const uint32_t i = i0 + j * kRowThreads;
                        kk[j] = i < ncand ? ld_cg(ck + i) : 0u;
                    }
                    #pragma unroll
                    for (int j = 0; j < kCandBatch; ++j)
                        if (kk[j] && (kk[j] & pmask) == prefix)
                            atomicAdd(&sh.h[(kk[j] >> shift) & (uint32_t)(nb - 1)], 1u);
                }
            } else {  // the list overflowed: stream the row
                for (int i0 = 4 * tid; i0 < len; i0 += 4 * kRowThreads) {
                    uint32_t kk[4];
                    topk_detail::load4(rowp, i0, len, vec, kk);
                    #pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (kk[e] && (kk[e] & pmask) == prefix)
                            atomicAdd(&sh.h[(kk[e] >> shift) & (uint32_t)(nb - 1)], 1u);
                }
            }
            __syncthreads();
            row_find_bin(sh.h, nb, krem, sh.wsum, sh.sel);
            prefix |= sh.sel[0] << shift;
            pmask |= (uint32_t)(nb - 1) << shift;
            krem = sh.sel[1];
        }
        T = prefix;
        ties = krem;
        // per-chunk counts of keys > T and == T
        if (!overflow) {
            const uint32_t *ciw = reinterpret_cast<const uint32_t *>(ci);
            for (uint32_t i0 = tid; i0 < ncand; i0 += kCandBatch * kRowThreads) {
                uint32_t kk[kCandBatch], cc[kCandBatch];
                #pragma unroll
                for (int j = 0; j < kCandBatch; ++j) {
                    const uint32_t i = i0 + j * kRowThreads;
                    kk[j] = i < ncand ? ld_cg(ck + i) : 0u;  // 0 is neither > T nor == T
                    cc[j] = i < ncand ? ld_cg(ciw + i) : 0u;
                }
                #pragma unroll
                for (int j = 0; j < kCandBatch; ++j) {
                    const int ch = (int)cc[j] / kCh;
                    if (kk[j] > T)
                        atomicAdd(&sh.cgt[ch], 1u);
                    else if (kk[j] == T)
                        atomicAdd(&sh.ceq[ch], 1u);
                }
            }
        } else {
            for (int i0 = 4 * tid; i0 < len; i0 += 4 * kRowThreads) {
                uint32_t kk[4];
                topk_detail::load4(rowp, i0, len, vec, kk);
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (kk[e] > T)
                        atomicAdd(&sh.cgt[(i0 + e) / kCh], 1u);
                    else if (kk[e] == T)
                        atomicAdd(&sh.ceq[(i0 + e) / kCh], 1u);
                }
            }
        }
    }
    __syncthreads();
    // chunk offsets in index order; thread t owns chunks CPT*t .. CPT*t+CPT-1.
    // Ties go to the lowest chunks first.
    constexpr int CPT = kChunksPerThread;
    uint32_t gt[CPT], eq[CPT], eq_sum = 0;
    #pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const int ch = CPT * tid + j;
        gt[j] = 0;
        eq[j] = 0;
        if (ch < nch) {
            if (take_all) {
                gt[j] = ld_cg(ws.cvalid + (size_t)row * P + ch);
            } else {
                gt[j] = sh.cgt[ch] + (overflow ? 0u : ld_cg(ws.cgt + (size_t)row * P + ch));
                eq[j] = sh.ceq[ch];
            }
        }
        eq_sum += eq[j];
    }
    uint32_t eq_tot, sel_tot;
    uint32_t eq_run = block_excl(eq_sum, sh.wsum, &eq_tot);
    uint32_t take[CPT], sel_sum = 0;
    #pragma unroll
    for (int j = 0; j < CPT; ++j) {
        take[j] = eq_run >= ties ? 0u : min(eq[j], ties - eq_run);
        eq_run += eq[j];
        sel_sum += gt[j] + take[j];
    }
    uint32_t base = block_excl(sel_sum, sh.wsum, &sel_tot);
    #pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const int ch = CPT * tid + j;
        if (ch < nch) {
            ws.cbase[(size_t)row * P + ch] = base;
            ws.cquota[(size_t)row * P + ch] = take[j];
        }
        base += gt[j] + take[j];
    }
    if (tid == 0)
        ws.tkey[(size_t)row * 2] = T;
    int32_t *orow = out + (size_t)row * ld_out;
    for (int j = (int)sel_tot + tid; j < k; j += kRowThreads)
        orow[j] = -1;
    __syncthreads();  // sh is reused by the next row
}

// ------------------------------------------------------------ phase write
//
// Ranks in index order over a chunk.  Step u of the chunk covers elements
// first + 1024u + 4 * tid + e, so index order is (u, warp, lane, e).  f[u]
// holds the thread's flags of step u (bit e).  The per-lane counts of the
// eight steps are packed 8 bits each into two words, so two warp scans give
// every step's lane prefix and warp total at once (a field never exceeds
// 128); warp 0 then scans the 64 (step, warp) totals in shared memory.
// rank[u] receives the number of flagged elements of the chunk before the
// thread's first element of step u.  All threads call it; it ends with a
// barrier, so tab may be reused right after.
constexpr int kTab = kVec * (kThreads / 32) + 1;

__device__ __forceinline__ void chunk_ranks(const uint32_t (&f)[kVec], uint32_t *tab,
                                            uint32_t (&rank)[kVec])
{
    constexpr int NW = kThreads / 32;
    static_assert(kVec == 8 && kVec * NW == 64, "packed layout assumes 8 steps of 8 warps");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t p0 = 0, p1 = 0;
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
        p0 |= (uint32_t)__popc(f[u]) << (8 * u);
        p1 |= (uint32_t)__popc(f[u + 4]) << (8 * u);
    }
    uint32_t x0 = p0, x1 = p1;
    #pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n0 = __shfl_up_sync(0xffffffffu, x0, o);
        const uint32_t n1 = __shfl_up_sync(0xffffffffu, x1, o);
        if (lane >= o) {
            x0 += n0;
            x1 += n1;
        }
    }
    const uint32_t t0 = __shfl_sync(0xffffffffu, x0, 31);
    const uint32_t t1 = __shfl_sync(0xffffffffu, x1, 31);
    x0 -= p0;  // exclusive lane prefixes
    x1 -= p1;
    if (lane < kVec)
        tab[lane * NW + w] = ((lane < 4 ? t0 : t1) >> (8 * (lane & 3))) & 0xFFu;
    __syncthreads();
    if (w == 0) {
        const uint32_t a0 = tab[2 * lane], a1 = tab[2 * lane + 1];
        uint32_t t;
        const uint32_t ex = topk_detail::warp_excl(a0 + a1, lane, &t);
        tab[2 * lane] = ex;
        tab[2 * lane + 1] = ex + a0;
    }
    __syncthreads();
    #pragma unroll
    for (int u = 0; u < kVec; ++u)
        rank[u] = tab[u * NW + w] + (((u < 4 ? x0 : x1) >> (8 * (u & 3))) & 0xFFu);
    __syncthreads();
}

__device__ __forceinline__ void write_item(const float *logits, int64_t ld, int k, int P,
                                           const Ws &ws, bool vec, int4 item, const float *slot,
                                           uint32_t *tab, int32_t *out, int64_t ld_out)
{
    const int row = item.x;
    uint32_t key[kVec][4];
    chunk_keys(slot, logits, ld, item, vec, key);
    const bool take_all = ld_cg(ws.valid + row) <= (uint32_t)k;
    const uint32_t tk = ld_cg(ws.tkey + (size_t)row * 2);
    const uint32_t quota = ld_cg(ws.cquota + (size_t)row * P + item.y);
    const uint32_t base = ld_cg(ws.cbase + (size_t)row * P + item.y);
    // keys equal to T are taken in index order up to the chunk's quota;
    // T = 0 under take_all, and key 0 is never taken
    const uint32_t T = take_all ? 0u : tk;
    uint32_t ftake[kVec], feq[kVec];
    #pragma unroll
    for (int u = 0; u < kVec; ++u) {
        ftake[u] = 0;
        feq[u] = 0;
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
            ftake[u] |= (uint32_t)(key[u][e] > T) << e;
            feq[u] |= (uint32_t)(key[u][e] == T && T != 0u) << e;
        }
    }
    uint32_t rank[kVec];
    if (quota > 0) {  // CTA-uniform
        chunk_ranks(feq, tab, rank);
        #pragma unroll
        for (int u = 0; u < kVec; ++u)
            #pragma unroll
            for (int e = 0; e < 4; ++e)
                if ((feq[u] >> e) & 1u) {
                    const uint32_t r = rank[u] + __popc(feq[u] & ((1u << e) - 1u));
                    ftake[u] |= (uint32_t)(r < quota) << e;
                }
    }
    chunk_ranks(ftake, tab, rank);
    int32_t *orow = out + (size_t)row * ld_out;
    #pragma unroll
    for (int u = 0; u < kVec; ++u) {
        uint32_t pos = base + rank[u];
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((ftake[u] >> e) & 1u)
                orow[pos++] = item.z + 4 * (u * kThreads + (int)threadIdx.x) + e;
    }
}

// ------------------------------------------------------------ the phases
//
// Grid barrier for a cooperative launch (every CTA resident).  ctrl[1]
// counts arrivals over the whole call (the plan kernel clears it): the n-th
// barrier is passed once the count reaches n * gridDim.x.  Thread 0 arrives
// with a release add, so the CTA's earlier writes (ordered before it by the
// CTA barrier) are visible to every CTA that then reads the count with an
// acquire load.  The wait is bounded (limit_ns, two seconds by default),
// after which the status gets the timeout bit and the CTA stops.
__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.add.release.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool grid_sync(uint32_t *ctrl, unsigned *status,
                                          volatile uint32_t *abort_sh,
                                          uint64_t limit_ns = 2000000000ull)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t *count = ctrl + 1;
        const uint32_t old = atom_add_release_gpu(count, 1u);
        const uint32_t target = (old / gridDim.x + 1u) * gridDim.x;
        if (ld_acquire_gpu(count) < target) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(count) < target) {
                __nanosleep(20);
                if (globaltimer_ns() - t0 > limit_ns) {
                    atomicOr(status, kDevTimeout);
                    *abort_sh = 1u;
                    break;
                }
            }
        }
    }
    __syncthreads();
    return *abort_sh == 0u;
}

struct PhaseArgs {
    const float *logits;
    int64_t ld;
    const int32_t *lengths;
    int R, P, k;
    int32_t *out;
    int64_t ld_out;
    int vec_ok;
    int hist_done;  // the row histograms and valid counts are already in ws
    unsigned *status;
    Ws ws;
};

union PhaseShared {
    HistShared hist;
    FilterShared filter;
    ResolveShared resolve;
    uint32_t tab[kTab];
};

static_assert(kRowThreads == kThreads, "the resolve phase runs in the chunk CTAs");

// Dynamic shared memory of the phases kernel: kResident chunk slots.
constexpr int kPhaseDynSmem = kResident * kSlotBytes;

__global__ void __launch_bounds__(kThreads, 2) phases_kernel(const __grid_constant__ PhaseArgs a)
{
    __shared__ PhaseShared sh;
    __shared__ uint32_t abort_flag;
    __shared__ int wait_abort;
    __shared__ __align__(8) uint64_t slot_full[kResident];
    extern __shared__ __align__(128) uint8_t dyn[];
    const bool vec = a.vec_ok != 0;
    const uint32_t nitems = a.ws.nitems[0];
    uint32_t *ctrl = a.ws.nitems;
    // The CTA's j-th item is blockIdx.x + j * gridDim.x; the first kResident
    // of them are copied into shared memory once (one bulk copy each, needs
    // 16-byte aligned rows) and every phase reads them from there.
    const bool resident = vec;
    if (threadIdx.x == 0) {
        abort_flag = 0u;
        wait_abort = 0;
        for (int j = 0; j < kResident; ++j)
            mbar_init(&slot_full[j], 1);
        fence_mbar_init();
        if (resident)
            for (int j = 0; j < kResident; ++j) {
                const uint32_t it = blockIdx.x + (uint32_t)j * gridDim.x;
                if (it >= nitems)
                    break;
                const int4 item = a.ws.items[it];
                // whole 16-byte groups: the row holds ld (a multiple of 4) floats
                const uint32_t bytes = (uint32_t)(((item.w - item.z) * 4 + 15) & ~15);
                mbar_arrive_expect_tx(&slot_full[j], bytes);
                bulk_load(dyn + j * kSlotBytes, a.logits + (size_t)item.x * a.ld + item.z, bytes,
                          &slot_full[j]);
            }
    }
    __syncthreads();
    auto slot_of = [&](int j) -> const float * {
        return resident && j < kResident ? reinterpret_cast<const float *>(dyn + j * kSlotBytes)
                                         : nullptr;
    };
    // the first phase that reads a resident chunk waits for its copy
    auto slot_wait = [&](int j) {
        if (resident && j < kResident && !mbar_wait(&slot_full[j], 0u, &wait_abort, a.status))
            abort_flag = 1u;  // a copy did not land in time: stop at the next barrier
    };
    // leaving after an abort: the chunk copies this CTA issued land first
    auto drain_slots = [&]() {
        if (threadIdx.x == 0 && resident)
            for (int jj = 0; jj < kResident; ++jj) {
                if (blockIdx.x + (uint32_t)jj * gridDim.x >= nitems)
                    break;
                mbar_wait_drain(&slot_full[jj], 0u);
            }
    };
    int j = 0;
    if (!a.hist_done) {
        for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x, ++j) {
            slot_wait(j);
            hist_item(a.logits, a.ld, a.P, a.ws, vec, a.ws.items[it], slot_of(j), sh.hist);
        }
        if (!grid_sync(ctrl, a.status, &abort_flag)) {
            drain_slots();
            return;
        }
    }
    j = 0;
    for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x, ++j) {
        if (a.hist_done)
            slot_wait(j);
        filter_item(a.logits, a.ld, a.k, a.P, a.ws, vec, a.ws.items[it], slot_of(j), sh.filter);
    }
    if (!grid_sync(ctrl, a.status, &abort_flag)) {
        drain_slots();
        return;
    }
    for (int row = blockIdx.x; row < a.R; row += gridDim.x)
        resolve_row(a.logits, a.ld, a.lengths, a.k, a.P, a.ws, vec, row, sh.resolve, a.out,
                    a.ld_out);
    if (!grid_sync(ctrl, a.status, &abort_flag)) {
        drain_slots();
        return;
    }
    j = 0;
    for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x, ++j)
        write_item(a.logits, a.ld, a.k, a.P, a.ws, vec, a.ws.items[it], slot_of(j), sh.tab,
                   a.out, a.ld_out);
}

} // namespace topk_chunked
} // namespace idx
