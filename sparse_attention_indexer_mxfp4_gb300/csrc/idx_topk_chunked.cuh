// idx_topk_chunked.cuh -- per-row top-k for long rows, spread over the
// whole GPU: every row is cut into chunks of kCh elements and each kernel
// below runs one CTA per (row, chunk) or per row, so a 131072-key row is
// worked on by 16 CTAs at once and rows of different lengths balance out.
//
// Same selection as idx_topk.cuh (order-preserving keys, non-finite keys
// never selected, 11/11/10-bit radix digits, ties taken lowest index first,
// output in ascending index order).  Cross-CTA state lives in the caller's
// workspace; the steps are separate launches, so no CTA waits for another.
//   hist     (row, chunk): digit-1 histogram merged into the row's histogram
//   pick     (row):        threshold bin b1 and the rank left in it
//   filter   (row, chunk): keys in b1 appended to the row's candidate list;
//                          keys above b1 counted per chunk
//   resolve  (row):        digits 2-3 on the candidates -> threshold key T
//                          and ties; per-chunk output offsets and tie quotas
//   write    (row, chunk): ordered write of the chunk's selected indices
#pragma once

#include <cstdint>

#include "idx_topk.cuh"

namespace idx {
namespace topk_chunked {

constexpr int kCh = 8192;             // elements per chunk
constexpr int kThreads = 256;         // per chunk CTA
constexpr int kVec = kCh / kThreads / 4;  // 8 float4 loads per thread
constexpr int kCap = 8192;            // candidates kept per row
constexpr int kRowThreads = 1024;
constexpr int kMaxChunks = 1024;      // chunks per row (ld <= 8M elements)
static_assert(kMaxChunks <= kRowThreads, "resolve takes one thread per chunk");

// Workspace layout (all 32-bit words; rows R, chunks per row P).  The first
// three arrays must be zero when a call starts.
struct Ws {
    uint32_t *hist;      // [R][2048]  row histograms of digit 1
    uint32_t *valid;     // [R]        valid (finite) keys per row
    uint32_t *ncand;     // [R]        candidates appended per row
    uint32_t *state;     // [R][4]     take_all, b1, rank left in b1
    uint32_t *cvalid;    // [R][P]     valid keys per chunk
    uint32_t *cgt;       // [R][P]     keys with digit 1 > b1 per chunk
    uint32_t *cbase;     // [R][P]     output offset of the chunk
    uint32_t *cquota;    // [R][P]     keys equal to T the chunk takes
    uint32_t *tkey;      // [R][2]     threshold key T
    uint32_t *cand_key;  // [R][kCap]
    int32_t *cand_idx;   // [R][kCap]
};

__host__ __device__ inline size_t ws_zeroed_bytes(int R)
{
    return (size_t)R * (2048 + 2) * 4;
}

__host__ __device__ inline size_t ws_bytes(int R, int P)
{
    return ws_zeroed_bytes(R) + (size_t)R * 4 * 4 + (size_t)R * P * 4 * 4 + (size_t)R * 2 * 4 +
           (size_t)R * kCap * 8;
}

__host__ __device__ inline Ws ws_carve(void *base, int R, int P)
{
    Ws w;
    uint32_t *p = static_cast<uint32_t *>(base);
    w.hist = p;
    p += (size_t)R * 2048;
    w.valid = p;
    p += R;
    w.ncand = p;
    p += R;
    w.state = p;
    p += (size_t)R * 4;
    w.cvalid = p;
    p += (size_t)R * P;
    w.cgt = p;
    p += (size_t)R * P;
    w.cbase = p;
    p += (size_t)R * P;
    w.cquota = p;
    p += (size_t)R * P;
    w.tkey = p;
    p += (size_t)R * 2;
    w.cand_key = p;
    p += (size_t)R * kCap;
    w.cand_idx = reinterpret_cast<int32_t *>(p);
    return w;
}

struct ChunkPos {
    int row, ch, c0, c1;  // chunk covers [c0, c1) of row; c0 >= c1 when empty
};

__device__ __forceinline__ ChunkPos chunk_pos(const int32_t *lengths, int64_t ld, int P)
{
    ChunkPos c;
    c.row = blockIdx.x / P;
    c.ch = blockIdx.x - c.row * P;
    const int len = max(0, min(lengths[c.row], (int)ld));
    c.c0 = c.ch * kCh;
    c.c1 = min(len, c.c0 + kCh);
    return c;
}

// The thread's 32 keys: elements c0 + 4 * (u * kThreads + tid) + e, u < 8,
// e < 4 (0 past c1).  Block-wide, step u covers a contiguous 1024-element run.
__device__ __forceinline__ void load_chunk(const float *rowp, int c0, int c1, bool vec,
                                           uint32_t (&k)[kVec][4])
{
    #pragma unroll
    for (int u = 0; u < kVec; ++u)
        topk_detail::load4(rowp, c0 + 4 * (u * kThreads + (int)threadIdx.x), c1, vec, k[u]);
}

// Sum over the CTA; red holds one word per warp.  Barriers on both sides,
// so red may be reused right after.
__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t *red)
{
    v = topk_detail::warp_sum(v);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0)
        red[w] = v;
    __syncthreads();
    uint32_t t = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
        t += red[i];
    __syncthreads();
    return t;
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

// ------------------------------------------------------------------ hist
__global__ void __launch_bounds__(kThreads)
    hist_kernel(const float *__restrict__ logits, int64_t ld, const int32_t *__restrict__ lengths,
                int P, Ws ws, int vec_ok)
{
    __shared__ uint32_t h[2048];
    __shared__ uint32_t red[kThreads / 32];
    const ChunkPos cp = chunk_pos(lengths, ld, P);
    if (cp.c0 >= cp.c1) {
        if (threadIdx.x == 0)
            ws.cvalid[(size_t)cp.row * P + cp.ch] = 0;
        return;
    }
    for (int i = threadIdx.x; i < 2048; i += kThreads)
        h[i] = 0u;
    __syncthreads();
    uint32_t k[kVec][4];
    load_chunk(logits + (size_t)cp.row * ld, cp.c0, cp.c1, vec_ok != 0, k);
    uint32_t n = 0;
    #pragma unroll
    for (int u = 0; u < kVec; ++u)
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if (k[u][e]) {
                ++n;
                atomicAdd(&h[k[u][e] >> 21], 1u);
            }
    n = block_sum(n, red);  // its barriers also publish h
    uint32_t *gh = ws.hist + (size_t)cp.row * 2048;
    for (int i = threadIdx.x; i < 2048; i += kThreads)
        if (h[i])
            atomicAdd(&gh[i], h[i]);
    if (threadIdx.x == 0) {
        atomicAdd(&ws.valid[cp.row], n);
        ws.cvalid[(size_t)cp.row * P + cp.ch] = n;
    }
}

// Descending-bin search over a shared histogram h[nb] with kRowThreads
// threads (2 bins each); result in sel[0..1].
__device__ __forceinline__ void row_find_bin(const uint32_t *h, int nb, uint32_t krem,
                                             uint32_t *wsum, uint32_t *sel)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    uint32_t loc[2];
    uint32_t lsum = 0;
    #pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int b = nb - 1 - (tid * 2 + j);
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
    for (int j = 0; j < 2; ++j) {
        const int b = nb - 1 - (tid * 2 + j);
        if (b >= 0 && before < krem && before + loc[j] >= krem) {
            sel[0] = (uint32_t)b;
            sel[1] = krem - before;
        }
        before += loc[j];
    }
    __syncthreads();
}

// ------------------------------------------------------------------ pick
__global__ void __launch_bounds__(kRowThreads) pick_kernel(int k, Ws ws)
{
    __shared__ uint32_t h[2048];
    __shared__ uint32_t wsum[kRowThreads / 32];
    __shared__ uint32_t sel[2];
    const int row = blockIdx.x;
    const uint32_t total = ws.valid[row];
    uint32_t *st = ws.state + (size_t)row * 4;
    if (total <= (uint32_t)k) {
        if (threadIdx.x == 0) {
            st[0] = 1;
            st[1] = 0;
            st[2] = 0;
        }
        return;
    }
    for (int i = threadIdx.x; i < 2048; i += kRowThreads)
        h[i] = ws.hist[(size_t)row * 2048 + i];
    __syncthreads();
    row_find_bin(h, 2048, (uint32_t)k, wsum, sel);
    if (threadIdx.x == 0) {
        st[0] = 0;
        st[1] = sel[0];
        st[2] = sel[1];
    }
}

// ---------------------------------------------------------------- filter
__global__ void __launch_bounds__(kThreads)
    filter_kernel(const float *__restrict__ logits, int64_t ld,
                  const int32_t *__restrict__ lengths, int P, Ws ws, int vec_ok)
{
    __shared__ uint32_t red[kThreads / 32];
    __shared__ uint32_t blk_base;
    const ChunkPos cp = chunk_pos(lengths, ld, P);
    const uint32_t *st = ws.state + (size_t)cp.row * 4;
    if (cp.c0 >= cp.c1 || st[0]) {
        if (threadIdx.x == 0)
            ws.cgt[(size_t)cp.row * P + cp.ch] = 0;
        return;
    }
    const uint32_t b1 = st[1];
    uint32_t k[kVec][4];
    load_chunk(logits + (size_t)cp.row * ld, cp.c0, cp.c1, vec_ok != 0, k);
    uint32_t gt = 0, nc = 0;
    #pragma unroll
    for (int u = 0; u < kVec; ++u)
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t d = k[u][e] >> 21;
            gt += k[u][e] && d > b1;
            nc += k[u][e] && d == b1;
        }
    // one reservation in the row's candidate list per CTA
    uint32_t ntot;
    const uint32_t off = block_excl(nc, red, &ntot);
    if (threadIdx.x == 0)
        blk_base = atomicAdd(&ws.ncand[cp.row], ntot);
    const uint32_t gtot = block_sum(gt, red);  // its barriers also publish blk_base
    if (threadIdx.x == 0)
        ws.cgt[(size_t)cp.row * P + cp.ch] = gtot;
    uint32_t pos = blk_base + off;
    uint32_t *ck = ws.cand_key + (size_t)cp.row * kCap;
    int32_t *ci = ws.cand_idx + (size_t)cp.row * kCap;
    #pragma unroll
    for (int u = 0; u < kVec; ++u)
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if (k[u][e] && (k[u][e] >> 21) == b1) {
                if (pos < (uint32_t)kCap) {
                    ck[pos] = k[u][e];
                    ci[pos] = cp.c0 + 4 * (u * kThreads + (int)threadIdx.x) + e;
                }
                ++pos;
            }
}

// --------------------------------------------------------------- resolve
struct ResolveShared {
    uint32_t h[2048];
    uint32_t wsum[kRowThreads / 32];
    uint32_t sel[2];
    uint32_t cgt[kMaxChunks];  // candidates > T per chunk (all keys > T when streaming)
    uint32_t ceq[kMaxChunks];  // keys == T per chunk
};

__global__ void __launch_bounds__(kRowThreads)
    resolve_kernel(const float *__restrict__ logits, int64_t ld,
                   const int32_t *__restrict__ lengths, int k, int P, Ws ws,
                   int32_t *__restrict__ out, int64_t ld_out, int vec_ok)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    ResolveShared &sh = *reinterpret_cast<ResolveShared *>(dsm);
    const int row = blockIdx.x, tid = threadIdx.x;
    const int len = max(0, min(lengths[row], (int)ld));
    const int nch = (len + kCh - 1) / kCh;
    const uint32_t *st = ws.state + (size_t)row * 4;
    const bool take_all = st[0] != 0;
    const float *rowp = logits + (size_t)row * ld;
    const bool vec = vec_ok != 0;
    for (int i = tid; i < nch; i += kRowThreads) {
        sh.cgt[i] = 0;
        sh.ceq[i] = 0;
    }
    uint32_t T = 0, ties = 0;
    bool overflow = false;
    if (!take_all) {
        const uint32_t ncand = ws.ncand[row];
        overflow = ncand > (uint32_t)kCap;
        const uint32_t *ck = ws.cand_key + (size_t)row * kCap;
        const int32_t *ci = ws.cand_idx + (size_t)row * kCap;
        uint32_t prefix = st[1] << 21, pmask = 0xFFE00000u, krem = st[2];
        for (int pass = 1; pass < 3; ++pass) {
            const int shift = pass == 1 ? 10 : 0;
            const int nb = pass == 1 ? 2048 : 1024;
            __syncthreads();
            for (int i = tid; i < 2048; i += kRowThreads)
                sh.h[i] = 0u;
            __syncthreads();
            if (!overflow) {
                for (uint32_t i = tid; i < ncand; i += kRowThreads) {
                    const uint32_t kk = ck[i];
                    if ((kk & pmask) == prefix)
                        atomicAdd(&sh.h[(kk >> shift) & (uint32_t)(nb - 1)], 1u);
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
            for (uint32_t i = tid; i < ncand; i += kRowThreads) {
                const uint32_t kk = ck[i];
                const int ch = ci[i] / kCh;
                if (kk > T)
                    atomicAdd(&sh.cgt[ch], 1u);
                else if (kk == T)
                    atomicAdd(&sh.ceq[ch], 1u);
            }
        } else {
            for (int i0 = 4 * tid; i0 < len; i0 += 4 * kRowThreads) {
                uint32_t kk[4];
                topk_detail::load4(rowp, i0, len, vec, kk);
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (kk[e] > T)
                        atomicAdd(&sh.cgt[(i0 + e) / kCh], 1u);
                    else if (kk[e] == T && kk[e])
                        atomicAdd(&sh.ceq[(i0 + e) / kCh], 1u);
                }
            }
        }
    }
    __syncthreads();
    // chunk offsets in index order, one thread per chunk; ties go to the
    // lowest chunks first
    uint32_t gt = 0, eq = 0;
    if (tid < nch) {
        if (take_all) {
            gt = ws.cvalid[(size_t)row * P + tid];
        } else {
            gt = sh.cgt[tid] + (overflow ? 0u : ws.cgt[(size_t)row * P + tid]);
            eq = sh.ceq[tid];
        }
    }
    uint32_t eq_tot, sel_tot;
    const uint32_t eq_run = block_excl(eq, sh.wsum, &eq_tot);
    const uint32_t take = eq_run >= ties ? 0u : min(eq, ties - eq_run);
    const uint32_t base = block_excl(gt + take, sh.wsum, &sel_tot);
    if (tid < nch) {
        ws.cbase[(size_t)row * P + tid] = base;
        ws.cquota[(size_t)row * P + tid] = take;
    }
    if (tid == 0)
        ws.tkey[(size_t)row * 2] = T;
    int32_t *orow = out + (size_t)row * ld_out;
    for (int j = (int)sel_tot + tid; j < k; j += kRowThreads)
        orow[j] = -1;
}

// ----------------------------------------------------------------- write
__global__ void __launch_bounds__(kThreads)
    write_kernel(const float *__restrict__ logits, int64_t ld,
                 const int32_t *__restrict__ lengths, int P, Ws ws, int32_t *__restrict__ out,
                 int64_t ld_out, int vec_ok)
{
    __shared__ uint32_t red[kThreads / 32];
    const ChunkPos cp = chunk_pos(lengths, ld, P);
    if (cp.c0 >= cp.c1)
        return;
    const bool take_all = ws.state[(size_t)cp.row * 4] != 0;
    const uint32_t T = take_all ? 0u : ws.tkey[(size_t)cp.row * 2];
    const uint32_t quota = ws.cquota[(size_t)cp.row * P + cp.ch];
    const uint32_t base = ws.cbase[(size_t)cp.row * P + cp.ch];
    uint32_t k[kVec][4];
    load_chunk(logits + (size_t)cp.row * ld, cp.c0, cp.c1, vec_ok != 0, k);
    int32_t *orow = out + (size_t)cp.row * ld_out;
    uint32_t written = 0, eq_seen = 0;
    #pragma unroll
    for (int u = 0; u < kVec; ++u) {
        // keys equal to T are taken in index order up to the chunk's quota
        uint32_t neq = 0;
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            neq += k[u][e] == T && k[u][e];
        uint32_t eq_tot = 0, er = 0;
        if (quota > 0)  // CTA-uniform
            er = eq_seen + block_excl(neq, red, &eq_tot);
        uint32_t take[4], nt = 0;
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
            bool t = k[u][e] > T;
            if (k[u][e] == T && k[u][e]) {
                t = er < quota;
                ++er;
            }
            take[e] = t;
            nt += t;
        }
        uint32_t tot;
        uint32_t pos = base + written + block_excl(nt, red, &tot);
        #pragma unroll
        for (int e = 0; e < 4; ++e)
            if (take[e])
                orow[pos++] = cp.c0 + 4 * (u * kThreads + (int)threadIdx.x) + e;
        written += tot;
        eq_seen += eq_tot;
    }
}

} // namespace topk_chunked
} // namespace idx
