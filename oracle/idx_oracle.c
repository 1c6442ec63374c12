/*
 * idx_oracle.c -- plain scalar CPU oracle for the sparse-attention lightning
 * indexer.  TEST INFRASTRUCTURE ONLY: the product library never links,
 * loads or calls anything in this directory; only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg do.
 *
 * Everything here is written for a reader checking it against the vLLM API
 * pages it restates, not for speed:
 *   - "vllm.v1.attention.ops.rocm_aiter_mla_sparse", section
 *     fp8_mqa_logits_torch: logits[m,n] = sum_h w[m,h] * relu(k_scale[n] *
 *     (q[m,h,:] . k[n,:])), masked to -inf outside [ks[m], ke[m]).
 *   - same page, rocm_fp8_paged_mqa_logits / rocm_fp8_paged_mqa_logits_triton:
 *     the same score over a K cache cut into pages reached through a block
 *     table; page layout "[block_size * D e4m3 bytes][block_size fp32 scales]".
 *   - same page, _apply_candidate_mask_strided: keep only candidate blocks of
 *     each row inside [0, end).
 *   - "vllm.v1.attention.ops.rocm_paged_mxfp4_indexer", section _topk: top-k
 *     over each row's [0, lengths[row]), -1 pads rows shorter than k;
 *     section rocm_mxfp4_sparse_attn_indexer: MXFP4 q/k (packed e2m1 with one
 *     ue8m0 scale per 32 elements).
 *   - rocm_aiter_mla_sparse, build_prefill_topk_ragged_indices and the page
 *     "rocm_aiter_mla" (_expand_page_indices_kernel): position p of a
 *     sequence lives at cache slot block_table[b, p / P] * P + p % P.
 *
 * Arithmetic: every stored byte is decoded exactly to double; dot products,
 * scales, ReLU and the head sum are done in double in the order the formula
 * reads (d ascending, then h ascending) and rounded once to float at the end.
 * The pages' reference rounds the per-head score to bf16 (its einsum runs in
 * bf16); the oracle drops that intermediate rounding on purpose, so it is the
 * exact formula.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_*.py against
 * closed forms, exhaustive decode tables, integer recomputation, brute force
 * on tiny inputs and invariants.  None is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_FMT_FP8 0
#define ORC_FMT_MXFP4 1

/* ------------------------------------------------------------------------ */
/* Exact decoders.                                                          */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there
 * is no infinity.  Largest finite magnitude 448. */
double orc_e4m3_to_double(uint8_t v)
{
    int s = (v >> 7) & 1;
    int e = (v >> 3) & 0xF;
    int m = v & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* OCP FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * exponent 0 is subnormal (m/2); magnitudes of codes 0..7 are
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_to_double(uint8_t nibble)
{
    int s = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 0x3;
    int m = nibble & 0x1;
    double mag;
    if (e == 0)
        mag = (double)m * 0.5;
    else
        mag = ldexp(1.0 + (double)m / 2.0, e - 1);
    return s ? -mag : mag;
}

/* OCP E8M0 scale: 2^(v - 127); 0xFF is NaN. */
double orc_e8m0_to_double(uint8_t v)
{
    if (v == 0xFF)
        return NAN;
    return ldexp(1.0, (int)v - 127);
}

/* Element i of a packed e2m1 vector: element 2j is the low nibble of byte j,
 * element 2j+1 the high nibble (OCP MX convention). */
static double mx_elem(const uint8_t *packed, const uint8_t *scales, int i)
{
    uint8_t byte = packed[i / 2];
    uint8_t nib = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    return orc_e2m1_to_double(nib) * orc_e8m0_to_double(scales[i / 32]);
}

/* Decode one stored vector of D elements to double.
 * FP8: D bytes of e4m3.  MXFP4: D/2 packed bytes + D/32 e8m0 scale bytes. */
static void decode_vec(int fmt, const uint8_t *vals, const uint8_t *scales,
                       int D, double *out)
{
    for (int d = 0; d < D; ++d) {
        if (fmt == ORC_FMT_FP8)
            out[d] = orc_e4m3_to_double(vals[d]);
        else
            out[d] = mx_elem(vals, scales, d);
    }
}

/* ------------------------------------------------------------------------ */
/* A tiny parallel-for over rows (threads own disjoint rows).               */
/* ------------------------------------------------------------------------ */

typedef void (*row_fn)(void *ctx, int row);

struct par_arg {
    row_fn fn;
    void *ctx;
    int rows, tid, nthreads;
};

static void *par_worker(void *p)
{
    struct par_arg *a = (struct par_arg *)p;
    for (int r = a->tid; r < a->rows; r += a->nthreads)
        a->fn(a->ctx, r);
    return NULL;
}

int orc_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void parallel_rows(row_fn fn, void *ctx, int rows, int nthreads)
{
    if (nthreads <= 0)
        nthreads = orc_default_threads();
    if (nthreads > rows)
        nthreads = rows;
    if (nthreads <= 1) {
        for (int r = 0; r < rows; ++r)
            fn(ctx, r);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    struct par_arg *args = (struct par_arg *)malloc(sizeof(struct par_arg) * nthreads);
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn;
        args[t].ctx = ctx;
        args[t].rows = rows;
        args[t].tid = t;
        args[t].nthreads = nthreads;
        pthread_create(&th[t], NULL, par_worker, &args[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    free(th);
    free(args);
}

/* ------------------------------------------------------------------------ */
/* The per-(row, key) score.                                                */
/* ------------------------------------------------------------------------ */

/* logit = sum_h w[h] * max(0, k_scale * q_scale[h] * (q[h,:] . k[:])),
 * all in double, d ascending then h ascending, rounded once to float.
 * qd is the row's decoded queries [H][D]; qs its per-head scales (1.0 when
 * the format has none); kd the decoded key; ksc the key's scale. */
static float score_one(const double *qd, const double *qs, const float *w,
                       const double *kd, double ksc, int H, int D)
{
    double acc = 0.0;
    for (int h = 0; h < H; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qd[(size_t)h * D + d] * kd[d];
        double s = ksc * qs[h] * dot;
        double relu = s > 0.0 ? s : 0.0;
        if (isnan(s))
            relu = s; /* NaN propagates; it is never produced by valid data */
        acc += (double)w[h] * relu;
    }
    return (float)acc;
}

/* Decode the H query vectors (and per-head scales) of logits row r. */
static void decode_row_q(int fmt, const uint8_t *q, const void *q_scale, int r,
                         int H, int D, double *qd, double *qs)
{
    for (int h = 0; h < H; ++h) {
        if (fmt == ORC_FMT_FP8) {
            decode_vec(fmt, q + ((size_t)r * H + h) * D, NULL, D, qd + (size_t)h * D);
            qs[h] = q_scale ? (double)((const float *)q_scale)[(size_t)r * H + h] : 1.0;
        } else {
            const uint8_t *sc = (const uint8_t *)q_scale + ((size_t)r * H + h) * (D / 32);
            decode_vec(fmt, q + ((size_t)r * H + h) * (D / 2), sc, D, qd + (size_t)h * D);
            qs[h] = 1.0;
        }
    }
}

static int clampi(int v, int lo, int hi)
{
    return v < lo ? lo : (v > hi ? hi : v);
}

/* ------------------------------------------------------------------------ */
/* Contiguous (non-paged) logits: fp8_mqa_logits_torch semantics.           */
/* ------------------------------------------------------------------------ */

struct mqa_ctx {
    int fmt, M, N, H, D;
    const uint8_t *q;
    const void *q_scale;
    const float *w;
    const uint8_t *k;
    const void *k_scale;
    const int32_t *ks, *ke;
    float *logits;
    int64_t ld;
};

static void mqa_row(void *vc, int r)
{
    struct mqa_ctx *c = (struct mqa_ctx *)vc;
    int H = c->H, D = c->D;
    double *qd = (double *)malloc(sizeof(double) * (size_t)H * D);
    double *qs = (double *)malloc(sizeof(double) * H);
    double *kd = (double *)malloc(sizeof(double) * D);
    decode_row_q(c->fmt, c->q, c->q_scale, r, H, D, qd, qs);
    int ks = clampi(c->ks[r], 0, c->N);
    int ke = clampi(c->ke[r], 0, c->N);
    float *out = c->logits + (size_t)r * c->ld;
    for (int t = 0; t < c->N; ++t) {
        if (t < ks || t >= ke) {
            out[t] = -INFINITY;
            continue;
        }
        double ksc;
        if (c->fmt == ORC_FMT_FP8) {
            decode_vec(c->fmt, c->k + (size_t)t * D, NULL, D, kd);
            ksc = (double)((const float *)c->k_scale)[t];
        } else {
            const uint8_t *sc = (const uint8_t *)c->k_scale + (size_t)t * (D / 32);
            decode_vec(c->fmt, c->k + (size_t)t * (D / 2), sc, D, kd);
            ksc = 1.0;
        }
        out[t] = score_one(qd, qs, c->w + (size_t)r * H, kd, ksc, H, D);
    }
    free(qd);
    free(qs);
    free(kd);
}

/* logits[M, ld] (columns [0, N) written): -inf outside [ks[r], ke[r]).
 * FP8: q [M,H,D] e4m3, q_scale NULL or fp32 [M,H], k [N,D] e4m3, k_scale fp32 [N].
 * MXFP4: q [M,H,D/2] packed e2m1, q_scale uint8 [M,H,D/32] e8m0,
 *        k [N,D/2] packed e2m1, k_scale uint8 [N,D/32] e8m0. */
int orc_mqa_logits(int fmt, const uint8_t *q, const void *q_scale, const float *w,
                   const uint8_t *k, const void *k_scale, const int32_t *ks,
                   const int32_t *ke, int M, int N, int H, int D, float *logits,
                   int64_t ld, int nthreads)
{
    if ((fmt == ORC_FMT_MXFP4 && D % 32 != 0) || D <= 0 || M < 0 || N < 0 || H <= 0)
        return 1;
    struct mqa_ctx c = {fmt, M, N, H, D, q, q_scale, w, k, k_scale, ks, ke, logits, ld};
    parallel_rows(mqa_row, &c, M, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Paged logits.                                                            */
/* ------------------------------------------------------------------------ */

/* Row r of a batch with next_n query tokens per sequence belongs to sequence
 * b = r / next_n and is its j = r % next_n-th token.  When context_lens holds
 * one length per sequence (ctx_per_row == 0), token j of an n-token step sees
 * keys [0, L - next_n + j + 1): the last token sees the whole context and each
 * earlier one stops at its own position.  With one length per row it is
 * simply context_lens[r]. */
int orc_row_end(const int32_t *context_lens, int ctx_per_row, int next_n, int r)
{
    if (ctx_per_row)
        return context_lens[r];
    int b = r / next_n, j = r % next_n;
    return context_lens[b] - next_n + j + 1;
}

struct paged_ctx {
    int fmt, H, D, P, next_n, ctx_per_row, num_pages, width;
    const uint8_t *q;
    const void *q_scale;
    const float *w;
    const uint8_t *pages;
    int64_t page_stride;
    const int32_t *bt;
    int64_t bt_stride;
    int max_blocks;
    const int32_t *ctx, *row_ks;
    float *logits;
    int64_t ld;
    int bad; /* keys whose block-table entry pointed outside the pool */
};

static void paged_row(void *vc, int r)
{
    struct paged_ctx *c = (struct paged_ctx *)vc;
    int H = c->H, D = c->D, P = c->P;
    int b = r / c->next_n;
    double *qd = (double *)malloc(sizeof(double) * (size_t)H * D);
    double *qs = (double *)malloc(sizeof(double) * H);
    double *kd = (double *)malloc(sizeof(double) * D);
    decode_row_q(c->fmt, c->q, c->q_scale, r, H, D, qd, qs);
    int ke = clampi(orc_row_end(c->ctx, c->ctx_per_row, c->next_n, r), 0, c->width);
    int ks = c->row_ks ? clampi(c->row_ks[r], 0, ke) : 0;
    float *out = c->logits + (size_t)r * c->ld;
    int bad = 0;
    for (int t = 0; t < ke; ++t) {
        if (t < ks) {
            out[t] = -INFINITY;
            continue;
        }
        int logical = t / P, slot = t % P;
        int page = logical < c->max_blocks ? c->bt[(size_t)b * c->bt_stride + logical] : -1;
        if (page < 0 || page >= c->num_pages) {
            out[t] = -INFINITY;
            ++bad;
            continue;
        }
        const uint8_t *base = c->pages + (size_t)page * c->page_stride;
        double ksc;
        if (c->fmt == ORC_FMT_FP8) {
            /* block-flat page: P*D e4m3 bytes, then P fp32 scales */
            decode_vec(c->fmt, base + (size_t)slot * D, NULL, D, kd);
            float f;
            memcpy(&f, base + (size_t)P * D + (size_t)slot * 4, 4);
            ksc = (double)f;
        } else {
            /* P*(D/2) packed e2m1 bytes, then P*(D/32) e8m0 bytes */
            const uint8_t *sc = base + (size_t)P * (D / 2) + (size_t)slot * (D / 32);
            decode_vec(c->fmt, base + (size_t)slot * (D / 2), sc, D, kd);
            ksc = 1.0;
        }
        out[t] = score_one(qd, qs, c->w + (size_t)r * H, kd, ksc, H, D);
    }
    if (bad)
        __atomic_add_fetch(&c->bad, bad, __ATOMIC_RELAXED);
    free(qd);
    free(qs);
    free(kd);
}

/* logits[B*next_n, ld]: columns [0, ke_r) of row r are written (-inf below
 * ks_r); columns [ke_r, width) are left untouched.  Returns the number of keys
 * whose page id was outside [0, num_pages) (written -inf), or -1 on bad args. */
int orc_paged_mqa_logits(int fmt, const uint8_t *q, const void *q_scale, const float *w,
                         const uint8_t *pages, int64_t page_stride, int num_pages,
                         const int32_t *bt, int64_t bt_stride, int max_blocks,
                         const int32_t *context_lens, int ctx_per_row,
                         const int32_t *row_ks, int B, int next_n, int H, int D,
                         int page_size, float *logits, int64_t ld, int width,
                         int nthreads)
{
    if ((fmt == ORC_FMT_MXFP4 && D % 32 != 0) || D <= 0 || B < 0 || next_n <= 0 || H <= 0 ||
        page_size <= 0)
        return -1;
    struct paged_ctx c = {fmt, H, D, page_size, next_n, ctx_per_row, num_pages, width,
                          q, q_scale, w, pages, page_stride, bt, bt_stride, max_blocks,
                          context_lens, row_ks, logits, ld, 0};
    parallel_rows(paged_row, &c, B * next_n, nthreads);
    return c.bad;
}

/* ------------------------------------------------------------------------ */
/* Candidate mask: _apply_candidate_mask_strided semantics.                 */
/* ------------------------------------------------------------------------ */

/* Row r keeps column t iff ks_r <= t < ke_r and t's candidate block,
 * (t - ks_r) / block_size, is listed in candidate row r / row_repeat; every
 * other column of [0, ke_r) becomes -inf and [ke_r, width) is not touched.
 * Block ids are counted from the row's start ks_r (ks_r = 0 when row_ks is
 * NULL); ids that are negative or name no block of the row are ignored. */
struct mask_ctx {
    float *logits;
    int64_t ld;
    int width;
    const int32_t *ks, *ke, *cand;
    int64_t cand_stride;
    int num_cand, block_size, row_repeat;
};

static void mask_row(void *vc, int r)
{
    struct mask_ctx *c = (struct mask_ctx *)vc;
    int ke = clampi(c->ke[r], 0, c->width);
    int ks = c->ks ? clampi(c->ks[r], 0, ke) : 0;
    const int32_t *cand = c->cand + (size_t)(r / c->row_repeat) * c->cand_stride;
    float *out = c->logits + (size_t)r * c->ld;
    for (int t = 0; t < ke; ++t) {
        int keep = 0;
        if (t >= ks) {
            int blk = (t - ks) / c->block_size;
            for (int i = 0; i < c->num_cand; ++i)
                if (cand[i] == blk)
                    keep = 1;
        }
        if (!keep)
            out[t] = -INFINITY;
    }
}

int orc_apply_candidate_mask(float *logits, int64_t ld, int rows, int width,
                             const int32_t *row_ks, const int32_t *row_ke,
                             const int32_t *cand, int64_t cand_stride, int num_cand,
                             int block_size, int row_repeat, int nthreads)
{
    if (block_size <= 0 || row_repeat <= 0 || num_cand < 0)
        return 1;
    struct mask_ctx c = {logits, ld, width, row_ks, row_ke, cand, cand_stride,
                         num_cand, block_size, row_repeat};
    parallel_rows(mask_row, &c, rows, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Block maxima of the candidate source: rocm_paged_mxfp4_indexer, module   */
/* description (the candidate source "takes its block maxima from the same  */
/* walk that writes its logits") and reserve_rocm_mxfp4_indexer_workspace   */
/* (block scores [rows, cdiv(logits_width, candidate_block_size)] fp32).    */
/* Block j of row r holds the keys [ks + j*bs, ks + (j+1)*bs) clipped to    */
/* [ks, ke), numbered from the row start like the candidate ids of          */
/* _apply_candidate_mask_strided; its score is the largest logit there,     */
/* -inf for an empty block.  NaN logits never win (fmax semantics).        */
/* ------------------------------------------------------------------------ */

struct bmax_ctx {
    const float *logits;
    int64_t ld;
    int width;
    const int32_t *row_ks, *row_ke;
    int block_size;
    float *out;
    int64_t ld_out;
    int nblocks;
};

static void bmax_row(void *vc, int r)
{
    struct bmax_ctx *c = (struct bmax_ctx *)vc;
    const int ke = clampi(c->row_ke[r], 0, c->width);
    const int ks = c->row_ks ? clampi(c->row_ks[r], 0, ke) : 0;
    const float *row = c->logits + (size_t)r * c->ld;
    float *o = c->out + (size_t)r * c->ld_out;
    for (int j = 0; j < c->nblocks; ++j) {
        float m = -INFINITY;
        const long long lo = (long long)ks + (long long)j * c->block_size;
        for (long long t = lo; t < lo + c->block_size && t < ke; ++t)
            if (row[t] > m)
                m = row[t];
        o[j] = m;
    }
}

/* out[r, 0:nblocks) = the block maxima of row r (see above). */
int orc_block_max(const float *logits, int64_t ld, int rows, int width,
                  const int32_t *row_ks, const int32_t *row_ke, int block_size,
                  float *out, int64_t ld_out, int nblocks, int nthreads)
{
    if (block_size <= 0 || nblocks < 0 || ld_out < nblocks)
        return 1;
    struct bmax_ctx c = {logits, ld, width, row_ks, row_ke, block_size, out, ld_out, nblocks};
    parallel_rows(bmax_row, &c, rows, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Per-row top-k: rocm_paged_mxfp4_indexer _topk semantics.                 */
/* ------------------------------------------------------------------------ */

struct kv_pair {
    float v;
    int32_t i;
};

/* Larger value first; equal values in ascending index order.  With the index
 * as the final key the order is total, so the sort is deterministic. */
static int cmp_desc(const void *a, const void *b)
{
    const struct kv_pair *x = (const struct kv_pair *)a, *y = (const struct kv_pair *)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->i > y->i) - (x->i < y->i);
}

struct topk_ctx {
    const float *logits;
    int64_t ld;
    int width;
    const int32_t *lengths;
    int k;
    int32_t *out;
    int64_t ld_out;
};

static void topk_row(void *vc, int r)
{
    struct topk_ctx *c = (struct topk_ctx *)vc;
    int len = clampi(c->lengths[r], 0, c->width);
    const float *row = c->logits + (size_t)r * c->ld;
    struct kv_pair *buf = (struct kv_pair *)malloc(sizeof(struct kv_pair) * (len > 0 ? len : 1));
    int n = 0;
    for (int t = 0; t < len; ++t)
        if (isfinite(row[t])) { /* -inf (masked) and NaN are never selected */
            buf[n].v = row[t];
            buf[n].i = t;
            ++n;
        }
    qsort(buf, n, sizeof(struct kv_pair), cmp_desc);
    int32_t *o = c->out + (size_t)r * c->ld_out;
    for (int j = 0; j < c->k; ++j)
        o[j] = j < n ? buf[j].i : -1;
    free(buf);
}

/* out[r, 0:k): indices of the k largest finite logits of row r within
 * [0, lengths[r]), largest first (ties: lower index first), -1 padded. */
int orc_topk(const float *logits, int64_t ld, int rows, int width,
             const int32_t *lengths, int k, int32_t *out, int64_t ld_out, int nthreads)
{
    if (k < 0)
        return 1;
    struct topk_ctx c = {logits, ld, width, lengths, k, out, ld_out};
    parallel_rows(topk_row, &c, rows, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-k positions -> ragged cache slots.                                   */
/* ------------------------------------------------------------------------ */

/* Row r belongs to sequence row_to_seq[r] (r / next_n when NULL).  Each entry
 * p >= 0 of its top-k row, in order, becomes slot block_table[b, p / P] * P
 * + p % P; -1 entries are dropped.  An entry whose logical page is past
 * max_blocks or whose page id is outside [0, num_pages) is dropped too and
 * counted.  indptr is the exclusive prefix sum of lens; slots holds the
 * concatenated rows.  Returns the dropped-invalid count. */
int orc_topk_to_ragged_slots(const int32_t *topk, int64_t ld, int rows, int k,
                             const int32_t *row_to_seq, int next_n,
                             const int32_t *bt, int64_t bt_stride, int max_blocks,
                             int page_size, int num_pages, int32_t *slots,
                             int32_t *indptr, int32_t *lens)
{
    int bad = 0;
    int64_t pos = 0;
    indptr[0] = 0;
    for (int r = 0; r < rows; ++r) {
        int b = row_to_seq ? row_to_seq[r] : r / next_n;
        int cnt = 0;
        for (int j = 0; j < k; ++j) {
            int p = topk[(size_t)r * ld + j];
            if (p < 0)
                continue;
            int logical = p / page_size;
            int page = logical < max_blocks ? bt[(size_t)b * bt_stride + logical] : -1;
            if (page < 0 || page >= num_pages) {
                ++bad;
                continue;
            }
            slots[pos++] = page * page_size + p % page_size;
            ++cnt;
        }
        lens[r] = cnt;
        indptr[r + 1] = (int32_t)pos;
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* K and Q producers.                                                       */
/*   - deepseek_v41 rocm.py, rocm_mxfp4_indexer_k_store: the key is RMS-     */
/*     normalised (weight, eps), rotated by RoPE at its position and         */
/*     written quantised into the cache slot kv_slot_mapping[t];             */
/*   - same page, rocm_mxfp4_indexer_q_quant: the query heads are rotated    */
/*     and quantised, and the weights are multiplied by the softmax scale    */
/*     times the head scale;                                                 */
/*   - RoPE: GPT-J pairs on the trailing rope_dim of a head with the cache   */
/*     row laid out cos | sin, the forward rotation of the inverse one of    */
/*     rocm_aiter_mla_sparse _inverse_rope_gptj_kernel;                      */
/*   - quantiser: rocm_aiter_mla_sparse _mxfp8_scale_bits (biased E8M0       */
/*     exponent that puts amax at the top of the element range) with top    */
/*     448 (e4m3) or 6 (e2m1), values multiplied by 2^(127 - bits) and      */
/*     rounded to the nearest element code, ties to the even code.          */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Forward GPT-J rotation of the pairs (x[n + 2i], x[n + 2i + 1]),
 * n = D - rope_dim: even' = a cos - b sin, odd' = b cos + a sin, with
 * cos = cs[i], sin = cs[rope_dim / 2 + i]. */
static void rope_gptj(double *x, int D, int rope_dim, const float *cs)
{
    const int n = D - rope_dim, half = rope_dim / 2;
    for (int i = 0; i < half; ++i) {
        const double a = x[n + 2 * i], b = x[n + 2 * i + 1];
        const double c = cs[i], s = cs[half + i];
        x[n + 2 * i] = a * c - b * s;
        x[n + 2 * i + 1] = b * c + a * s;
    }
}

/* Biased E8M0 exponent putting amax at the top `top` of the element range. */
static int scale_bits(double amax, double top)
{
    const double floor_amax = ldexp(1.0, -126);
    if (amax < floor_amax)
        amax = floor_amax;
    double bits = ceil(log2(amax / top)) + 127.0;
    if (bits < 0.0)
        bits = 0.0;
    if (bits > 254.0)
        bits = 254.0;
    return (int)bits;
}

/* Nearest code among the non-negative codes 0..ncodes-1 of a decoder,
 * ties to the even code; the sign bit `sign_bit` copies y's sign bit (so
 * -0 and negatives that round to zero give negative zero, as a cast does). */
static uint8_t encode_nearest(double y, double (*dec)(uint8_t), int ncodes, uint8_t sign_bit)
{
    const double a = fabs(y);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c < ncodes; ++c) {
        const double d = fabs(dec((uint8_t)c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)((signbit(y) ? sign_bit : 0) | best);
}

uint8_t orc_e4m3_encode(double y)
{
    return encode_nearest(y, orc_e4m3_to_double, 0x7F, 0x80); /* 0..0x7E finite */
}

uint8_t orc_e2m1_encode(double y)
{
    return encode_nearest(y, orc_e2m1_to_double, 8, 0x8);
}

int orc_scale_bits(double amax, double top)
{
    return scale_bits(amax, top);
}

/* Quantise one head vector y[D]: FP8 -> codes[D] and one exponent; MXFP4 ->
 * packed[D/2] and D/32 exponents.  Returns nothing; bits[] receives the
 * exponents. */
static void quantise_vec(const double *y, int D, int fmt, uint8_t *codes, int *bits)
{
    if (fmt == ORC_FMT_FP8) {
        double amax = 0.0;
        for (int d = 0; d < D; ++d)
            if (fabs(y[d]) > amax)
                amax = fabs(y[d]);
        bits[0] = scale_bits(amax, 448.0);
        const double inv = ldexp(1.0, 127 - bits[0]);
        for (int d = 0; d < D; ++d)
            codes[d] = orc_e4m3_encode(y[d] * inv);
        return;
    }
    for (int j = 0; j < D / 32; ++j) {
        double amax = 0.0;
        for (int d = 32 * j; d < 32 * j + 32; ++d)
            if (fabs(y[d]) > amax)
                amax = fabs(y[d]);
        bits[j] = scale_bits(amax, 6.0);
    }
    memset(codes, 0, (size_t)D / 2);
    for (int d = 0; d < D; ++d) {
        const uint8_t nib = orc_e2m1_encode(y[d] * ldexp(1.0, 127 - bits[d / 32]));
        codes[d / 2] |= (uint8_t)(d % 2 == 0 ? nib : nib << 4);
    }
}

/* K producer: token t (slot_mapping[t] >= 0) -> RMSNorm -> RoPE at
 * positions[t] -> quantise -> the block-flat page of cache slot
 * slot_mapping[t] (FP8: P*D codes then P fp32 scales 2^(bits-127); MXFP4:
 * P*D/2 packed bytes then P*D/32 e8m0 bytes).  pre (nullable, [T, D]) gets
 * the rotated values before scaling, bits_out (nullable, [T, D/32]) the
 * exponents (FP8: one, in column 0).  Returns the number of tokens skipped
 * for a slot outside the pool or a position outside the cos/sin table. */
int orc_k_norm_rope_store(const uint16_t *k_pre, int64_t ld_k, const int32_t *positions,
                          const float *cos_sin, int64_t ld_cs, int num_pos, int rope_dim,
                          const float *norm_w, double eps, uint8_t *pages, int64_t page_stride,
                          int num_pages, int page_size, const int64_t *slots, int T, int D,
                          int fmt, double *pre, int32_t *bits_out)
{
    int bad = 0;
    double *y = (double *)malloc(sizeof(double) * D);
    uint8_t *codes = (uint8_t *)malloc((size_t)D);
    int *bits = (int *)malloc(sizeof(int) * (D / 32 > 0 ? D / 32 : 1));
    const int rowb = fmt == ORC_FMT_FP8 ? D : D / 2;
    for (int t = 0; t < T; ++t) {
        const int64_t slot = slots[t];
        if (slot < 0)
            continue;
        const int64_t page = slot / page_size, off = slot % page_size;
        const int pos = positions[t];
        if (page >= num_pages || pos < 0 || pos >= num_pos) {
            ++bad;
            continue;
        }
        double ss = 0.0;
        for (int d = 0; d < D; ++d) {
            y[d] = bf16_to_double(k_pre[(size_t)t * ld_k + d]);
            ss += y[d] * y[d];
        }
        const double r = 1.0 / sqrt(ss / D + eps);
        for (int d = 0; d < D; ++d)
            y[d] = y[d] * r * (double)norm_w[d];
        rope_gptj(y, D, rope_dim, cos_sin + (size_t)pos * ld_cs);
        if (pre)
            memcpy(pre + (size_t)t * D, y, sizeof(double) * D);
        quantise_vec(y, D, fmt, codes, bits);
        uint8_t *pg = pages + page * page_stride;
        memcpy(pg + off * rowb, codes, (size_t)rowb);
        if (fmt == ORC_FMT_FP8) {
            const float sc = (float)ldexp(1.0, bits[0] - 127);
            memcpy(pg + (int64_t)page_size * rowb + off * 4, &sc, 4);
        } else {
            for (int j = 0; j < D / 32; ++j)
                pg[(int64_t)page_size * rowb + off * (D / 32) + j] = (uint8_t)bits[j];
        }
        if (bits_out)
            for (int j = 0; j < (fmt == ORC_FMT_FP8 ? 1 : D / 32); ++j)
                bits_out[(size_t)t * (D / 32) + j] = bits[j];
    }
    free(y);
    free(codes);
    free(bits);
    return bad;
}

/* Q producer: head (t, h) of q [T, H, D] -> RoPE at positions[t] ->
 * quantise.  FP8: codes [T, H, D], weights_out = w_in * w_scale *
 * 2^(bits-127) (the power-of-two query scale folded into the weight);
 * MXFP4: packed [T, H, D/2] and e8m0 bytes [T, H, D/32], weights_out =
 * w_in * w_scale.  pre / bits_out as for the K producer ([T*H, D],
 * [T*H, D/32]).  Returns the number of tokens with a position outside the
 * table (their heads are left untouched). */
int orc_q_rope_quant(const uint16_t *q, const int32_t *positions, const float *cos_sin,
                     int64_t ld_cs, int num_pos, int rope_dim, const float *w_in, double w_scale,
                     int T, int H, int D, int fmt, uint8_t *q_out, uint8_t *q_sf_out,
                     float *w_out, double *pre, int32_t *bits_out)
{
    int bad = 0;
    double *y = (double *)malloc(sizeof(double) * D);
    uint8_t *codes = (uint8_t *)malloc((size_t)D);
    int *bits = (int *)malloc(sizeof(int) * (D / 32 > 0 ? D / 32 : 1));
    const int rowb = fmt == ORC_FMT_FP8 ? D : D / 2;
    for (int t = 0; t < T; ++t) {
        const int pos = positions[t];
        if (pos < 0 || pos >= num_pos) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H; ++h) {
            const size_t th = (size_t)t * H + h;
            for (int d = 0; d < D; ++d)
                y[d] = bf16_to_double(q[th * D + d]);
            rope_gptj(y, D, rope_dim, cos_sin + (size_t)pos * ld_cs);
            if (pre)
                memcpy(pre + th * D, y, sizeof(double) * D);
            quantise_vec(y, D, fmt, codes, bits);
            memcpy(q_out + th * rowb, codes, (size_t)rowb);
            if (fmt == ORC_FMT_FP8) {
                w_out[th] = (float)((double)w_in[th] * w_scale * ldexp(1.0, bits[0] - 127));
            } else {
                for (int j = 0; j < D / 32; ++j)
                    q_sf_out[th * (D / 32) + j] = (uint8_t)bits[j];
                w_out[th] = (float)((double)w_in[th] * w_scale);
            }
            if (bits_out)
                for (int j = 0; j < (fmt == ORC_FMT_FP8 ? 1 : D / 32); ++j)
                    bits_out[th * (D / 32) + j] = bits[j];
        }
    }
    free(y);
    free(codes);
    free(bits);
    return bad;
}
