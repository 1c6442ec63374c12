/*
 * idx.h -- C ABI of the GB300 (sm_103a) sparse-attention lightning indexer.
 *
 * For every query row r the indexer scores each cached key token t:
 *
 *     logits[r, t] = sum_h w[r, h] * relu(k_scale[t] * q_scale[r, h] * (q[r, h, :] . k[t, :]))
 *
 * (vLLM API page "vllm.v1.attention.ops.rocm_aiter_mla_sparse", section
 * fp8_mqa_logits_torch), masks each row to [ks, ke) and optionally to
 * candidate blocks (same page, _apply_candidate_mask_strided), selects the
 * top-k token indices per row (page "vllm.v1.attention.ops.
 * rocm_paged_mxfp4_indexer", section _topk) and maps them to ragged cache
 * slots (page rocm_aiter_mla_sparse, build_prefill_topk_ragged_indices).
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller; the library
 *     never frees or keeps it.  Nothing on the compute path allocates device
 *     memory.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream), never
 *     synchronises the host, and derives its grid from the arguments alone, so
 *     a call can be recorded into a CUDA graph.
 *   - Host-side checks run before any launch and return IDX_ERR_INVALID_ARG
 *     (null pointer, negative size, bad stride) or IDX_ERR_UNSUPPORTED (a
 *     shape this build has no kernel for).  Nothing is launched then.
 *   - Faults found on the device (a block-table entry or candidate id outside
 *     its range) never trap: the affected keys are written -inf (logits) or
 *     dropped (slots) and a sticky bit is set in the device status word, read
 *     and cleared by idx_get_device_status().
 *   - Integers are int32 unless stated; row-major layouts; strides in elements
 *     unless the name ends in _bytes.
 *   - Kernels are launched with programmatic stream serialisation: one may
 *     start its set-up (barriers, tensor memory, shared-memory clears) while
 *     the kernel ahead of it on the stream finishes, and waits for that
 *     kernel to complete before it reads any argument array, so inputs that
 *     the previous kernel writes are safe.
 */
#ifndef IDX_H_
#define IDX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *idx_stream_t; /* same type as cudaStream_t */

typedef enum {
    IDX_OK = 0,
    IDX_ERR_INVALID_ARG = 1,
    IDX_ERR_UNSUPPORTED = 2,
    IDX_ERR_WORKSPACE = 3,
    IDX_ERR_CUDA = 4
} idx_status;

typedef enum {
    /* OCP e4m3 values, one fp32 scale per key. */
    IDX_KV_FP8_E4M3 = 0,
    /* OCP MX: packed e2m1 (element 2i = low nibble of byte i) with one e8m0
     * scale byte per 32 elements. */
    IDX_KV_MXFP4 = 1
} idx_kv_format;

/* Bits of the device status word. */
#define IDX_DEV_BAD_PAGE 1u      /* block-table entry outside [0, num_pages) */
#define IDX_DEV_BAD_CANDIDATE 2u /* reserved: candidate ids are range-checked and ignored */
#define IDX_DEV_TIMEOUT 4u       /* a bounded pipeline wait ran out; outputs undefined */
#define IDX_DEV_BAD_POSITION 8u  /* a producer's position outside its cos/sin table */

/* ------------------------------------------------------------------------
 * idx_mqa_logits -- non-paged logits for one key sequence.
 * Passage: rocm_aiter_mla_sparse, fp8_mqa_logits_torch (shapes, [ks, ke)
 * semantics) and rocm_fp8_mqa_logits.
 *
 *   q        FP8: e4m3 [M, H, D].  MXFP4: packed [M, H, D/2].
 *   q_scale  FP8: NULL or fp32 [M, H], applied inside the relu.
 *            MXFP4: e8m0 bytes [M, H, D/32] (one int32 per head at D = 128,
 *            byte i scaling elements [32i, 32i+32)).  Required.
 *   weights  fp32 [M, H].
 *   k        FP8: e4m3 [N, D].  MXFP4: packed [N, D/2].  16-byte aligned.
 *   k_scale  FP8: fp32 [N].  MXFP4: e8m0 bytes [N, D/32].
 *   row_ks, row_ke  [M]: key range [ks, ke) of each row; 0 <= ks, ke <= N.
 *   logits   fp32 [M, ld_logits], ld_logits >= N.  Columns [0, N) of every
 *            row are written: the score inside [ks, ke), -inf outside.
 *   ws, ws_bytes  unused (may be NULL / 0); kept for ABI stability.
 * Supported: D = 128, H in {32, 64, 128}.  Keys are scored in tiles of 128
 * on tcgen05 tensor cores with fp32 accumulation.
 * ---------------------------------------------------------------------- */
idx_status idx_mqa_logits(const void *q, const void *q_scale, const float *weights,
                          const void *k, const void *k_scale, const int32_t *row_ks,
                          const int32_t *row_ke, int M, int N, int H, int D,
                          idx_kv_format fmt, float *logits, int64_t ld_logits, void *ws,
                          size_t ws_bytes, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_paged_mqa_logits -- logits over a paged K cache for decode / MTP rows.
 * Passage: rocm_aiter_mla_sparse, rocm_fp8_paged_mqa_logits and
 * rocm_fp8_paged_mqa_logits_triton; MXFP4 inputs as in
 * rocm_paged_mxfp4_indexer, rocm_mxfp4_sparse_attn_indexer.
 *
 *   q         [B, next_n, H, D] e4m3 or [B, next_n, H, D/2] packed e2m1.
 *   q_scale   as for idx_mqa_logits, with M = B * next_n rows.
 *   weights   fp32 [B * next_n, H].
 *   kv_pages  the page pool, page p at kv_pages + p * page_stride_bytes
 *             (16-byte aligned, stride a multiple of 16).  Block-flat pages:
 *             FP8:   page_size * D e4m3 bytes (token-major), then page_size
 *                    fp32 scales;
 *             MXFP4: page_size * D/2 packed bytes, then page_size * D/32 e8m0
 *                    bytes (token-major).
 *   block_table [B, bt_stride] (>= ceil(max_model_len / page_size) columns
 *             used): logical page j of sequence b is physical page
 *             block_table[b * bt_stride + j].
 *   context_lens [B] (ctx_per_row = 0) or [B * next_n] (ctx_per_row = 1).
 *             Row j of sequence b ends at ke = context_lens[b] - next_n + j + 1
 *             in the first case, at context_lens[b * next_n + j] in the second.
 *   row_ks    NULL (all 0) or [B * next_n] row starts; keys below ks are -inf.
 *   candidate_blocks NULL, or [B * next_n, cand_stride] int32 block ids of
 *             cand_block keys counted from the row's ks: a fused candidate mask
 *             (see idx_apply_candidate_mask); num_cand ids per row are read,
 *             negative or out-of-range ids are ignored.
 *   logits    fp32 [B * next_n, ld_logits], ld_logits >= max_model_len.  Only
 *             columns [0, ke) of each row are written; [ke, max_model_len) is
 *             left untouched (consumers read each row up to its length).
 *   num_ctas  0 = one persistent CTA per resident slot: the CTAs the
 *             occupancy calculator places on an SM for the launched kernel and
 *             its shared memory, times the SMs; otherwise the grid size.
 *   ws, ws_bytes  optional device scratch, 16-byte aligned.  With a fused
 *             candidate mask and ws_bytes >= idx_paged_mqa_logits_workspace_size
 *             (B, next_n, max_model_len, num_cand), a first kernel writes a
 *             plan of the tiles and 64-key boxes that hold a candidate key of
 *             any row of a sequence, and the logits kernel loads and scores
 *             only those (every other key of [0, ke) is written -inf, as the
 *             mask requires): the same logits, fewer K bytes read.  Block-table
 *             entries of pages that are never loaded are then not checked.
 *             Calls sharing one ws must not overlap in time.
 * Supported: D = 128, page_size a multiple of 64, next_n * H <= 256.
 * ---------------------------------------------------------------------- */
idx_status idx_paged_mqa_logits(const void *q, const void *q_scale, const float *weights,
                                const uint8_t *kv_pages, int64_t page_stride_bytes,
                                int num_pages, const int32_t *block_table, int64_t bt_stride,
                                const int32_t *context_lens, int ctx_per_row,
                                const int32_t *row_ks, int B, int next_n, int H, int D,
                                int page_size, idx_kv_format fmt,
                                const int32_t *candidate_blocks, int64_t cand_stride,
                                int num_cand, int cand_block, float *logits,
                                int64_t ld_logits, int max_model_len, int num_ctas, void *ws,
                                size_t ws_bytes, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_paged_mqa_logits_block_max -- the candidate source: idx_paged_mqa_logits
 * without a candidate mask, which also writes the block maxima of its logits
 * from the same walk.
 * Passage: vllm.v1.attention.ops.rocm_paged_mxfp4_indexer, module description
 * (the candidate source "takes its block maxima from the same walk that writes
 * its logits"), reserve_rocm_mxfp4_indexer_workspace (block scores
 * [rows, cdiv(logits_width, candidate_block_size)] fp32) and
 * rocm_mxfp4_sparse_attn_indexer (candidate_write: the source's scores are
 * not masked to a pool).
 *
 *   Arguments as idx_paged_mqa_logits with no candidates and no scratch, plus
 *   block_max   fp32 [B * next_n, ld_block_max], ld_block_max >=
 *               nb = ceil(max_model_len / block_size), caller-owned.  Block j
 *               of row r covers the keys [ks + j * block_size,
 *               ks + (j + 1) * block_size) clipped to [ks, ke) (numbered
 *               from the row start, like candidate ids); block_max[r, j] is
 *               the largest logit there, -inf for an empty block.  Columns
 *               [0, nb) of every row are written (a first kernel fills them
 *               with -inf, the logits kernel raises them with atomics).
 *   block_size  keys per block, >= 32.
 *   Selecting a row's candidate blocks is then idx_topk over block_max with
 *   lengths ceil((ke - ks) / block_size).
 * Errors: IDX_ERR_INVALID_ARG for a null block_max, block_size <= 0 or
 *   ld_block_max < nb; IDX_ERR_UNSUPPORTED for block_size < 32 or next_n > 2;
 *   otherwise as idx_paged_mqa_logits.
 * ---------------------------------------------------------------------- */
idx_status idx_paged_mqa_logits_block_max(
    const void *q, const void *q_scale, const float *weights, const uint8_t *kv_pages,
    int64_t page_stride_bytes, int num_pages, const int32_t *block_table, int64_t bt_stride,
    const int32_t *context_lens, int ctx_per_row, const int32_t *row_ks, int B, int next_n, int H,
    int D, int page_size, idx_kv_format fmt, float *logits, int64_t ld_logits, int max_model_len,
    float *block_max, int64_t ld_block_max, int block_size, int num_ctas, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_paged_mqa_logits_topk -- the paged logits (with block maxima when
 * block_max is given) and the per-row top-k of them in one call, the logits
 * kernel counting the top-k's first radix digit as it writes the logits.
 * Passage: as idx_paged_mqa_logits_block_max and idx_topk; the fusion (a
 * logits -> top-k prefilter) is a design of this library with no counterpart
 * in the pages.
 *
 *   Arguments as idx_paged_mqa_logits_block_max (block_max NULL: none), plus
 *   lengths   [B * next_n] int32: each row's ke as the logits define it (the
 *             top-k's row lengths; other values break the fused counts).
 *   k, out_idx, ld_out  as idx_topk.
 *   ws, ws_bytes  the top-k's scratch (idx_topk_workspace_size(B * next_n,
 *             ld_logits, k), 16-byte aligned).
 *   With that scratch, ld_logits > 8192, next_n <= 2 and cooperative launch,
 *   the top-k's plan kernel runs first, the logits kernel adds every written
 *   logit's digit-1 bin to the top-k's row histogram (shared-memory
 *   histograms per warpgroup, flushed per row group) and its valid counts,
 *   and the top-k starts at its filter phase: the same logits and indices as
 *   the two calls, one pass over the logits fewer.  Otherwise it is
 *   idx_paged_mqa_logits_block_max (or idx_paged_mqa_logits) followed by
 *   idx_topk.
 * Errors: as those calls; nothing is launched when a host check fails.
 * ---------------------------------------------------------------------- */
idx_status idx_paged_mqa_logits_topk(
    const void *q, const void *q_scale, const float *weights, const uint8_t *kv_pages,
    int64_t page_stride_bytes, int num_pages, const int32_t *block_table, int64_t bt_stride,
    const int32_t *context_lens, int ctx_per_row, const int32_t *row_ks, int B, int next_n, int H,
    int D, int page_size, idx_kv_format fmt, float *logits, int64_t ld_logits, int max_model_len,
    float *block_max, int64_t ld_block_max, int block_size, const int32_t *lengths, int k,
    int32_t *out_idx, int64_t ld_out, int num_ctas, void *ws, size_t ws_bytes,
    idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_paged_mqa_logits_candidates -- idx_paged_mqa_logits for a consumer
 * that reads only the candidate blocks (idx_topk_candidates).
 * Passage: as idx_paged_mqa_logits; the candidate mask of rocm_aiter_mla_sparse,
 * _apply_candidate_mask_strided, applied by reading only candidate keys.
 *
 *   Arguments as idx_paged_mqa_logits; candidate_blocks (num_cand > 0) and
 *   ws_bytes >= idx_paged_mqa_logits_workspace_size(...) are required.
 *   Writes the logits of every key of the tiles that hold a candidate key
 *   (keys of those tiles outside every candidate block get -inf) and leaves
 *   every other column untouched.
 * Errors: IDX_ERR_INVALID_ARG without candidates, IDX_ERR_WORKSPACE when ws
 *   is missing or too small; otherwise as idx_paged_mqa_logits.
 * ---------------------------------------------------------------------- */
idx_status idx_paged_mqa_logits_candidates(
    const void *q, const void *q_scale, const float *weights, const uint8_t *kv_pages,
    int64_t page_stride_bytes, int num_pages, const int32_t *block_table, int64_t bt_stride,
    const int32_t *context_lens, int ctx_per_row, const int32_t *row_ks, int B, int next_n, int H,
    int D, int page_size, idx_kv_format fmt, const int32_t *candidate_blocks, int64_t cand_stride,
    int num_cand, int cand_block, float *logits, int64_t ld_logits, int max_model_len,
    int num_ctas, void *ws, size_t ws_bytes, idx_stream_t stream);

/* Bytes of ws the gather path of idx_paged_mqa_logits needs (0 without a
 * candidate mask: num_cand <= 0).  Pure host arithmetic. */
size_t idx_paged_mqa_logits_workspace_size(int B, int next_n, int max_model_len, int num_cand);

/* ------------------------------------------------------------------------
 * idx_apply_candidate_mask -- in-place candidate mask on existing logits.
 * Passage: rocm_aiter_mla_sparse, _apply_candidate_mask_strided.
 *
 * Row r keeps column t iff ks_r <= t < ke_r and the block (t - ks_r) /
 * block_size is one of the num_cand ids in candidate row r / row_repeat;
 * every other column of [0, ke_r) is set to -inf.  Columns [ke_r, width) are
 * not touched.  Only -inf is written; logits are never read.
 *   logits [rows, ld], width <= ld; row_ks NULL (0) or [rows]; row_ke [rows]
 *   (0 <= ke <= width); candidate_blocks [ceil(rows / row_repeat), cand_stride].
 * ---------------------------------------------------------------------- */
idx_status idx_apply_candidate_mask(float *logits, int64_t ld, int rows, int width,
                                    const int32_t *row_ks, const int32_t *row_ke,
                                    const int32_t *candidate_blocks, int64_t cand_stride,
                                    int num_cand, int block_size, int row_repeat,
                                    idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_topk -- per-row top-k token indices.
 * Passage: rocm_paged_mxfp4_indexer, _topk: the k largest logits of each
 * row over [0, lengths[row]), -1 where a row has fewer than k.
 *
 *   logits  fp32 [rows, ld]; lengths [rows] with 0 <= lengths[r] <= ld.
 *   out_idx int32 [rows, ld_out], ld_out >= k.  Row r receives the indices of
 *           its min(k, #finite) largest finite values in [0, lengths[r]), in
 *           ASCENDING index order, then -1 padding.  -inf and NaN are never
 *           selected.  Among equal values at the k-th place the lower indices
 *           win, so the selected set is unique.
 *   k >= 0 (k == 0 writes nothing).  ld <= INT32_MAX.
 *   The launch depends on ld alone (one launch unless noted):
 *           ld <= 8192: one CTA of 256 threads per row, the row's keys in
 *           registers.  ld <= 262144 and rows * ceil(ld / 32768) at most
 *           the number of SMs: one thread-block cluster of ceil(ld / 32768)
 *           CTAs per row, each CTA holding 32768 keys in shared memory and
 *           reading the others' histograms through distributed shared
 *           memory (when the device cannot hold such a cluster, the rules
 *           for longer rows apply).  Otherwise (more or longer rows): with
 *           ws, chunks of 8192 keys over the whole GPU in two launches (a
 *           plan kernel that clears the part of ws that must start at zero,
 *           then one cooperative launch whose phases meet at grid barriers;
 *           each wait is bounded, a timeout sets IDX_DEV_TIMEOUT in the
 *           device status and leaves the output undefined); without ws one
 *           CTA streams each row.  Every path gives the same indices.
 *   ws, ws_bytes  optional caller-owned device scratch, 16-byte aligned,
 *           used only by the chunked path (ws_bytes >=
 *           idx_topk_workspace_size(rows, ld, k)).  Calls that share one ws
 *           must not overlap in time (same stream, or ordered by events); ws
 *           holds nothing the caller needs after the call.
 * Errors: IDX_ERR_INVALID_ARG for negative sizes, ld_out < k or NULL
 *   pointers; IDX_ERR_CUDA when a launch fails.
 * ---------------------------------------------------------------------- */
idx_status idx_topk(const float *logits, int64_t ld, int rows, const int32_t *lengths, int k,
                    int32_t *out_idx, int64_t ld_out, void *ws, size_t ws_bytes,
                    idx_stream_t stream);

/* Bytes of ws that idx_topk needs for its chunked path with these sizes;
 * 0 when the chunked path does not apply (rows <= 0, ld <= 0, ld above
 * 8192 * 1024, or rows * chunks above INT32_MAX).  Pure host arithmetic:
 * no CUDA call, no device touched. */
size_t idx_topk_workspace_size(int rows, int64_t ld, int k);

/* ------------------------------------------------------------------------
 * idx_topk_noalloc -- idx_topk without caller scratch.
 * The pages have no counterpart of this call: it is a library convenience.
 * It exists for callers that cannot hand over device scratch or allocate it
 * at call time: a serving engine that reserves nearly all free device
 * memory for its KV cache at start-up and allows no allocation afterwards,
 * a latency-critical loop where cudaMalloc / cudaFree may synchronise the
 * device, or a plain C caller with no device allocator of its own.
 *
 *   Same arguments and results as idx_topk, and it succeeds wherever
 *   idx_topk succeeds.  Calls that idx_topk serves with one CTA or one
 *   cluster per row take those scratch-free paths.  The others take the
 *   chunked path when its scratch fits one fixed array of
 *   IDX_TOPK_NOALLOC_MAX_BYTES per device (part of the library's device
 *   image: the call allocates nothing; that is up to about 450 rows of
 *   262144 keys), and otherwise the scratch-free kernel that streams each row
 *   in one CTA (slower on many long rows, same indices).
 *   The first chunked call on a device looks up the array's address with
 *   the device current, and so does the first one after the device's primary
 *   context was replaced (cudaDeviceReset); make that call before any stream
 *   capture on the device.  Every chunked call clears the part of the array
 *   that must start at zero (its first kernel, on `stream`) before the
 *   others run, so nothing a previous call left there is read.
 *   Calls on one device share the array: two calls that overlap in time
 *   (different streams, not ordered by events) race and give wrong indices.
 * Errors: as idx_topk; IDX_ERR_CUDA also when the address lookup fails.
 * ---------------------------------------------------------------------- */
#define IDX_TOPK_NOALLOC_MAX_BYTES (32u << 20)

idx_status idx_topk_noalloc(const float *logits, int64_t ld, int rows, const int32_t *lengths,
                            int k, int32_t *out_idx, int64_t ld_out, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_topk_candidates -- per-row top-k over a row's candidate blocks only.
 * Passage: rocm_paged_mxfp4_indexer, _topk, after the candidate mask of
 * rocm_aiter_mla_sparse, _apply_candidate_mask_strided.
 *
 *   Same result as idx_apply_candidate_mask (with row_ke = lengths) followed
 *   by idx_topk, reading only the candidate keys: row r selects among the
 *   keys t of [ks_r, lengths[r]) whose block (t - ks_r) / block_size is one
 *   of the num_cand ids of candidate row r / row_repeat (negative, repeated
 *   and out-of-range ids are ignored).  Output as idx_topk: ascending token
 *   indices, -1 padding, ties at the k-th value to the lowest index.
 *   logits [rows, ld] (columns outside the candidate blocks are never read);
 *   row_ks NULL (0) or [rows]; candidate_blocks [ceil(rows / row_repeat),
 *   cand_stride].
 * Supported: num_cand <= 512 and num_cand * block_size <= 16384.
 * Errors: IDX_ERR_INVALID_ARG for bad sizes or NULL pointers,
 *   IDX_ERR_UNSUPPORTED beyond the supported sizes, IDX_ERR_CUDA on launch.
 * ---------------------------------------------------------------------- */
idx_status idx_topk_candidates(const float *logits, int64_t ld, int rows, const int32_t *lengths,
                               const int32_t *row_ks, const int32_t *candidate_blocks,
                               int64_t cand_stride, int num_cand, int block_size, int row_repeat,
                               int k, int32_t *out_idx, int64_t ld_out, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_topk_to_ragged_slots -- top-k positions to a ragged list of cache slots.
 * Passage: rocm_aiter_mla_sparse, build_prefill_topk_ragged_indices; the
 * slot of position p is block_table[b, p / page_size] * page_size +
 * p % page_size (page rocm_aiter_mla, _expand_page_indices_kernel).
 *
 *   topk [rows, ld] int32 positions (-1 = none).  Row r belongs to sequence
 *   row_to_seq[r] (row_to_seq NULL: r / next_n).  Entries are kept in order;
 *   -1 entries are dropped, and so is an entry whose logical page is
 *   >= max_blocks or whose page id is outside [0, num_pages) (status bit
 *   IDX_DEV_BAD_PAGE is then set).
 *   slots  [rows * k] capacity; indptr [rows + 1] (exclusive prefix sum of
 *   lens, indptr[0] = 0); lens [rows].
 * ---------------------------------------------------------------------- */
idx_status idx_topk_to_ragged_slots(const int32_t *topk, int64_t ld, int rows, int k,
                                    const int32_t *row_to_seq, int next_n,
                                    const int32_t *block_table, int64_t bt_stride,
                                    int max_blocks, int page_size, int num_pages,
                                    int32_t *slots, int32_t *indptr, int32_t *lens,
                                    idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_topk_ragged_slots -- idx_topk, then idx_topk_to_ragged_slots of its
 * result, in one call.
 * Passage: as those two calls (rocm_paged_mxfp4_indexer, _topk;
 * rocm_aiter_mla_sparse, build_prefill_topk_ragged_indices).
 *
 *   Arguments as idx_topk (logits .. ws_bytes), then as
 *   idx_topk_to_ragged_slots for its topk = out_idx, ld = ld_out (row_to_seq
 *   .. lens).  Every output is exactly what the two calls write.  Where the
 *   top-k runs one thread-block cluster per row (8192 < ld <= 262144 and the
 *   clusters fit the GPU) and the slot map would take its count-and-write
 *   form (more than four (row, 1024-entry step) pairs or 32768 block-table
 *   words a CTA of a 16-CTA cluster), the top-k kernel also counts each
 *   row's valid slots as it writes the row, and the slot map runs only its
 *   ordered write.
 * Errors: as the two calls.
 * ---------------------------------------------------------------------- */
idx_status idx_topk_ragged_slots(const float *logits, int64_t ld, int rows,
                                 const int32_t *lengths, int k, int32_t *out_idx, int64_t ld_out,
                                 void *ws, size_t ws_bytes, const int32_t *row_to_seq, int next_n,
                                 const int32_t *block_table, int64_t bt_stride, int max_blocks,
                                 int page_size, int num_pages, int32_t *slots, int32_t *indptr,
                                 int32_t *lens, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_row_ends -- each paged row's end ke, derived on the device from the
 * context lengths by the rule idx_paged_mqa_logits applies to its rows.
 * Passage: rocm_aiter_mla_sparse, rocm_fp8_paged_mqa_logits_triton (one
 * length per row with ctx_per_row); rocm_aiter_mla, the DCP verify path (row
 * t of a qlen-token verify attends to [0, seq_len - qlen + t]).
 *
 *   context_lens [B] (ctx_per_row = 0) or [B * next_n] (ctx_per_row = 1).
 *   row_ends     int32 [B * next_n] out: row j of sequence b gets
 *                context_lens[b] - next_n + j + 1, or context_lens[b * next_n
 *                + j], clamped to [0, max_model_len].  These are the lengths
 *                idx_topk, idx_topk_candidates and idx_fill_logits_tail take
 *                for paged logits.
 * Errors: IDX_ERR_INVALID_ARG for negative sizes, next_n <= 0 or NULL
 *   pointers with rows > 0; IDX_ERR_CUDA when the launch fails.
 * ---------------------------------------------------------------------- */
idx_status idx_row_ends(const int32_t *context_lens, int ctx_per_row, int B, int next_n,
                        int max_model_len, int32_t *row_ends, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_fill_logits_tail -- -inf over [row_ends[r], width) of every row.
 * Passage: rocm_aiter_mla_sparse, rocm_fp8_paged_mqa_logits: the stage-1
 * path fills its whole logits workspace with -inf before scoring, so every
 * column past a row's end reads -inf.  idx_paged_mqa_logits leaves those
 * columns untouched (its consumers read each row up to its end); a caller
 * that hands the full-width rows to code expecting the filled workspace calls
 * this after it.
 *
 *   logits   fp32 [rows, ld], width <= ld; columns [row_ends[r], width) of
 *            row r are written -inf (row_ends clamped to [0, width]).
 *   row_ends int32 [rows] (e.g. from idx_row_ends).
 * Errors: IDX_ERR_INVALID_ARG for negative sizes, ld < width or NULL
 *   pointers with rows > 0; IDX_ERR_CUDA when the launch fails.
 * ---------------------------------------------------------------------- */
idx_status idx_fill_logits_tail(float *logits, int64_t ld, int rows, const int32_t *row_ends,
                                int width, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_k_norm_rope_store -- the K producer: normalise, rotate, quantise and
 * write each new key into its cache slot.
 * Passage: vllm/models/deepseek_v41/amd/rocm.py, rocm_mxfp4_indexer_k_store
 * (RMS norm with weight and eps, RoPE at the token's position, quantised
 * store into kv_slot_mapping[t]); RoPE as the forward of
 * rocm_aiter_mla_sparse _inverse_rope_gptj_kernel (GPT-J pairs on the
 * trailing rope_dim, cos/sin row = cos | sin); quantiser as
 * rocm_aiter_mla_sparse _mxfp8_scale_bits (E8M0 exponent putting the block's
 * amax at 448 for e4m3 / 6 for e2m1; values times 2^(127 - bits) rounded to
 * the nearest code, ties to even).
 *
 *   k_pre       bf16 bits [T, ld_k], ld_k >= D (multiple of 4), 8-byte
 *               aligned: the keys before the norm.
 *   positions   [T] int32, each in [0, num_positions).
 *   cos_sin     fp32 [num_positions, ld_cos_sin]: row p = cos(p * f_i) for
 *               i < rope_dim / 2, then sin(p * f_i); nullable when rope_dim = 0.
 *   rope_dim    even, 0 <= rope_dim <= D: the trailing rope_dim elements of
 *               the key are rotated in pairs (2i, 2i + 1).
 *   norm_weight fp32 [D] (16-byte aligned); eps >= 0:
 *               y = x / sqrt(mean(x^2) + eps) * norm_weight.
 *   kv_pages, page_stride_bytes, num_pages, page_size  the cache of
 *               idx_paged_mqa_logits (same block-flat layout).  FP8: codes
 *               of y * 2^(127 - bits) with one exponent per token, its scale
 *               2^(bits - 127) stored as the token's fp32 scale; MXFP4: one
 *               e8m0 exponent per 32 elements.
 *   slot_mapping [T] int64: cache slot page * page_size + offset; -1 skips
 *               the token.
 * Supported: D = 128.  A slot outside the pool sets IDX_DEV_BAD_PAGE, a
 * position outside the table IDX_DEV_BAD_POSITION; those tokens are skipped.
 * ---------------------------------------------------------------------- */
idx_status idx_k_norm_rope_store(const uint16_t *k_pre, int64_t ld_k, const int32_t *positions,
                                 const float *cos_sin, int64_t ld_cos_sin, int num_positions,
                                 int rope_dim, const float *norm_weight, float eps, int T, int D,
                                 idx_kv_format fmt, uint8_t *kv_pages, int64_t page_stride_bytes,
                                 int num_pages, int page_size, const int64_t *slot_mapping,
                                 idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_q_rope_quant -- the Q producer: rotate and quantise the query heads
 * and scale their weights, in the formats idx_paged_mqa_logits reads.
 * Passage: vllm/models/deepseek_v41/amd/rocm.py, rocm_mxfp4_indexer_q_quant
 * (packed [T, H, D/2] + one int32 of four e8m0 bytes per head, fp32 weights
 * times index_weights_softmax_scale * index_weights_head_scale); RoPE and
 * quantiser as idx_k_norm_rope_store.
 *
 *   q           bf16 bits [T, H, D] contiguous, 8-byte aligned.
 *   positions, cos_sin, ld_cos_sin, num_positions, rope_dim  as above.
 *   weights     fp32 [T, H]; weight_scale the product of the softmax and
 *               head scales.
 *   q_out       FP8: e4m3 [T, H, D]; MXFP4: packed e2m1 [T, H, D/2].
 *   q_scale_out MXFP4: [T, H] int32 (byte j = e8m0 exponent of elements
 *               [32 j, 32 j + 32)); unused (nullable) for FP8.
 *   weights_out fp32 [T, H]: weights * weight_scale, and for FP8 also times
 *               the head's power-of-two scale 2^(bits - 127) (relu(s x) =
 *               s relu(x) for s > 0, so the logits need no q_scale).
 * Supported: D = 128.  Tokens with a position outside the table set
 * IDX_DEV_BAD_POSITION and are left unwritten.
 * ---------------------------------------------------------------------- */
idx_status idx_q_rope_quant(const uint16_t *q, const int32_t *positions, const float *cos_sin,
                            int64_t ld_cos_sin, int num_positions, int rope_dim,
                            const float *weights, float weight_scale, int T, int H, int D,
                            idx_kv_format fmt, uint8_t *q_out, void *q_scale_out,
                            float *weights_out, idx_stream_t stream);

/* ------------------------------------------------------------------------
 * idx_get_device_status -- read and clear the sticky device status word of
 * the current device (IDX_DEV_* bits).  Synchronises `stream`; it is the
 * only call that does.  *out receives the bits.
 * ---------------------------------------------------------------------- */
idx_status idx_get_device_status(idx_stream_t stream, uint32_t *out);

/* ------------------------------------------------------------------------
 * idx_debug_wait_expiry -- diagnostic: make one of the library's bounded
 * device waits run out.  The pages have no counterpart; it exists so that
 * the timeout path can be tested without breaking a real kernel.
 *
 *   which     0: the mbarrier wait that every pipeline stage of the logits
 *             kernel uses, on a barrier that no thread arrives on;
 *             1: the grid barrier of the chunked top-k, in a launch of two
 *             CTAs of which only the first arrives.
 *   limit_ns  the wait's limit, 1 .. 10^10 ns (the kernels use 2 * 10^9).
 * The kernel returns after about limit_ns with IDX_DEV_TIMEOUT set in the
 * device status word (read it with idx_get_device_status); the context stays
 * usable for the next call.  Errors: IDX_ERR_INVALID_ARG for other values,
 * IDX_ERR_CUDA when the launch fails.
 * ---------------------------------------------------------------------- */
idx_status idx_debug_wait_expiry(int which, uint64_t limit_ns, idx_stream_t stream);

/* Library version string, e.g. "idx 0.1 sm_103a". */
const char *idx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H_ */
