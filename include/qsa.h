/*
 * qsa.h -- C ABI of the QSA decode-attention library (libqsa.so).
 *
 * QSA decode attention: a handful of decode/verify queries (1-4 per step, the
 * MTP window) attend to a sparse selection of cells (one cell = one token's
 * K/V entry) drawn from INT8 K/V pools.  Cells are reached through a permuted
 * page table; each KV head is shared by q_per_kv query heads (12 on the
 * pages) at head_dim 256.  The selected list is split into chunks; each chunk
 * emits partials (running max m, sum of exponentials l, unnormalised P.V o)
 * and a merge combines them by log-sum-exp rescaling into the fp32 output.
 *
 * Defining passages: "Strata PR #2220, attn_chunk_q8_v3_kernel" (opening
 * description: decode attention over the QSA selection, INT8 pools, 12 query
 * heads, chunk partials and merged output, the two entry points
 * qsa_decode_attn_step / qsa_decode_attn_batch; kernel table: permuted page
 * table, 600 / 2,051 selected cells, 1-4 queries; prompt-shaped parity:
 * 2,048 queries against 32K INT8 cells), and "Strata issue #8, round 9:
 * performance candidate set on v0.2.9", R9-gpu-11 (page -1 masking; partial
 * accumulators, maxima and denominators; 0/1/2/3/63/64/65 selected cells).
 *
 * Conventions (all entry points):
 *   - Every pointer argument of a compute call is a DEVICE pointer, except the
 *     qsa_shape pointer, which is host memory read during the call only.
 *   - The caller owns every buffer.  The library allocates nothing, never
 *     synchronises, and is stateless and thread-safe; calls are asynchronous
 *     on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - Host-visible argument errors return a negative qsa_status and launch
 *     nothing.  A failed launch returns QSA_ERR_CUDA.
 *   - Device-side input errors never trap: an out-of-range list entry or page
 *     slot is treated as masked and raises a bit in the optional status word.
 *   - Kernels are launched with programmatic dependent launch: a call's first
 *     kernel may start while the previous kernel on the stream is still
 *     running, if that kernel allows it (a kernel that calls
 *     cudaTriggerProgrammaticLaunchCompletion, as this library's do).  Until
 *     it has waited for that kernel, a call only reads its own inputs
 *     (queries, pools, scales, page table, list, offsets) and writes nothing
 *     but status bits; so a kernel that triggers early must not write the
 *     next call's inputs after its trigger.  Copies, events and ordinary
 *     launches before a call are complete before it starts.  The next kernel
 *     on the stream may start early too: a kernel launched after a call with
 *     the programmatic-serialization attribute must call
 *     cudaGridDependencySynchronize() before it reads the call's outputs (the
 *     CUDA contract for such launches); ordinary launches, copies and events
 *     see the call complete.
 *
 * Dequantised values: k_hat = k_scale[cell] * K[cell][d] (same for V), a
 * symmetric per-cell fp32 scale with no zero point.  Scores
 * s = softmax_scale * (q . k_hat).  A page entry of -1 masks its cell: the
 * cell is left out of the softmax exactly as if it were not listed.  A row
 * with no valid cell outputs zeros.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qsa_status {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned buffer */
    QSA_ERR_UNSUPPORTED = -2, /* a shape outside what the kernels implement */
    QSA_ERR_WORKSPACE = -3,   /* workspace smaller than qsa_workspace_bytes() */
    QSA_ERR_CUDA = -4         /* a CUDA launch or runtime call failed */
} qsa_status;

typedef enum qsa_dtype {
    QSA_F32 = 0,  /* fp32 queries (decode) */
    QSA_BF16 = 1  /* bf16 queries (the prompt-shaped case) */
} qsa_dtype;

/* Which kernel family runs the chunk step.  AUTO picks by shape: the
 * cells-on-M tensor-core kernel for decode windows (q_per_kv * n_queries
 * <= 80 rows: up to six queries of 12 heads), the rows-on-M tensor-core
 * kernel for wider calls (prompt-shaped; chunk_cells >= 128).
 * SIMT forces the CUDA-core kernel (kept as an independent second path). */
typedef enum qsa_algo {
    QSA_ALGO_AUTO = 0,
    QSA_ALGO_SIMT = 1,
    QSA_ALGO_TCGEN05 = 2
} qsa_algo;

/* Bits of the optional device status word (OR-ed in by the kernels; the
 * library never clears it -- the caller zeroes it when it wants a fresh read). */
#define QSA_STATUS_BAD_POSITION 0x1u /* a position outside [0, page_table_len * P) */
#define QSA_STATUS_BAD_SLOT 0x2u     /* a page entry outside [0, pool_cells / P) and not -1 */
#define QSA_STATUS_BAD_OFFSETS 0x4u  /* batch offsets decreasing or a list above max_selected */
#define QSA_STATUS_TIMEOUT 0x8u      /* a bounded device-side wait ran out: outputs invalid */
#define QSA_STATUS_NOT_RESIDENT 0x10u /* qsa_kv_append: a position whose page entry is -1 */
#define QSA_STATUS_BAD_LIMITS 0x20u  /* causal limits that decrease along a window */
#define QSA_STATUS_LAUNCH 0x40u      /* a kernel's shared-memory window was misplaced: outputs invalid */
#define QSA_STATUS_BAD_EXTENT 0x80u  /* qsa_select_blocks: a live extent outside [0, max_blocks * R] (clamped) */

typedef struct qsa_shape {
    int32_t n_kv_heads;     /* G: KV heads per sequence (>= 1) */
    int32_t q_per_kv;       /* H: query heads per KV head (1..64; 12 on the pages) */
    int32_t head_dim;       /* D: must be 256 */
    int32_t n_queries;      /* T: queries per sequence (1-4 decode; up to 65536) */
    int32_t pool_cells;     /* N_pool: pool rows per (sequence, KV head) (>= 1),
                               a multiple of the page size P */
    int32_t page_table_len; /* page-table entries (pages) per sequence (>= 1); the
                               logical positions are 0 .. page_table_len * P - 1 */
    int32_t chunk_cells;    /* C: selected-list positions per chunk (>= 1) */
    float softmax_scale;    /* multiplies q . k_hat (1/16 on the pages' shapes) */
    int32_t q_dtype;        /* qsa_dtype */
    int32_t algo;           /* qsa_algo */
    int32_t page_cells;     /* P: cells per page; 0 means 1 (one entry per cell).
                               Position pos lies on page pos / P at offset pos % P;
                               a page entry e (a page of the pool, or -1: masked)
                               puts it in pool slot e * P + pos % P.  The pages
                               leave the page size open; P = 1 is the configs'
                               permuted per-cell table. */
} qsa_shape;

/*
 * Workspace size for a call with this shape, n_seq sequences and at most
 * max_selected selected cells per sequence.  Writes the byte count to
 * *bytes.  The workspace holds the chunk partials (and, for prompt-shaped
 * calls, converted operand images).  It needs no initialisation and no
 * clearing between calls; its base must be 256-byte aligned.
 * Errors: QSA_ERR_INVALID_ARG for a null pointer or a non-positive field;
 * QSA_ERR_UNSUPPORTED for head_dim != 256 or sizes beyond the limits above.
 */
qsa_status qsa_workspace_bytes(const qsa_shape *shape, int32_t n_seq, int32_t max_selected,
                               size_t *bytes);

/*
 * One sequence.
 *   q          [T][G*H][D]  fp32 or bf16 (per shape->q_dtype); query head j
 *              of KV head g is head index g*H + j.  16-byte aligned.
 *   k_pool     [G][pool_cells][D] int8 codes; v_pool the same.  16-byte aligned.
 *   k_scale    [G][pool_cells] fp32 per-cell scales; v_scale the same.
 *   page_table [page_table_len] int32: pool page of each page of logical
 *              positions (with P = 1: pool slot of each position), or -1
 *              (masked).
 *   sel        [n_sel] int32 logical positions (the QSA selection), in list
 *              order; chunk c covers list positions [c*C, min((c+1)*C, n_sel)).
 *   out        [T][G*H][D] fp32, fully written (zeros for rows with no valid
 *              cell).  Must not alias any input.
 *   workspace  >= qsa_workspace_bytes(shape, 1, n_sel) bytes.
 *   status     optional (may be NULL) device uint32 word; see QSA_STATUS_*.
 *   stream     cudaStream_t.
 * n_sel = 0 is valid and writes zeros.
 */
qsa_status qsa_decode_attn_step(const qsa_shape *shape, const void *q, const int8_t *k_pool,
                                const int8_t *v_pool, const float *k_scale,
                                const float *v_scale, const int32_t *page_table,
                                const int32_t *sel, int32_t n_sel, float *out, void *workspace,
                                size_t workspace_bytes, uint32_t *status, void *stream);

/*
 * n_seq independent sequences in one launch sequence.
 *   q          [n_seq][T][G*H][D]
 *   k_pool     [n_seq][G][pool_cells][D] (v_pool the same)
 *   k_scale    [n_seq][G][pool_cells]    (v_scale the same)
 *   page_table [n_seq][page_table_len]
 *   sel        concatenated lists; sequence b uses
 *              sel[sel_offsets[b] .. sel_offsets[b+1]).
 *   sel_offsets [n_seq+1] int32, device, non-decreasing, sel_offsets[0] = 0.
 *   max_selected  host-side upper bound on every list length; it sizes the
 *              grid and the workspace, so one captured CUDA graph serves any
 *              lists within the bound.  A longer list is clamped to
 *              max_selected and raises QSA_STATUS_BAD_OFFSETS.
 *   out        [n_seq][T][G*H][D] fp32.
 *   workspace  >= qsa_workspace_bytes(shape, n_seq, max_selected) bytes.
 */
qsa_status qsa_decode_attn_batch(const qsa_shape *shape, int32_t n_seq, const void *q,
                                 const int8_t *k_pool, const int8_t *v_pool,
                                 const float *k_scale, const float *v_scale,
                                 const int32_t *page_table, const int32_t *sel,
                                 const int32_t *sel_offsets, int32_t max_selected, float *out,
                                 void *workspace, size_t workspace_bytes, uint32_t *status,
                                 void *stream);

/*
 * qsa_decode_attn_batch with a causal limit per query of the window: query t
 * of sequence b sees only the selected cells whose logical position is below
 * q_limit[b][t]; a cell beyond it is left out of that query's softmax, as a
 * masked cell is.  The pages leave a causal order inside a verify window open;
 * this is the library's reading (the window's queries are consecutive tokens,
 * each seeing the positions before its own).
 *   q_limit    [n_seq][T] int32, device, non-decreasing in t within each
 *              sequence (a decreasing pair raises QSA_STATUS_BAD_LIMITS and
 *              leaves that sequence's outputs unspecified).
 * Other arguments and the workspace are those of qsa_decode_attn_batch.
 * Every kernel family takes limits (a causal prefill is a wide window whose
 * limits are its own positions plus one).
 */
qsa_status qsa_decode_attn_batch_limited(const qsa_shape *shape, int32_t n_seq, const void *q,
                                         const int8_t *k_pool, const int8_t *v_pool,
                                         const float *k_scale, const float *v_scale,
                                         const int32_t *page_table, const int32_t *sel,
                                         const int32_t *sel_offsets, int32_t max_selected,
                                         const int32_t *q_limit, float *out, void *workspace,
                                         size_t workspace_bytes, uint32_t *status, void *stream);

/*
 * Where the chunk partials of the last call with this (shape, n_seq,
 * max_selected) sit inside `workspace` (device pointers, read-only).
 *   m, l  [n_seq][G][n_chunks][T*H]      fp32; row r = t*H + j
 *   o     [n_seq][G][n_chunks][T*H][D]   fp32
 * with n_chunks = ceil(max_selected / chunk_cells).  For chunk c of sequence
 * b: m = max score (natural-log units, -inf when the chunk has no valid
 * cell), l = sum exp(s - m), o = sum exp(s - m) * v_hat.  Chunks at or past
 * ceil(n_b / C) are not written.  Any of m, l, o may be NULL.
 * A decode-window call (at most 80 rows per KV head, tensor-core path) with
 * more chunks than its CTAs (n_seq * G * n_chunks above the SM count, per
 * block of rows) lets a CTA accumulate up to eight consecutive chunks of a
 * (sequence, KV head) into one partial, the same m, l, o over those cells:
 * slot k then holds the pair's k-th such run, in chunk order, and the slots
 * past its last run are not written.
 */
qsa_status qsa_partials_view(const qsa_shape *shape, int32_t n_seq, int32_t max_selected,
                             const void *workspace, const float **m, const float **l,
                             const float **o, int32_t *n_chunks);

/*
 * qsa_decode_attn_step without a workspace, for callers that cannot allocate
 * device memory where they run this call (a serving path whose memory budget
 * is fixed after start-up, or a plugin inside an application that owns all
 * device memory).  The pages have no counterpart; this is an addition of
 * this library.
 *   Arguments are those of qsa_decode_attn_step minus workspace and
 *   workspace_bytes.  The chunk partials go to a fixed 8 MiB array that the
 *   library keeps in every GPU that loads it, until the process exits.
 *   A call whose qsa_workspace_bytes(shape, 1, n_sel) exceeds 8 MiB returns
 *   QSA_ERR_WORKSPACE and launches nothing (e.g. 48 query rows at chunk 128
 *   fit about 21,000 selected cells).
 *   Each call on a stream that is not being captured looks up the array's
 *   device address in the current context (no allocation); a call made
 *   during stream capture reuses the last address found on that device.  So
 *   make the first call on each device, and the first after a
 *   cudaDeviceReset or a change of the current context, outside capture (a
 *   captured first call returns QSA_ERR_CUDA).
 *   All calls share the array: calls whose kernels may overlap on the GPU
 *   (different streams) race and must be ordered by the caller.
 *   It allocates nothing and calls no allocating routine.
 */
qsa_status qsa_decode_attn_step_noalloc(const qsa_shape *shape, const void *q,
                                        const int8_t *k_pool, const int8_t *v_pool,
                                        const float *k_scale, const float *v_scale,
                                        const int32_t *page_table, const int32_t *sel,
                                        int32_t n_sel, float *out, uint32_t *status,
                                        void *stream);

/*
 * INT8 K/V append: quantise new K and V rows and write them into the pools
 * the attention calls read.  The step is the KV append that follows a QSA
 * layer's K/V projections ("Strata issue #8, round 9: performance candidate
 * set on v0.2.9", R9-gpu-8, implementation handoff); the format is the pools' of
 * "attn_chunk_q8_v3_kernel" (INT8 codes, one fp32 scale per cell).  The
 * pages print no quantiser; this library's reading, per (cell, KV head) and
 * separately for K and V: scale = max|x| / 127 (fp32, correctly rounded),
 * code = x / scale (fp32, correctly rounded) rounded to nearest, ties to
 * even; a row of zeros gets scale 0 and zero codes.
 *   shape      the attention calls' shape; n_kv_heads, head_dim (256),
 *              pool_cells, page_table_len and page_cells are read, the rest
 *              ignored.
 *   n_seq, n_new  sequences and new cells per sequence (either 0: no work).
 *   kv_dtype   QSA_F32 or QSA_BF16: the element type of k_new and v_new.
 *   k_new      [n_seq][n_new][G][D] finite values, 16-byte aligned; v_new
 *              the same.  Row i of sequence b is that sequence's new cell i.
 *   positions  [n_seq][n_new] int32: logical position of each new cell.
 *   page_table [n_seq][page_table_len] int32: pool page of each page of
 *              positions (pages of shape->page_cells cells).
 *   k_pool     [n_seq][G][pool_cells][D] int8, 16-byte aligned; written at
 *              the new cells' slots only; v_pool the same.
 *   k_scale    [n_seq][G][pool_cells] fp32; written at those slots; v_scale
 *              the same.
 *   status     optional device word: QSA_STATUS_BAD_POSITION (a position
 *              outside the page table), QSA_STATUS_NOT_RESIDENT (its page
 *              entry is -1), QSA_STATUS_BAD_SLOT (an entry outside the pool):
 *              such a cell is skipped and nothing is written for it.
 * Two new cells of one call that resolve to the same slot leave either row
 * there.  Asynchronous on `stream`, graph-capturable, allocates nothing.
 * Errors: QSA_ERR_INVALID_ARG (null or misaligned pointer, negative count,
 * bad kv_dtype, new rows or scales aliasing the pools); QSA_ERR_UNSUPPORTED
 * (head_dim != 256); QSA_ERR_CUDA (launch failed).
 */
qsa_status qsa_kv_append(const qsa_shape *shape, int32_t n_seq, int32_t n_new, int32_t kv_dtype,
                         const void *k_new, const void *v_new, const int32_t *positions,
                         const int32_t *page_table, int8_t *k_pool, int8_t *v_pool,
                         float *k_scale, float *v_scale, uint32_t *status, void *stream);

/*
 * QSA block selection: the scorer over pooled indexer keys and its top-k,
 * which produce the selected-cell list a qsa_decode_attn_batch call reads.
 * The step is the QSA selection scorer of "Strata issue #8, round 9:
 * performance candidate set on v0.2.9" (R9-gpu-9: qsa_block_scores_rows over
 * pooled keys, a dead tail, per-query indexer vectors and steps) and its
 * top-k (the long-context select and TOPK_SPLIT on the same page).  The pages
 * print no formula; this library's reading:
 *   - block j of a sequence covers positions [j*R, (j+1)*R) and has one
 *     pooled key of F = idx_heads * idx_dim values; it is live while
 *     j*R < n_live, and a candidate for query t if also j*R <= steps[t];
 *   - score s[t][j] = sum over f of q_idx[t][f] * pooled[j][f] (fp32
 *     accumulation), -inf for a block that is not a candidate;
 *   - query t keeps its top_k candidates by score, equal scores going to the
 *     lower block id (all candidates if there are fewer);
 *   - the sequence's list is the union of its queries' kept blocks, expanded
 *     to their live positions in ascending order.
 */
typedef struct qsa_select_shape {
    int32_t n_queries;   /* T: queries of the window (1..8) */
    int32_t idx_heads;   /* indexer heads */
    int32_t idx_dim;     /* values per indexer head; F = idx_heads * idx_dim is
                            a multiple of 8 and at most 1024 */
    int32_t block_cells; /* R: positions per block (>= 1) */
    int32_t max_blocks;  /* pooled keys per sequence (1..16384); capacity
                            max_blocks * R positions */
    int32_t top_k;       /* blocks kept per query (1..max_blocks) */
} qsa_select_shape;

/* Workspace of a qsa_select_blocks call on n_seq sequences (block bitmaps and
 * counts; 256-byte aligned base, no initialisation needed).  Errors as for
 * qsa_select_blocks' shape checks. */
qsa_status qsa_select_workspace_bytes(const qsa_select_shape *shape, int32_t n_seq, size_t *bytes);

/*
 * Score, keep and list.  All pointers device pointers (shape: host).
 *   q_idx       [n_seq][T][F] fp32, 16-byte aligned.
 *   pooled      [n_seq][max_blocks][F] bf16 bit patterns, 16-byte aligned;
 *               rows of dead blocks are not read.
 *   n_live      [n_seq] int32 live positions (a value outside
 *               [0, max_blocks * R] is clamped and raises QSA_STATUS_BAD_EXTENT).
 *   steps       [n_seq][T] int32 position of each query, or NULL (every live
 *               block is a candidate).
 *   scores      [n_seq][T][max_blocks] fp32, written (-inf off candidates).
 *   kept        [n_seq][T][top_k] int32, written: kept block ids ascending,
 *               then -1.
 *   sel         positions, written: sequence b's list at
 *               sel[sel_offsets[b] .. sel_offsets[b+1]); capacity needed
 *               n_seq * min(T * top_k, max_blocks) * R entries.
 *   sel_offsets [n_seq + 1] int32, written (CSR; sel_offsets[0] = 0): pass
 *               sel and sel_offsets, with max_selected =
 *               min(T * top_k, max_blocks) * R, to qsa_decode_attn_batch.
 *   workspace   >= qsa_select_workspace_bytes(shape, n_seq) bytes.
 * Four kernel launches on `stream`; allocates nothing.  Errors:
 * QSA_ERR_INVALID_ARG (null or misaligned pointer, non-positive field),
 * QSA_ERR_UNSUPPORTED (T > 8, F not a multiple of 8 or above 1024,
 * max_blocks above 16384, top_k above max_blocks), QSA_ERR_WORKSPACE,
 * QSA_ERR_CUDA.
 */
qsa_status qsa_select_blocks(const qsa_select_shape *shape, int32_t n_seq, const float *q_idx,
                             const uint16_t *pooled, const int32_t *n_live, const int32_t *steps,
                             float *scores, int32_t *kept, int32_t *sel, int32_t *sel_offsets,
                             void *workspace, size_t workspace_bytes, uint32_t *status, void *stream);

/*
 * Testing aid: the bound, in SM clock cycles, of every device-side wait of the
 * tensor-core kernels in calls launched after this one, process-wide (0
 * restores the default of 2^32 cycles, about two seconds).  A wait that runs
 * out sets QSA_STATUS_TIMEOUT, the kernel stops waiting, drains its own
 * tensor-core operations and copies (each with a bound of its own), frees its
 * tensor memory and returns; that call's outputs are invalid.  A bound of a
 * few cycles makes a correct call's waits run out, which is how the time-out
 * path is tested.  Not for production use: it affects calls from every
 * thread.
 */
void qsa_set_wait_limit(int64_t cycles);

/* Static description of a status code. */
const char *qsa_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
