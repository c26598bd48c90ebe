/*
 * sparsecos: exact bulk cosine similarity between two CSR batches of
 * high-dimensional sparse embeddings, on one NVIDIA GB300 (sm_103a).
 *
 *   S[q, i] = (Q_q . I_i) / (|Q_q|_2 |I_i|_2)
 *
 * for every query row q of Q and every item row i of I, written as a dense
 * row-major float32 matrix.  The operation is the one set out in the blog
 * post "Engineering practice for bulk similarity calculation over sparse
 * embeddings": section 2.3 (the full n_query x n_item float32 result, every
 * entry exact, not a top-K), section 3.1 (cosine; the sparse dot product
 * summed over the intersection of the two supports), section 5.2 (norms over
 * the stored nonzeros only, computed once and passed in), section 2.2 and
 * 4.4 (items streamed in chunks of 8,192 rows; normalise right after the
 * product).
 *
 * Conventions for every call:
 *  - Matrices are CSR: int64 indptr[n_rows + 1] with indptr[0] = 0 and
 *    indptr non-decreasing, int32 indices[nnz] strictly increasing within a
 *    row and in [0, dim), float32 values[nnz].  Explicit zero values are
 *    allowed and count as ordinary entries.
 *  - A row with no nonzeros (norm 0) has cosine 0 with every row.
 *  - Device pointers are device memory of the handle's device, owned by the
 *    caller, and must stay valid until the work queued on `stream` is done.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call that takes a stream only queues work on it and
 *    returns; a fault in a kernel shows at the next synchronisation or via
 *    ss_check_device.
 *  - No call throws; each returns an ss_status.  A call that returns an error
 *    before queueing work leaves the handle usable.  ss_last_error gives a
 *    message for the last error on a handle.
 *  - A handle is used by one host thread at a time and drives one GPU.
 */
#ifndef SPARSECOS_H
#define SPARSECOS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ss_status;

#define SS_OK 0
#define SS_ERR_INVALID_ARG 1  /* null pointer, bad size, mismatched shapes */
#define SS_ERR_UNSORTED 2     /* indices not strictly increasing in a row */
#define SS_ERR_OUT_OF_RANGE 3 /* an index outside [0, dim), or bad indptr */
#define SS_ERR_OOM 4          /* a device or pinned-host allocation failed */
#define SS_ERR_CUDA 5         /* a CUDA runtime call failed */
#define SS_ERR_DEVICE_CHECK 6 /* a kernel found an input it could not use */
#define SS_ERR_TIMEOUT 7      /* a host wait on the GPU ran out of time */
#define SS_ERR_LIMIT 8        /* a size beyond a documented maximum */

/* ss_create flags */
#define SS_VALIDATE 0x1 /* check CSR inputs on the device (synchronises) */
/* Scoring algorithm of the chunk indexes.
 *  - item tiles ("hybrid"): a few dense "hot" dimensions multiplied as a
 *    small dense product, the rest through per-tile inverted indexes in
 *    shared memory; float32 products summed in ascending dimension order,
 *    then scaled by inv_q * inv_i.  Best for short rows with a skewed
 *    (Zipf-like) dimension distribution.
 *  - posting lists: per query row, the chunk's posting list of each of its
 *    dimensions is walked and the products of the normalised values
 *    (q_k inv_q)(v_ik inv_i) are summed exactly in fixed point (resolution
 *    2^-38), then rounded to float32 once.  Best for long or evenly spread
 *    rows.  Needs inverse norms whose products bound the scores by 1 (those
 *    of ss_row_norms); larger normalised products end the call with
 *    SS_ERR_DEVICE_CHECK.
 * With no algorithm flag the handle chooses per item matrix, once (one
 * synchronisation per item matrix): the tensor path (SS_ALGO_TENSOR below)
 * when a row sample of the matrix has at least 64 frequent ("hot")
 * dimensions and leaves at most 0.25 expected shared dimensions per pair
 * outside them; otherwise posting lists when more than half of the first
 * build's item tiles found no room for their inverted index, else item
 * tiles.  Every algorithm gives the cosines within 2e-6 of the exact ones
 * and is bitwise deterministic.  Setting more than one flag is
 * SS_ERR_INVALID_ARG. */
#define SS_ALGO_POSTING_LISTS 0x2
#define SS_ALGO_TILES 0x8
/* Tensor-core path: the (at most 160) dimensions held by the largest share of
 * a row sample of the item matrix are multiplied on the tensor cores as a
 * dense product of the normalised values, each split into two fp16 parts
 * (hi = fp16(x), lo = fp16(x - hi)) so that hi*hi + hi*lo + lo*hi carries
 * about 22 bits, accumulated in float32; the other ("cold") dimensions'
 * products are summed exactly in fixed point (resolution 2^-28) and added
 * once.  The cosines are within 2e-6 of the exact ones and bitwise the same
 * for any chunking.  Best when the rows share a Zipf-like head of frequent
 * dimensions (BM25/TF-IDF text).  Needs inverse norms of the rows (those of
 * ss_row_norms): a normalised value above 1 + 2^-10 or a normalised row whose
 * squares sum above 1 + 2^-6 ends the call with SS_ERR_DEVICE_CHECK.
 * The query side is prepared once per query matrix, inverse-norm array and
 * item matrix: changing the contents of either array under the same
 * pointers needs ss_invalidate.  Exclusive with the two flags above. */
#define SS_ALGO_TENSOR 0x10
/* ss_bulk_cosine_host verifies every streamed chunk: its checksum (see
 * ss_tile_checksum) is taken on the device before the copy and on the host
 * after it, and must agree; the pass then always goes through the ring. */
#define SS_VERIFY_STREAM 0x4

/* Largest chunk the index builder accepts (item numbers in a chunk are
 * stored in 16 bits). */
#define SS_MAX_CHUNK_ROWS 65536

typedef struct ss_handle ss_handle;
typedef struct ss_index ss_index;

/* A CSR matrix.  For calls marked "device" the three arrays are device
 * memory; for ss_bulk_cosine_host they are host memory. */
typedef struct ss_csr {
  const int64_t *indptr;  /* [n_rows + 1] */
  const int32_t *indices; /* [nnz] */
  const float *values;    /* [nnz] */
  int64_t n_rows;
  int64_t nnz; /* = indptr[n_rows] */
  int64_t dim; /* number of dimensions d; indices lie in [0, d) */
} ss_csr;

/*
 * Creates a handle on `device` for matrices of dimension `dim` whose items
 * are streamed in chunks of `chunk_rows` rows (the post picks 8,192,
 * section 3.3).  Allocates the handle's device workspace (the chunk index
 * and its scratch).  chunk_rows must lie in [1, SS_MAX_CHUNK_ROWS].
 * Errors: SS_ERR_INVALID_ARG, SS_ERR_LIMIT, SS_ERR_OOM, SS_ERR_CUDA.
 */
ss_status ss_create(ss_handle **out, int device, int64_t dim, int32_t chunk_rows,
                    int32_t flags);

/*
 * Row norms (section 5.2, computed once, section 4.4): for every row r of m
 * (device CSR), inv_norms[r] = 1 / sqrt(sum_j values[j]^2) over the row's
 * stored values, or 0 when that sum is 0.  The squares are summed exactly
 * split into pairs of floats (about 48 significant bits), so the result is
 * within one unit in the last place of the correctly rounded value; rows
 * whose squares leave the float range are rescaled by a power of two.
 * inv_norms: device, float32[m->n_rows], written.
 * With SS_VALIDATE the CSR is checked first (SS_ERR_UNSORTED,
 * SS_ERR_OUT_OF_RANGE) and the call synchronises `stream`.
 */
ss_status ss_row_norms(ss_handle *h, const ss_csr *m, float *inv_norms, void *stream);

/*
 * Per-chunk inverted index (the chunk's CSR turned into lists by dimension):
 * indexes item rows [row_begin, row_end) of `items` (device CSR), with
 * 0 < row_end - row_begin <= chunk_rows.  The index is owned by the handle
 * and stays valid until the next build (ss_build_item_index or
 * ss_build_item_indexes) or ss_destroy on it;
 * `*out` receives a pointer to it.  Work on `stream` must not overlap a
 * score call still using the previous index (queue both on one stream).
 * Errors: SS_ERR_INVALID_ARG, SS_ERR_LIMIT, SS_ERR_OOM, SS_ERR_CUDA.
 */
ss_status ss_build_item_index(ss_handle *h, const ss_csr *items, int64_t row_begin,
                              int64_t row_end, ss_index **out, void *stream);

/*
 * Scores every query row against one indexed chunk and normalises in the
 * same kernel (section 4.4):
 *   out[q * ld_out + c] = dot(Q_q, I_{row_begin + c}) * inv_q[q] * inv_i[c]
 * for q < queries->n_rows and c < row_end - row_begin.
 * queries: device CSR; inv_q: device float32[n_q] from ss_row_norms;
 * inv_i: device float32 pointer to the chunk's first item norm (the item
 * norm array + row_begin); out: device float32, row-major with leading
 * dimension ld_out >= chunk width.  Item tiles: float32 products and sums;
 * posting lists: exact fixed-point sums of float32 products of the
 * normalised values (see SS_ALGO_POSTING_LISTS); tensor path: split-fp16
 * tensor-core product of the hot dimensions plus exact fixed-point sums of
 * the others (see SS_ALGO_TENSOR).  All within 2e-6 of the exact cosine.
 * Errors: SS_ERR_INVALID_ARG, SS_ERR_CUDA.
 */
ss_status ss_score_chunk(ss_handle *h, const ss_csr *queries, const float *inv_q,
                         const ss_index *idx, const float *inv_i, float *out, int64_t ld_out,
                         void *stream);

/*
 * Number of chunks one ss_build_item_indexes call can build: enough that the
 * builder's blocks (one per 256-item tile) cover the GPU's SMs, at most 8.
 * The same for both algorithms.  Fixed at ss_create.
 */
int32_t ss_build_batch(const ss_handle *h);

/*
 * Builds, in one launch, the indexes of the consecutive chunks that split
 * [row_begin, row_end) into pieces of chunk_rows items starting at row_begin
 * (the last may be shorter); at most ss_build_batch(h) chunks, else
 * SS_ERR_LIMIT.  out (host array of at least ss_build_batch(h) pointers)
 * receives one handle-owned index per chunk, in order, and *n_out their
 * number; each is scored with ss_score_chunk exactly as one from
 * ss_build_item_index, and all stay valid until the next build on this
 * handle or ss_destroy.  Results equal those of building the chunks one by
 * one.  Errors: SS_ERR_INVALID_ARG (bad range, null pointers), SS_ERR_LIMIT,
 * SS_ERR_CUDA.
 */
ss_status ss_build_item_indexes(ss_handle *h, const ss_csr *items, int64_t row_begin,
                                int64_t row_end, ss_index **out, int32_t *n_out, void *stream);

/*
 * The whole device-resident pass: splits the items into chunks of the
 * handle's chunk_rows (section 2.2, "streaming batch"), and for each chunk
 * builds the index and scores it into
 *   out[q * ld_out + i], i in [0, items->n_rows).
 * inv_q / inv_i: device norms from ss_row_norms.  out: device float32 with
 * ld_out >= items->n_rows.  Equivalent to calling ss_build_item_index and
 * ss_score_chunk per chunk in order on `stream`.  No rows: SS_OK, no work.
 * Errors: SS_ERR_INVALID_ARG (null or mismatched arguments, ld_out too
 * small), and those of ss_build_item_index and ss_score_chunk; device-side
 * checks surface at the next ss_check_device.
 */
ss_status ss_score_all(ss_handle *h, const ss_csr *queries, const float *inv_q,
                       const ss_csr *items, const float *inv_i, float *out, int64_t ld_out,
                       void *stream);

/*
 * Top-k epilogue (the post's downstream uses are ranking and threshold
 * filtering of the scores, section 2.3): instead of storing a chunk's
 * scores, keep for every query row q the k items of largest cosine seen so
 * far, larger score first and equal scores by smaller item number, in
 *   best_val[q * k + r], best_item[q * k + r], r < k
 * (device float32 and int64, row-major; -INFINITY and -1 where fewer than k
 * items have been seen).  The scores are the very values ss_score_chunk
 * would store (either algorithm); 1 <= k <= SS_TOPK_MAX and k * (ceil(chunk_rows / 256) + 1) <= 8192, else
 * SS_ERR_LIMIT.
 *
 * ss_topk_reset: starts a pass for n_q query rows (fills best_val with
 * -INFINITY and best_item with -1, and sizes the handle's candidate
 * workspace; may synchronise the device when that grows).
 * ss_score_chunk_topk: scores one chunk (an index from ss_build_item_index
 * or ss_build_item_indexes) and merges its best items into the running
 * result; chunks may come in any order, each once per pass.
 * ss_topk_all: reset, then every chunk of `items` (built chunk_rows at a
 * time, ss_build_batch chunks per build).
 * All are asynchronous on `stream`.  Errors: SS_ERR_INVALID_ARG (null
 * pointers, an index of another handle, no reset for these rows and k),
 * SS_ERR_LIMIT, SS_ERR_OOM, SS_ERR_CUDA.
 */
#define SS_TOPK_MAX 64
ss_status ss_topk_reset(ss_handle *h, int64_t n_q, int32_t k, float *best_val, int64_t *best_item,
                        void *stream);
ss_status ss_score_chunk_topk(ss_handle *h, const ss_csr *queries, const float *inv_q,
                              const ss_index *idx, const float *inv_i, int32_t k, float *best_val,
                              int64_t *best_item, void *stream);
ss_status ss_topk_all(ss_handle *h, const ss_csr *queries, const float *inv_q, const ss_csr *items,
                      const float *inv_i, int32_t k, float *best_val, int64_t *best_item,
                      void *stream);

/*
 * Receives one finished chunk of the result in host memory:
 *   tile[q * ld + c] = S[q, item_begin + c], q < n_q, c < item_end - item_begin.
 * The tile is only valid during the call.  A nonzero return stops the pass
 * (ss_bulk_cosine_host then returns SS_ERR_INVALID_ARG).
 */
typedef int (*ss_chunk_consumer)(void *user, int64_t chunk, int64_t item_begin,
                                 int64_t item_end, const float *tile, int64_t ld, int64_t n_q);

/*
 * End to end from host memory (sections 2.2 and 4.4): copies the host CSR
 * batches to the device, computes both norm vectors, then for each item
 * chunk builds the index, scores it, and delivers the chunk's result to the
 * host.  out_host (row-major, ld_out >= items->n_rows) may be NULL;
 * `consumer` may be NULL; not both.
 *  - out_host page-locked (cudaHostAlloc, or registered as mapped) and no
 *    consumer: the scoring kernel stores each chunk straight into out_host
 *    through the buffer's device address; nothing is staged.
 *  - otherwise: each chunk is scored into one of two device buffers and
 *    copied, on a second stream that overlaps the next chunk's kernels, into
 *    a ring of `ring_depth` (>= 2) page-locked host buffers; from there its
 *    rows are copied into out_host (if given) and the tile is handed to
 *    `consumer` (if given).
 * Blocks until the last chunk has been delivered.  Streams, device buffers
 * and ring buffers belong to the handle and are kept (grown when needed)
 * between calls; ss_destroy frees them.  timeout_ms bounds each host wait
 * on the GPU (0 = 60000 ms); SS_ERR_TIMEOUT if one runs out.
 *
 * Under a device limit (ss_set_device_limit) that the whole pass does not
 * fit, the items are copied in batches of rows (the next batch on a third
 * stream while the current one is scored, two batch buffers) and, where the
 * queries and their output tiles do not fit half the limit, the queries in
 * tiles of rows; each chunk of a batch is then scored against each query
 * tile, and the tiles reach out_host at their own rows.  Per batch the
 * norms, the choice of algorithm and the hot dimensions are taken from the
 * batch alone, so the values agree with the unlimited pass within the
 * stated accuracy, not bit for bit.  A consumer receives whole columns of
 * the result: with more than one query tile the call returns SS_ERR_LIMIT
 * before any work.  With SS_VERIFY_STREAM one checksum is logged per
 * delivered tile (chunk x query tile, in delivery order).  The ranges come
 * from ss_plan_host_pass.
 */
ss_status ss_bulk_cosine_host(ss_handle *h, const ss_csr *queries_host,
                              const ss_csr *items_host, float *out_host, int64_t ld_out,
                              ss_chunk_consumer consumer, void *user, int32_t ring_depth,
                              int32_t timeout_ms);

/*
 * Reduced-precision input values for ss_bulk_cosine_host (the post's
 * suggestion of 16-bit values to halve memory and transfers, section 5.3):
 * after ss_set_host_values(h, SS_VALUES_BF16 or SS_VALUES_F16) the `values`
 * arrays of the host CSRs given to ss_bulk_cosine_host hold 2-byte values
 * of that type (the pointer is read as const uint16_t *: bfloat16 or IEEE
 * binary16 bit patterns).  They cross to the device at 2 bytes a value and
 * are widened there to float32, exactly; from then on the pass is the
 * float32 one, so the scores are bit for bit those of the float32 pass on
 * the widened values when both passes split alike (no device limit; under
 * one the 2-byte staging copies can change the item batches, and each batch
 * takes its own hot dimensions: equal within 2e-6 then).  Against the cosines of the unrounded values the
 * input rounding adds at most 2 asin(u) (u = 2^-9 for bfloat16, 2^-11 for
 * binary16, round-to-nearest inputs).  The post allows 16-bit data where an
 * error below 1e-3 is acceptable (section 5.3): binary16 meets that bar
 * (at most 9.8e-4, measured 2.3e-4); bfloat16 is OUTSIDE it (measured up
 * to 1.8e-3 on the 1.2M-dimension workload) and is offered only for data
 * already stored as bfloat16, whose scores are then exact for the values as
 * stored.  Neither is ever a default.  Values must be finite.  The setting
 * stays with the handle; SS_VALUES_F32 (the default) restores float32.
 * Errors: SS_ERR_INVALID_ARG (null handle, unknown type).
 */
#define SS_VALUES_F32 0
#define SS_VALUES_BF16 1
#define SS_VALUES_F16 2
ss_status ss_set_host_values(ss_handle *h, int32_t value_type);

/*
 * Caps the device memory ss_bulk_cosine_host holds for its copies of the
 * inputs, their inverse norms and its output tiles at `bytes` (0 = no cap,
 * the default).  The chunk indexes and the scoring workspace are sized by a
 * chunk, not by the matrices, and are not counted.  Errors:
 * SS_ERR_INVALID_ARG (null handle, negative bytes).
 */
ss_status ss_set_device_limit(ss_handle *h, int64_t bytes);

/*
 * How ss_bulk_cosine_host splits a pass under a device limit (host only; no
 * device is touched).  q_indptr[n_q + 1] and i_indptr[n_i + 1] are the host
 * CSR row pointers; direct_output != 0 when the output is page-locked and
 * written in place (no output tiles on the device); value_type is the host
 * values' SS_VALUES_* type (16-bit values add a 2-byte staging copy per
 * nonzero to the device copy).  On return *n_q_tiles
 * query tiles and *n_i_batches item batches, with boundaries
 * q_bounds[0..*n_q_tiles] (0, ..., n_q) and i_bounds[0..*n_i_batches]
 * (0, ..., n_i) when those arrays are given (NULL: counts only).  Rules: no
 * limit, or a pass that fits it whole: one tile and one batch.  Otherwise
 * the queries stay whole if their copy (8 bytes per row pointer, 8 per
 * nonzero, 4 per row for the norms) and their two output tiles of
 * rows x min(chunk_rows, n_i) floats take at most half the limit; else
 * tiles whose copy takes at most a quarter of the limit and whose output
 * tiles at most another quarter.  What the query side leaves is halved into
 * two item batch slots; each batch is the longest run of rows whose copy
 * fits a slot, cut to a multiple of chunk_rows when it holds at least one
 * chunk.  Every tile and batch has fewer than 2^31 nonzeros.  Errors:
 * SS_ERR_INVALID_ARG (null pointers, negative sizes, chunk_rows < 1, an
 * unknown value type, a bounds array too short: counts are still written),
 * SS_ERR_LIMIT (one row does not fit its share).
 */
ss_status ss_plan_host_pass(const int64_t *q_indptr, int64_t n_q, const int64_t *i_indptr, int64_t n_i,
                            int32_t chunk_rows, int64_t device_limit, int32_t direct_output,
                            int32_t value_type, int64_t *q_bounds, int64_t q_cap, int64_t *n_q_tiles,
                            int64_t *i_bounds, int64_t i_cap, int64_t *n_i_batches);

/*
 * Checksums of a row-major float32 tile of n_rows x n_cols with leading
 * dimension ld (the integrity check of a streamed result):
 *   bits_sum  = sum of the values' 32-bit patterns read as unsigned integers,
 *               modulo 2^64 (exact and order-independent: two copies of a
 *               tile agree exactly when, as a rule, they are bit-identical);
 *   value_sum = sum of the values in double, for reporting (its last bits
 *               depend on the summation order).
 * ss_tile_checksum: tile, bits_sum and value_sum are device pointers; the
 * sums are ADDED to *bits_sum / *value_sum (zero them first; several tiles
 * may add up), asynchronously on `stream`.  ss_tile_checksum_host: host
 * pointers, results written.  Errors: SS_ERR_INVALID_ARG, SS_ERR_CUDA.
 */
ss_status ss_tile_checksum(ss_handle *h, const float *tile, int64_t n_rows, int64_t n_cols,
                           int64_t ld, uint64_t *bits_sum, double *value_sum, void *stream);
ss_status ss_tile_checksum_host(const float *tile, int64_t n_rows, int64_t n_cols, int64_t ld,
                                uint64_t *bits_sum, double *value_sum);

/*
 * Checksums of chunk `chunk` of the last ss_bulk_cosine_host pass run with
 * SS_VERIFY_STREAM (as found on the host copy, equal to the device's).
 * Errors: SS_ERR_INVALID_ARG (no such chunk, or no verified pass).
 */
ss_status ss_stream_checksum(const ss_handle *h, int64_t chunk, uint64_t *bits_sum,
                             double *value_sum);

/*
 * Checks a device CSR on the device (indptr[0] = 0, indptr non-decreasing
 * and ending at nnz, indices strictly increasing within rows and in
 * [0, dim)).  Synchronises `stream`.  Returns SS_OK, SS_ERR_UNSORTED or
 * SS_ERR_OUT_OF_RANGE.
 */
ss_status ss_validate_csr(ss_handle *h, const ss_csr *m, void *stream);

/*
 * Synchronises `stream` (and the streams of the handle's host pass, which
 * may still run work of a pass that returned early, e.g. on SS_ERR_TIMEOUT)
 * and reports whether a kernel of this handle flagged an input it could not
 * use (SS_ERR_DEVICE_CHECK, e.g. a chunk whose nnz exceeds the index
 * capacity), then clears the flag.
 */
ss_status ss_check_device(ss_handle *h, void *stream);

/*
 * Forgets what the handle derived from earlier inputs: the hot dimensions
 * chosen for an item matrix and the prepared query matrix.  The handle keys
 * both on the arrays' addresses and sizes, so call this after changing the
 * contents of a matrix in place; the next calls recompute them.  No GPU work.
 * Errors: SS_ERR_INVALID_ARG (null handle).
 */
ss_status ss_invalidate(ss_handle *h);

/*
 * Diagnostics for an index built by ss_build_item_index.  Synchronises
 * `stream` and writes stats[0..7]:
 *   [0] algorithm (0 = item tiles,                  [1] items in the chunk
 *       1 = posting lists, 2 = tensor path)
 *   [2] item tiles (item tiles)                     [3] hot dimensions H (posting
 *                                                       lists: those split off;
 *                                                       tensor: on the tensor cores)
 *   [4] entries in the heavy-item list              [5] widest ELL column
 *   [6] ELL entries stored, padding included        [7] item tiles without an
 *       (posting lists: entries in the chunk;           inverted-index image
 *       tensor: cold entries in the chunk)
 * Fields that do not apply to the algorithm are 0.  Errors:
 * SS_ERR_INVALID_ARG (null handle or stats, an index that is not one of the
 * handle's current ones), SS_ERR_CUDA.
 */
ss_status ss_index_stats(ss_handle *h, const ss_index *idx, int64_t *stats, void *stream);

/*
 * Reads a chunk index built as posting lists or for the tensor path back
 * into host memory, in one form for both: the chunk's CSR (item rows
 * [row_begin, row_end) of the item matrix) turned into lists by dimension
 * (a CSC of the chunk), with the frequent ("hot") dimensions that the index
 * holds dense instead of in lists given apart.  For tests and inspection;
 * synchronises `stream`.  Outputs (host memory; any may be NULL):
 *   *n_hot, hot[0 .. *n_hot): the dense dimensions, ascending
 *     (*n_hot <= SS_EXPORT_HOT_MAX; 0 when the index keeps every dimension
 *     in lists);
 *   hot_values[i * SS_EXPORT_HOT_MAX + j] = value of dimension hot[j] in
 *     chunk item i (0 where the item lacks it), i < row_end - row_begin;
 *     the rest of each row of SS_EXPORT_HOT_MAX is 0;
 *   col_ptr[0 .. dim]: the list of dimension k is entries
 *     [col_ptr[k], col_ptr[k + 1]) (col_ptr[0] = 0; hot dimensions have
 *     empty lists);
 *   item[e], value[e], e < *n_entries: chunk item (0-based) and stored value
 *     of entry e; inside a list the items ascend (the device keeps them in
 *     no particular order, which none of its sums depends on; they are
 *     sorted here).  item and value need capacity >= *n_entries.
 * Errors: SS_ERR_INVALID_ARG (not an index of this handle, an item-tile
 * index, negative capacity), SS_ERR_LIMIT (capacity too small; *n_entries
 * is still written), SS_ERR_DEVICE_CHECK (list offsets outside the index),
 * SS_ERR_CUDA.
 */
#define SS_EXPORT_HOT_MAX 160
ss_status ss_index_export(ss_handle *h, const ss_index *idx, int32_t *n_hot, int32_t *hot,
                          float *hot_values, int32_t *col_ptr, int32_t *item, float *value,
                          int64_t capacity, int64_t *n_entries, void *stream);

/*
 * Reads back the queries' lists that the tensor path's scoring calls walk,
 * into host memory; for tests and inspection; synchronises `stream`.  The
 * first call for a query matrix (with its inverse norms and the hot set)
 * sorts the queries' nonzeros outside the hot set by dimension; every
 * later call walks each item's nonzeros outside the hot set into the list
 * of its dimension (the other item nonzeros make no cold product):
 *   dims[0 .. n_dims - 1]: the dimensions some query row holds outside the
 *     hot set, ascending;
 *   col_ptr[0 .. n_dims]: list k (dimension dims[k]) is entries
 *     [col_ptr[k], col_ptr[k + 1]);
 *   query[e]: the query row, ascending inside a list (sorted here; the
 *     device keeps no order, which no sum depends on, and one set of lists
 *     per slice of query rows, merged here);
 *   value[e]: the query's value times its row's inverse norm (float32).
 * Any output may be NULL; dims and col_ptr need room for dim + 1 entries,
 * query and value capacity >= *n_entries.
 * Errors: SS_ERR_INVALID_ARG (no tensor-path scoring call made yet),
 * SS_ERR_LIMIT (capacity too small; *n_entries is still written),
 * SS_ERR_DEVICE_CHECK, SS_ERR_CUDA.
 */
ss_status ss_lists_export(ss_handle *h, int64_t *n_dims, int32_t *dims, int32_t *col_ptr, int32_t *query,
                          float *value, int64_t capacity, int64_t *n_entries, void *stream);

/* Size of the fixed scratch array behind ss_cosine_chunk_noalloc. */
#define SS_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Codes a kernel leaves in a device status word (the first problem found
 * wins; 0 = none).  ss_check_device reads the handle's own word and turns a
 * nonzero code into SS_ERR_DEVICE_CHECK; ss_cosine_chunk_noalloc hands its
 * word to the caller. */
#define SS_DEVICE_OK 0
#define SS_DEVICE_UNSORTED 1     /* indices not strictly increasing in a row */
#define SS_DEVICE_OUT_OF_RANGE 2 /* an index outside [0, dim) */
#define SS_DEVICE_CAPACITY 3     /* more list entries than the space given for them */
#define SS_DEVICE_STALL 4        /* a bounded wait inside a kernel ran out */
#define SS_DEVICE_RANGE 5        /* inverse norms that are not the rows' own */

/*
 * Scores one item chunk for callers that cannot allocate device memory.
 * Such callers exist: code running inside a host whose memory pool owns the
 * whole GPU (a serving runtime or framework allocator that forbids foreign
 * cudaMalloc calls), code called while a CUDA graph is being captured (an
 * allocation then fails or breaks the capture), and plug-ins given a fixed
 * memory budget up front.  The paper has no counterpart: this is a
 * packaging of the same computation.
 *
 *   out[q * ld_out + c] = cos(Q_q, I_{row_begin + c}),  c < row_end - row_begin
 *
 * for every query row, computed with the posting-list kernels (see
 * SS_ALGO_POSTING_LISTS for the arithmetic).  Needs no handle and calls no
 * cudaMalloc, cudaFree or allocating library routine: all scratch (both norm
 * vectors, the chunk's per-dimension counters and list offsets, the posting
 * lists) comes from one static device array of SS_NOALLOC_SCRATCH_BYTES that
 * every GPU loading this library holds until the process exits.  The caller
 * passes the inputs and the output, all in device memory of the current
 * device; `stream` as in the other calls.
 *   chunk_nnz: the number of nonzeros in item rows [row_begin, row_end)
 *   (indptr[row_end] - indptr[row_begin]), known to the caller; the lists
 *   are sized by it.
 *   device_status: device int32 or NULL.  The call sets it to SS_DEVICE_OK
 *   on `stream`, and its kernels then leave there the first problem they
 *   find: SS_DEVICE_CAPACITY when chunk_nnz is below the chunk's real count
 *   (the lists were cut short and the scores are wrong),
 *   SS_DEVICE_OUT_OF_RANGE for an index outside [0, dim).  Read it once
 *   `stream` has run the call's work.  With NULL such problems go unreported.
 * Returns SS_ERR_INVALID_ARG or SS_ERR_LIMIT without queueing work: the
 * latter when the scratch needed (about 8 * (dim + 1) + 14 * chunk_nnz +
 * 4 * (n_q + chunk rows) bytes) exceeds SS_NOALLOC_SCRATCH_BYTES or the
 * chunk exceeds SS_MAX_CHUNK_ROWS.  The first call on a device looks up the
 * array's device address (no allocation) and keeps it for the life of the
 * process: make that first call before any stream capture, use the device's
 * primary context (the runtime's default), and do not call it again after a
 * cudaDeviceReset.  Every call shares the one array and it keeps the last
 * call's contents (each call clears what must start at zero): calls that
 * overlap on the GPU, on different streams or host threads, race and corrupt
 * each other's results; order them on one stream.
 */
ss_status ss_cosine_chunk_noalloc(const ss_csr *queries, const ss_csr *items, int64_t row_begin,
                                  int64_t row_end, int64_t chunk_nnz, float *out, int64_t ld_out,
                                  int32_t *device_status, void *stream);

/* Number of kernels this handle has launched so far (every call that
 * queues kernels adds the number it queued).  Host-side count; no sync; 0
 * for a null handle. */
uint64_t ss_kernel_launches(const ss_handle *h);

/* Testing hook for failure handling: makes the nth device or page-locked
 * host allocation that the library makes from now on (counting every
 * handle and thread; nth >= 1) fail as if the memory were exhausted, once;
 * nth <= 0 disarms it.  The call that meets the failure returns
 * SS_ERR_OOM, after which the handle has waited for its device and freed
 * every buffer it allocates on demand: it stays usable and allocates them
 * again on its next call.  Returns how many allocations were still to go
 * before the previous arming fired (0: none was armed, or it has fired).
 * Host only; no synchronisation. */
int64_t ss_inject_alloc_failure(int64_t nth);

/* Timing of the scoring kernel itself (k_tc_score, k_score_tiles or
 * k_score_lists, whichever the index uses).  While on, every scoring call
 * records a CUDA event just before and just after its scoring kernel, on
 * the caller's stream; the other kernels of the call (operand preparation,
 * cold records, query preparation) fall outside the pair.  Turning it on or
 * off keeps the pairs recorded so far (so a caller can time a sample of its
 * calls); ss_scorer_time reads and forgets them.  No synchronisation.
 * Errors: SS_ERR_INVALID_ARG (null handle). */
ss_status ss_profile_scorer(ss_handle *h, int32_t on);

/* Sum of the recorded pairs' elapsed times in milliseconds and their count,
 * then forgets them.  Synchronises on the last recorded event.  Errors:
 * SS_ERR_INVALID_ARG (null pointers), SS_ERR_CUDA. */
ss_status ss_scorer_time(ss_handle *h, double *total_ms, int64_t *launches);

/* Frees the handle and its device workspace (synchronises the device).
 * Errors: SS_ERR_INVALID_ARG (null handle). */
ss_status ss_destroy(ss_handle *h);

/* Static text for a status code ("unknown status" for other values; never
 * NULL). */
const char *ss_status_string(ss_status s);

/* Message of the last error on the handle ("" if none); valid until the
 * next call on the handle. */
const char *ss_last_error(const ss_handle *h);

#ifdef __cplusplus
}
#endif

#endif /* SPARSECOS_H */
