// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "sparsecos.h"

// Device status word codes (first error wins; 0 = none).
enum : int32_t {
  DEV_OK = 0,
  DEV_UNSORTED = 1,
  DEV_OUT_OF_RANGE = 2,
  DEV_CAPACITY = 3,
  DEV_STALL = 4,  // a bounded loop ran out of iterations
  DEV_RANGE = 5,  // a normalised product above 1: inverse norms that are not the rows' own
};
static_assert(DEV_OK == SS_DEVICE_OK && DEV_UNSORTED == SS_DEVICE_UNSORTED &&
                  DEV_OUT_OF_RANGE == SS_DEVICE_OUT_OF_RANGE && DEV_CAPACITY == SS_DEVICE_CAPACITY &&
                  DEV_STALL == SS_DEVICE_STALL && DEV_RANGE == SS_DEVICE_RANGE,
              "device status codes are part of the C ABI");

// Scoring algorithms.
enum : int32_t {
  ALGO_HYBRID = 0,   // dense hot dimensions in registers + sparse cold lists in shared memory
  ALGO_POSTING = 1,  // one block per query row walking the chunk's posting lists
  ALGO_TENSOR = 2,   // up to 128 hot dimensions on the tensor cores + exact cold records
};

// How a handle picks the algorithm of its chunk indexes.
enum : int32_t {
  MODE_AUTO = 0,     // per item matrix, from the tile overflow of its first build
  MODE_TILES = 1,    // always ALGO_HYBRID
  MODE_POSTING = 2,  // always ALGO_POSTING
  MODE_TENSOR = 3,   // always ALGO_TENSOR
};
// Posting lists split off the hot dimensions (dense slab and dense product)
// when the item matrix has at least this many of them.
constexpr int kSplitMinHot = 8;

// The automatic choice takes posting lists when more than this share of the
// first build's item tiles have more cold entries than an image holds.
constexpr double kAutoOverflowShare = 0.5;

// Geometry of the hybrid scorer (see hybrid.cu).
namespace hyb {
constexpr int kTQ = 64;                    // query rows per tile
constexpr int kQGroup = 4;                 // query rows scored together by one warp
constexpr int kTI = 256;                   // items per tile (one thread per item)
constexpr int kThreads = 256;              // threads per block (8 warps)
constexpr int kHotMax = 32;                // dense ("hot") dimensions per item matrix
constexpr int kEllMaxW = 1024;             // cold entries per item kept in the ELL block
constexpr int kMetaInts = 16;              // per item tile: 8 warp lengths, heavy begin, count
constexpr int kBatchEntries = 4096;        // cold query entries per hashed batch
constexpr int kHashBits = 13;
constexpr int kHashSlots = 1 << kHashBits; // load factor <= 1/2
constexpr int kBitmapBits = 15;
constexpr int kBitmapWords = (1 << kBitmapBits) / 32;
constexpr int kHotSampleEntries = 8192;    // nonzeros sampled to choose the hot set
constexpr int kHotMinPercent = 14;         // a dimension is hot if >= 14% of sampled rows hold it

// Per item tile, the cold nonzeros as an inverted index (an "image" that the
// scoring block copies into shared memory as is): dimension -> segment of
// (item, value).  Tiles whose cold part does not fit keep the ELL format.
constexpr int kImgSlotsBits = 13;
constexpr int kImgSlots = 1 << kImgSlotsBits;      // {dim or -1, start | end << 16}
constexpr int kImgDCap = 6144;                     // distinct cold dims per tile (load <= 3/4)
constexpr int kImgECap = 9216;                     // cold nonzeros per tile
constexpr int kImgOffSlots = 16;                   // after the header {D, E, fits, 0}
constexpr int kImgBitsLog2 = 15;                   // membership bitmap of the tile's cold dims
constexpr int kImgOffBits = kImgOffSlots + kImgSlots * 8;       // u32 bits[2^15 / 32]
constexpr int kImgOffItem = kImgOffBits + (1 << kImgBitsLog2) / 8;  // u8 item[E]
constexpr int kImgOffVal = kImgOffItem + kImgECap;              // float value[E]
constexpr int kImgBytes = kImgOffVal + kImgECap * 4;
static_assert(kImgOffItem % 16 == 0 && kImgOffVal % 16 == 0 && kImgBytes % 16 == 0,
              "image sections must stay 16-byte aligned");
constexpr int kMetaFits = 10;              // meta slot: 1 if the tile has an image
constexpr int kMetaHeavyItems = 11;        // meta slot: heavy items of the tile (entries in heavy_tbl)
static_assert(kTQ % kQGroup == 0, "query tiles hold whole row groups");
}  // namespace hyb

// The per-chunk index.  ALGO_POSTING: one posting list of (item, value) per
// dimension, CSC-style.  ALGO_HYBRID: per tile of kTI items, the hot
// dimensions' posting lists stored dense (slab), every other nonzero in an
// item-major ELL block (items with many of them in a separate list).
struct ss_index {
  int32_t algo = ALGO_HYBRID;
  int64_t row_begin = 0;
  int64_t row_end = 0;
  int32_t n_items = 0;
  int64_t dim = 0;
  // ALGO_POSTING
  const int32_t *col_ptr = nullptr;    // [dim + 1], posting list k = [col_ptr[k], col_ptr[k+1]),
                                       // positions into the build's entry arrays
  const uint16_t *post_item = nullptr; // [capacity]: item within the chunk
  const float *post_val = nullptr;     // [capacity]
  int64_t capacity = 0;
  int32_t slab_ld = 0;                 // the hot slab's item stride (posting lists: chunk_rows)
  // ALGO_HYBRID
  int32_t n_tiles = 0;
  const int32_t *hot = nullptr;        // [1 + kHotMax]: H, then the H hot dims ascending
  const float *slab = nullptr;         // hybrid: [tile][kHotMax][kTI]; posting lists: [kHotMax][slab_ld];
                                       // value of hot dim h for item i (0 if absent)
  const int2 *ell = nullptr;           // [tile][kEllMaxW][kTI]: (dim, value bits), dims ascending, -1 pads
  const int32_t *meta = nullptr;       // [tile][kMetaInts]
  const int32_t *heavy_k = nullptr;    // heavy items' cold entries: dim
  const float *heavy_v = nullptr;      //   value
  const uint8_t *heavy_item = nullptr; //   item within its tile
  const int4 *heavy_tbl = nullptr;     // [tile][kTI]: heavy items {item, first entry - tile's heavy base, count, 0}
  const unsigned char *image = nullptr; // [tile][kImgBytes]
  const int32_t *counters = nullptr;   // [1] tiles without an image, [2..] their ids ([0] unused)
  // ALGO_TENSOR (also hot: the tensor hot set; slab: [item][tcp::kHotMax]
  // raw hot values, 0 if absent)
  const float *sq = nullptr;           // [n_items]: each item's raw sum of squares
  const int2 *icold = nullptr;         // the build's cold entries {dim, raw value bits}, rows in CSR order
  const int2 *icold_rng = nullptr;     // [n_items]: {first entry in icold, count}
};

// Tensor-core path (see tensor.cu).
namespace tcp {
constexpr int kHotMax = 160;   // hot dimensions multiplied on the tensor cores
constexpr int kM = 128;        // query rows per tile (MMA M)
constexpr int kN = 256;        // items per tile (MMA N)
constexpr int kColBlock = 32;  // items per cold-record bucket
// The automatic choice takes the tensor path when the estimated cold
// overlap (expected shared cold dimensions per pair) is at most this.
constexpr double kAutoMaxCold = 0.25;
constexpr int kAutoMinHot = 64;
}  // namespace tcp

// Most chunks one hybrid index build covers (one launch, one view per chunk).
constexpr int kMaxBuildBatch = 8;

// Largest k of the top-k epilogue, and the most entries (k running plus a
// chunk's candidates, at most k per item tile) one row's merge handles.
constexpr int kTopkMax = 64;
constexpr int kTopkEntries = 8192;

// Top-k epilogue: the running best k of every query row, and per row the
// candidates one chunk's tiles offer before they are merged in.
struct ss_topk {
  int32_t k = 0;           // 0: the scorers store full tiles instead
  const float *best_val = nullptr;  // [n_q][k], descending; -inf where fewer than k seen
  float *cand_val = nullptr;        // [n_q][cand_cap]
  int32_t *cand_item = nullptr;     // [n_q][cand_cap]: item within the chunk
  int32_t *cand_n = nullptr;        // [n_q]
  int32_t cand_cap = 0;             // tiles of the chunk * k
};

// Workspace of the host-buffer pass (ss_bulk_cosine_host), kept between
// calls and grown on demand: its streams and events, the device copies of the
// two CSR matrices and their inverse norms, two chunk output buffers, and the
// page-locked ring used when results cannot be written straight to the
// caller's memory.
struct ss_host_pass {
  // Device buffers: the query tile (indptr, indices, values, inverse norms),
  // two item batch slots (the same four each), two output tiles.
  // With 16-bit host values, their staging copies (query tile, item slots).
  enum { kQPtr, kQIdx, kQVal, kInvQ, kIPtr0, kIIdx0, kIVal0, kInvI0, kIPtr1, kIIdx1, kIVal1, kInvI1,
         kOut0, kOut1, kQHalf, kIHalf0, kIHalf1, kBuffers };
  static constexpr int kSlotRoles = 4;  // kIPtr1 - kIPtr0
  // comp: norms, builds, scoring; copy: results to the host ring; up: item
  // batches to the device (the next batch while the current one is scored).
  cudaStream_t comp = nullptr, copy = nullptr, up = nullptr;
  cudaEvent_t done[2] = {nullptr, nullptr}, out_free[2] = {nullptr, nullptr}, finished = nullptr;
  cudaEvent_t batch_ready[2] = {nullptr, nullptr}, batch_free[2] = {nullptr, nullptr};
  // Device bytes the pass may hold for its buffers above (0: no limit).
  int64_t device_limit = 0;
  // Type of the host CSRs' values (SS_VALUES_F32, _BF16, _F16).
  int32_t value_type = 0;
  std::vector<cudaEvent_t> copied;  // one per ring slot
  void *buf[kBuffers] = {};
  size_t cap[kBuffers] = {};
  std::vector<float *> slots;
  size_t slot_bytes = 0;
  // Stream verification: per ring slot, the device checksum {bits, value}
  // copied to page-locked host memory with the tile; per chunk of the last
  // pass, the checksums found on the host.
  void *dev_sums = nullptr;             // [ring][2] x 8 bytes, device
  void *host_sums = nullptr;            // [ring][2] x 8 bytes, page-locked
  int32_t sums_slots = 0;
  std::vector<uint64_t> log_bits;
  std::vector<double> log_values;
};
void free_host_pass(ss_host_pass &hp);

struct ss_handle {
  int device = 0;
  int64_t dim = 0;
  int32_t chunk_rows = 0;
  int32_t flags = 0;
  int32_t algo = ALGO_HYBRID;   // algorithm of the current item matrix's indexes
  int32_t mode = MODE_AUTO;
  int sm_count = 0;
  std::string last_error;
  uint64_t launches = 0;  // kernels queued by this handle
  // Timing of the scoring kernel (ss_profile_scorer): events recorded in
  // pairs around each scoring-kernel launch while on.
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_ev;
  size_t prof_used = 0;

  // Device workspace, owned by the handle.
  int32_t *d_status = nullptr;  // one status word
  // ALGO_POSTING (allocated when first needed)
  int32_t *col_cnt = nullptr;    // [build_batch][dim + 1]: histogram, then scatter cursors
  int32_t *col_ptr = nullptr;    // [build_batch][dim + 1]
  int32_t *scan_part = nullptr;  // [scan tiles + 1]
  int64_t scan_tiles = 0;
  uint16_t *post_item = nullptr; // [post_cap]
  float *post_val = nullptr;     // [post_cap]
  int2 *post_hat = nullptr;      // [post_cap]: {item, value * inv_i}, rewritten per scoring call
  int64_t post_cap = 0;
  int32_t *row_next = nullptr;   // [2]: the posting scorer's row counter and finished blocks
  int32_t *probe = nullptr;      // [2]: tiles probed, tiles above the image capacity
  float *slab_post = nullptr;    // [build_batch][kHotMax][chunk_rows]: hot values (split lists)
  // Dense hot values of the query matrix ([n_q][kHotMax]) for the posting
  // path's split, for the current hot set; and the matrix they were made for.
  float *qhot_dense = nullptr;
  int64_t qhot_dense_cap = 0;
  const void *qd_src[3] = {nullptr, nullptr, nullptr};
  int64_t qd_rows = -1, qd_nnz = -1;
  uint64_t qd_generation = ~0ull;
  // Top-k with split lists: the chunk's dense hot scores ([n_q][chunk_rows]).
  float *hot_scratch = nullptr;
  int64_t hot_scratch_cap = 0;
  // The automatic choice, made once per item matrix (same identity as hot_src).
  const void *auto_src[3] = {nullptr, nullptr, nullptr};
  int64_t auto_src_rows = -1, auto_src_nnz = -1;
  int32_t auto_algo = ALGO_HYBRID;
  // ALGO_HYBRID
  int32_t *hot = nullptr;        // [1 + kHotMax]
  float *slab = nullptr;         // [max tiles][kHotMax][kTI]
  int2 *ell = nullptr;           // [max tiles][kEllMaxW][kTI]
  int32_t *meta = nullptr;       // [max tiles][kMetaInts]
  int32_t *heavy_k = nullptr;    // [heavy_cap]
  float *heavy_v = nullptr;
  uint8_t *heavy_item = nullptr;
  int4 *heavy_tbl = nullptr;     // [max tiles][kTI]
  // counters: [0] heavy cursor, then per chunk k of a build, at 1 + k * (1 +
  // chunk_tiles): the count of its tiles without an image and their ids.
  int32_t *counters = nullptr;
  int64_t heavy_cap = 0;
  int32_t max_tiles = 0;        // build_batch * chunk_tiles
  int32_t chunk_tiles = 0;      // item tiles per full chunk
  int32_t build_batch = 1;      // chunks one build covers
  unsigned char *image = nullptr; // [max tiles][kImgBytes]
  // Queries prepared for the current hot set: hot values per query tile
  // ([tile][kHotMax][kTQ]); each row's cold nonzeros as {dim, value bits},
  // moved to the front of the row's own range; and each row's cold count.
  float *qhot = nullptr;
  int2 *qcold = nullptr;
  int32_t *qcold_n = nullptr;
  int64_t qhot_cap = 0, qcold_cap = 0, qcold_n_cap = 0;
  // The hot set is chosen once per item matrix: the matrix it was chosen for,
  // and a counter that changes whenever it is chosen again.
  const void *hot_src[3] = {nullptr, nullptr, nullptr};
  int64_t hot_src_rows = -1, hot_src_nnz = -1;
  uint64_t hot_generation = 0;
  // The query matrix (and hot generation) qhot / qcold were prepared for.
  const void *prep_src[3] = {nullptr, nullptr, nullptr};
  int64_t prep_rows = -1, prep_nnz = -1;
  uint64_t prep_generation = ~0ull;

  // ALGO_TENSOR: the tensor hot set ([1 + tcp::kHotMax]: H, dims ascending),
  // its selection table, and {estimated cold overlap per pair, H} on the
  // device and as read back once per item matrix.
  int32_t *tc_hot = nullptr;
  int32_t *tc_sel = nullptr;
  float *tc_stats = nullptr;
  double tc_est_cold = 0.0;
  int32_t tc_H = 0;
  const void *tc_hot_src[3] = {nullptr, nullptr, nullptr};
  int64_t tc_hot_rows = -1, tc_hot_nnz = -1;
  uint64_t tc_hot_generation = 0;
  // Query operand ([query tiles][kM x 2Hp] fp16) and cold entries ({dim,
  // normalised value bits} at the row's own CSR positions; counts per row),
  // for the query matrix, inverse norms and hot set they were made for.
  uint16_t *tc_A = nullptr;
  int64_t tc_A_cap = 0;
  int2 *tc_qcold = nullptr;
  int64_t tc_qcold_cap = 0;
  int32_t *tc_qcold_n = nullptr;
  int64_t tc_qcold_n_cap = 0;
  const void *tcq_src[4] = {nullptr, nullptr, nullptr, nullptr};
  int64_t tcq_rows = -1, tcq_nnz = -1;
  uint64_t tcq_generation = ~0ull;
  // The queries' lists by dimension (CSC of their cold entries), one set
  // per slice of tcq_slice_rows query rows: counters (then cursors) and
  // offsets [slices][dim + 1], the scan's tile sums, the entries {query
  // row, normalised value bits} [nnz of the queries].
  int64_t tcq_slice_rows = 1, tcq_slices = 0;
  int32_t *tc_qcnt = nullptr, *tc_qptr = nullptr, *tc_qpart = nullptr;
  int64_t tc_qcnt_cap = 0, tc_qptr_cap = 0, tc_qpart_cap = 0;
  int2 *tc_qlist = nullptr;
  int64_t tc_qlist_cap = 0;
  // Per chunk of a build: raw hot values [chunk_rows][kHotMax], sums of
  // squares and {first cold entry, count} per item [chunk_rows] (the cold
  // entries themselves go to post_hat).
  float *tc_slab = nullptr;
  float *tc_sq = nullptr;
  int2 *tc_icold_rng = nullptr;
  // Item operand of the chunk being scored ([item tiles][kN x 2Hp] fp16).
  uint16_t *tc_B = nullptr;
  int64_t tc_B_cap = 0;
  // Cold records of one scoring call: buckets of (32 query rows, 32 items)
  // and their counts (-1: did not fit).
  int2 *tc_rec = nullptr;
  int64_t tc_rec_cap = 0;
  int32_t *tc_rec_n = nullptr;
  int64_t tc_rec_n_cap = 0;

  // The last build's chunk indexes (views into the workspace above).
  ss_index views[kMaxBuildBatch];
  int32_t n_views = 0;
  ss_host_pass host;
  // Top-k candidate workspace, grown on demand.
  float *cand_val = nullptr;
  int32_t *cand_item = nullptr;
  int32_t *cand_n = nullptr;
  int64_t cand_elems = 0, cand_rows = 0;
};

// Every device and page-locked host allocation of the library goes through
// these two, so that a test can make the n-th one fail
// (ss_inject_alloc_failure); they return what cudaMalloc / cudaHostAlloc
// return.
cudaError_t dev_alloc(void **p, size_t bytes);
cudaError_t host_alloc(void **p, size_t bytes);
template <typename T>
cudaError_t dev_alloc(T **p, size_t bytes) {
  return dev_alloc(reinterpret_cast<void **>(p), bytes);
}
template <typename T>
cudaError_t host_alloc(T **p, size_t bytes) {
  return host_alloc(reinterpret_cast<void **>(p), bytes);
}

// After a failed allocation: waits for the device, frees every buffer the
// handle allocates on demand (they are then all absent, never half made) and
// forgets what was derived from earlier inputs, so the next call starts from
// a clean workspace.
void reset_after_oom(ss_handle *h);

// Forgets what was prepared from the current query matrix (its caches are
// keyed on the arrays' addresses, which a host pass reuses for new contents).
void invalidate_queries(ss_handle *h);

// Records the next timing event on s when the scoring kernel is being timed
// (called just before and just after each scoring-kernel launch).
void prof_mark(ss_handle *h, cudaStream_t s);

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device, once per kernel and device; callable from several threads.
cudaError_t ensure_dyn_smem(const void *kernel, size_t bytes);
template <typename K>
cudaError_t ensure_dyn_smem(K *kernel, size_t bytes) {
  return ensure_dyn_smem(reinterpret_cast<const void *>(kernel), bytes);
}

// Launchers (all asynchronous on `s`).
cudaError_t launch_row_norms(const ss_csr &m, float *inv_norms, int sm_count, cudaStream_t s);
cudaError_t launch_validate_csr(const ss_csr &m, int32_t *d_status, int sm_count, cudaStream_t s);
// Builds the posting lists of the chunks of h->chunk_rows items that split
// [row_begin, row_end) (at most h->build_batch of them), into h->views[0..n).
cudaError_t launch_build_index(ss_handle *h, const ss_csr &items, int64_t row_begin,
                               int64_t row_end, cudaStream_t s);
// Posting-list scorer: normalises the chunk's entries into h->post_hat, then
// scores (or offers top-k candidates); *queued gets the kernels queued.
cudaError_t launch_score_lists(ss_handle *h, const ss_csr &queries, const float *inv_q,
                               const ss_index &idx, const float *inv_i, float *out, int64_t ld_out,
                               cudaStream_t s, int *queued, const ss_topk *topk = nullptr);
// Hybrid path.  launch_hot_select returns the number of kernels it queued.
cudaError_t launch_hot_select(ss_handle *h, const ss_csr &items, cudaStream_t s, int *queued);
// Builds the chunks of h->chunk_rows items that split [row_begin, row_end)
// (at most h->build_batch of them) in one launch, into h->views[0..n).
cudaError_t launch_build_hybrid(ss_handle *h, const ss_csr &items, int64_t row_begin,
                                int64_t row_end, cudaStream_t s);
// Counts the item tiles of [row_begin, row_end) and those whose cold entries
// exceed an image's capacity (for the hot set in h->hot) into probe[0..1].
cudaError_t launch_auto_probe(ss_handle *h, const ss_csr &items, int64_t row_begin, int64_t row_end,
                              int32_t *probe, cudaStream_t s);
// Queues the query preparation (when needed), the fast tile scorer and the
// fallback scorer; *queued gets the number of kernels queued.
cudaError_t launch_score_hybrid(ss_handle *h, const ss_csr &queries, const float *inv_q,
                                const ss_index &idx, const float *inv_i, float *out,
                                int64_t ld_out, cudaStream_t s, int *queued,
                                const ss_topk *topk = nullptr);
// Top-k: fills best_val with -inf and best_item with -1; merges one chunk's
// candidates (items numbered from item_base) into the running best.
cudaError_t launch_topk_reset(int64_t n_q, int32_t k, float *best_val, int64_t *best_item,
                              int32_t *cand_n, int sm_count, cudaStream_t s);
cudaError_t launch_topk_merge(const ss_topk &t, int64_t n_q, int64_t item_base, float *best_val,
                              int64_t *best_item, int sm_count, cudaStream_t s);

// Checksums of a row-major float tile (see checksum.cu): the device version
// adds into *bits_sum / *value_sum (device), the host version writes them.
cudaError_t launch_tile_checksum(const float *tile, int64_t n_rows, int64_t n_cols, int64_t ld,
                                 uint64_t *bits_sum, double *value_sum, int sm_count,
                                 cudaStream_t s);
void tile_checksum_host(const float *tile, int64_t n_rows, int64_t n_cols, int64_t ld,
                        uint64_t *bits_sum, double *value_sum);

// Tensor-core path (tensor.cu).  The hot set is chosen once per item matrix
// (reads back its statistics: synchronises the stream then).
cudaError_t launch_tc_hot_select(ss_handle *h, const ss_csr &items, cudaStream_t s, int *queued);
cudaError_t launch_build_tc(ss_handle *h, const ss_csr &items, int64_t row_begin, int64_t row_end,
                            cudaStream_t s, int *queued);
cudaError_t launch_score_tc(ss_handle *h, const ss_csr &queries, const float *inv_q,
                            const ss_index &idx, const float *inv_i, float *out, int64_t ld_out,
                            cudaStream_t s, int *queued, const ss_topk *topk = nullptr);
// Exclusive scan of n counters (three kernels): col_ptr gets the scan, and
// count is reset to the same values (scatter cursors).
cudaError_t launch_count_scan(int32_t *count, int64_t n, int32_t *part, int32_t *col_ptr,
                              cudaStream_t s);

// Kernels queued by one launch_build_index call.
constexpr int kIndexKernels = 5;

// Number of scan tiles needed for n counters.
int64_t scan_tile_count(int64_t n);
