// The C ABI: handle lifecycle, argument checks, the chunk loop and the
// host-buffer streaming pass.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "internal.cuh"

namespace {

ss_status fail(ss_handle *h, ss_status st, const char *fmt, ...) {
  if (h) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    h->last_error = buf;
  }
  return st;
}

ss_status cuda_fail(ss_handle *h, cudaError_t e, const char *what) {
  const ss_status st = (e == cudaErrorMemoryAllocation) ? SS_ERR_OOM : SS_ERR_CUDA;
  if (h && st == SS_ERR_OOM) reset_after_oom(h);
  return fail(h, st, "%s: %s", what, cudaGetErrorString(e));
}

// Allocations left before the injected failure (0: none armed).
std::atomic<int64_t> g_alloc_countdown{0};

// True when this allocation is the one ss_inject_alloc_failure armed.
bool injected_failure() {
  int64_t left = g_alloc_countdown.load();
  while (left > 0) {
    if (g_alloc_countdown.compare_exchange_weak(left, left - 1)) return left == 1;
  }
  return false;
}

#define SS_CUDA(h, call)                                  \
  do {                                                    \
    cudaError_t e_ = (call);                              \
    if (e_ != cudaSuccess) return cuda_fail((h), e_, #call); \
  } while (0)

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

ss_status check_csr_args(ss_handle *h, const ss_csr *m, const char *what) {
  if (!m) return fail(h, SS_ERR_INVALID_ARG, "%s: null matrix", what);
  if (m->n_rows < 0 || m->nnz < 0)
    return fail(h, SS_ERR_INVALID_ARG, "%s: negative size", what);
  if (!m->indptr) return fail(h, SS_ERR_INVALID_ARG, "%s: null indptr", what);
  if (m->nnz > 0 && (!m->indices || !m->values))
    return fail(h, SS_ERR_INVALID_ARG, "%s: null indices/values", what);
  if (m->dim != h->dim)
    return fail(h, SS_ERR_INVALID_ARG, "%s: dim %lld differs from the handle's %lld", what,
                (long long)m->dim, (long long)h->dim);
  if (m->nnz >= ((int64_t)1 << 31))
    return fail(h, SS_ERR_LIMIT, "%s: nnz %lld exceeds 2^31 - 1", what, (long long)m->nnz);
  return SS_OK;
}

ss_status set_device(ss_handle *h) {
  SS_CUDA(h, cudaSetDevice(h->device));
  return SS_OK;
}

ss_status read_status(ss_handle *h, cudaStream_t s, int32_t *code) {
  SS_CUDA(h, cudaStreamSynchronize(s));
  SS_CUDA(h, cudaMemcpy(code, h->d_status, sizeof(int32_t), cudaMemcpyDeviceToHost));
  if (*code != DEV_OK) SS_CUDA(h, cudaMemset(h->d_status, 0, sizeof(int32_t)));
  return SS_OK;
}

ss_status status_from_device(ss_handle *h, int32_t code, const char *what) {
  switch (code) {
    case DEV_OK:
      return SS_OK;
    case DEV_UNSORTED:
      return fail(h, SS_ERR_UNSORTED, "%s: indices not strictly increasing within a row", what);
    case DEV_OUT_OF_RANGE:
      return fail(h, SS_ERR_OUT_OF_RANGE, "%s: index outside [0, dim) or bad indptr", what);
    case DEV_CAPACITY:
      return fail(h, SS_ERR_DEVICE_CHECK, "%s: chunk nnz exceeds the index capacity", what);
    case DEV_STALL:
      return fail(h, SS_ERR_DEVICE_CHECK, "%s: a kernel loop ran out of its iteration bound", what);
    case DEV_RANGE:
      return fail(h, SS_ERR_DEVICE_CHECK,
                  "%s: a product of normalised values exceeded 1 (inverse norms not those of the rows)", what);
    default:
      return fail(h, SS_ERR_DEVICE_CHECK, "%s: device check code %d", what, code);
  }
}

ss_status validate(ss_handle *h, const ss_csr &m, cudaStream_t s, const char *what) {
  SS_CUDA(h, launch_validate_csr(m, h->d_status, h->sm_count, s));
  h->launches += 1;
  int32_t code = 0;
  ss_status st = read_status(h, s, &code);
  if (st != SS_OK) return st;
  return status_from_device(h, code, what);
}

// Posting-list workspace (column counters and pointers for a build batch,
// the scorer's row counter); allocated on first use.
ss_status ensure_posting_workspace(ss_handle *h) {
  if (h->col_ptr) return SS_OK;  // the four exist together or not at all (reset_after_oom)
  const size_t n = (size_t)h->build_batch * (size_t)(h->dim + 1);
  h->scan_tiles = scan_tile_count((int64_t)n);
  SS_CUDA(h, cudaDeviceSynchronize());
  SS_CUDA(h, dev_alloc(&h->col_cnt, sizeof(int32_t) * n));
  SS_CUDA(h, dev_alloc(&h->scan_part, sizeof(int32_t) * (size_t)(h->scan_tiles + 1)));
  SS_CUDA(h, dev_alloc(&h->slab_post, sizeof(float) * (size_t)h->build_batch * hyb::kHotMax *
                                           (size_t)h->chunk_rows));
  SS_CUDA(h, dev_alloc(&h->col_ptr, sizeof(int32_t) * n));
  return SS_OK;
}

// Grows the entry capacity of one build (posting lists, or the hybrid
// path's heavy-item list) to hold `need` entries; synchronises the device
// when it has to reallocate.
ss_status ensure_capacity(ss_handle *h, int32_t algo, int64_t need) {
  if (algo == ALGO_POSTING || algo == ALGO_TENSOR) {
    if (need <= h->post_cap) return SS_OK;
    const int64_t cap = std::max<int64_t>(need, h->post_cap + h->post_cap / 2);
    SS_CUDA(h, cudaDeviceSynchronize());
    cudaFree(h->post_item);
    cudaFree(h->post_val);
    cudaFree(h->post_hat);
    h->post_item = nullptr;
    h->post_val = nullptr;
    h->post_hat = nullptr;
    h->post_cap = 0;
    SS_CUDA(h, dev_alloc(&h->post_item, sizeof(uint16_t) * (size_t)cap));
    SS_CUDA(h, dev_alloc(&h->post_val, sizeof(float) * (size_t)cap));
    SS_CUDA(h, dev_alloc(&h->post_hat, sizeof(int2) * (size_t)cap));
    h->post_cap = cap;
    return SS_OK;
  }
  if (need <= h->heavy_cap) return SS_OK;
  const int64_t cap = std::max<int64_t>(need, h->heavy_cap + h->heavy_cap / 2);
  SS_CUDA(h, cudaDeviceSynchronize());
  cudaFree(h->heavy_k);
  cudaFree(h->heavy_v);
  cudaFree(h->heavy_item);
  h->heavy_k = nullptr;
  h->heavy_v = nullptr;
  h->heavy_item = nullptr;
  h->heavy_cap = 0;
  SS_CUDA(h, dev_alloc(&h->heavy_k, sizeof(int32_t) * (size_t)cap));
  SS_CUDA(h, dev_alloc(&h->heavy_v, sizeof(float) * (size_t)cap));
  SS_CUDA(h, dev_alloc(&h->heavy_item, (size_t)cap));
  h->heavy_cap = cap;
  return SS_OK;
}

// Frees every buffer a handle allocates on demand and leaves them absent
// (null, no capacity): each is then made again, whole, when next needed.
void free_lazy_buffers(ss_handle *h) {
  cudaFree(h->col_cnt);
  cudaFree(h->col_ptr);
  cudaFree(h->scan_part);
  cudaFree(h->slab_post);
  h->col_cnt = h->col_ptr = h->scan_part = nullptr;
  h->scan_tiles = 0;
  h->slab_post = nullptr;
  cudaFree(h->post_item);
  cudaFree(h->post_val);
  cudaFree(h->post_hat);
  h->post_item = nullptr;
  h->post_val = nullptr;
  h->post_hat = nullptr;
  h->post_cap = 0;
  cudaFree(h->heavy_k);
  cudaFree(h->heavy_v);
  cudaFree(h->heavy_item);
  h->heavy_k = nullptr;
  h->heavy_v = nullptr;
  h->heavy_item = nullptr;
  h->heavy_cap = 0;
  cudaFree(h->cand_val);
  cudaFree(h->cand_item);
  cudaFree(h->cand_n);
  h->cand_val = nullptr;
  h->cand_item = h->cand_n = nullptr;
  h->cand_elems = h->cand_rows = 0;
  cudaFree(h->qhot);
  cudaFree(h->qcold);
  cudaFree(h->qcold_n);
  h->qhot = nullptr;
  h->qcold = nullptr;
  h->qcold_n = nullptr;
  h->qhot_cap = h->qcold_cap = h->qcold_n_cap = 0;
  cudaFree(h->qhot_dense);
  cudaFree(h->hot_scratch);
  h->qhot_dense = h->hot_scratch = nullptr;
  h->qhot_dense_cap = h->hot_scratch_cap = 0;
  void *tc[] = {h->tc_hot, h->tc_sel, h->tc_stats, h->tc_A, h->tc_qcold, h->tc_qcold_n, h->tc_qcnt,
                h->tc_qptr, h->tc_qpart, h->tc_qlist, h->tc_slab, h->tc_sq, h->tc_icold_rng, h->tc_B,
                h->tc_rec, h->tc_rec_n};
  for (void *p : tc) cudaFree(p);
  h->tc_hot = h->tc_sel = h->tc_qcold_n = nullptr;
  h->tc_qcnt = h->tc_qptr = h->tc_qpart = h->tc_rec_n = nullptr;
  h->tc_stats = h->tc_slab = h->tc_sq = nullptr;
  h->tc_A = h->tc_B = nullptr;
  h->tc_qcold = h->tc_qlist = h->tc_rec = h->tc_icold_rng = nullptr;
  h->tc_A_cap = h->tc_qcold_cap = h->tc_qcold_n_cap = h->tc_B_cap = h->tc_rec_cap = h->tc_rec_n_cap = 0;
  h->tc_qcnt_cap = h->tc_qptr_cap = h->tc_qpart_cap = h->tc_qlist_cap = 0;
  h->tcq_rows = -1;  // the query side is made again, whole
  h->n_views = 0;
}

void free_workspace(ss_handle *h) {
  free_host_pass(h->host);
  for (cudaEvent_t e : h->prof_ev) cudaEventDestroy(e);
  h->prof_ev.clear();
  h->prof_used = 0;
  free_lazy_buffers(h);
  void *ptrs[] = {h->d_status, h->row_next, h->probe, h->hot, h->slab, h->ell, h->meta,
                  h->counters, h->image, h->heavy_tbl};
  for (void *p : ptrs) cudaFree(p);
  h->d_status = nullptr;
  h->row_next = nullptr;
  h->probe = nullptr;
  h->hot = h->meta = h->counters = nullptr;
  h->slab = nullptr;
  h->ell = nullptr;
  h->image = nullptr;
  h->heavy_tbl = nullptr;
}

ss_status build_algo(ss_handle *h, int32_t algo, const ss_csr &items, int64_t rb, int64_t re,
                     cudaStream_t s) {
  // A build holds at most items.nnz entries: size the lists for that.
  ss_status st = ensure_capacity(h, algo, std::max<int64_t>(items.nnz, 1));
  if (st != SS_OK) return st;
  h->algo = algo;
  int queued = 0;
  if (algo == ALGO_TENSOR) {
    SS_CUDA(h, launch_tc_hot_select(h, items, s, &queued));
    h->launches += queued;
    SS_CUDA(h, launch_build_tc(h, items, rb, re, s, &queued));
    h->launches += queued;
    return SS_OK;
  }
  SS_CUDA(h, launch_hot_select(h, items, s, &queued));
  if (algo == ALGO_POSTING) {
    if ((st = ensure_posting_workspace(h)) != SS_OK) return st;
    SS_CUDA(h, launch_build_index(h, items, rb, re, s));
    h->launches += queued + kIndexKernels;
    return SS_OK;
  }
  SS_CUDA(h, launch_build_hybrid(h, items, rb, re, s));
  h->launches += queued + 1;
  return SS_OK;
}

bool same_auto_source(const ss_handle *h, const ss_csr &m) {
  return h->auto_src[0] == m.indptr && h->auto_src[1] == m.indices && h->auto_src[2] == m.values &&
         h->auto_src_rows == m.n_rows && h->auto_src_nnz == m.nnz;
}

// Builds the chunk indexes of [rb, re).  MODE_AUTO, for a new item matrix:
// the tensor path when a row sample shows a strong head (at least
// kAutoMinHot hot dimensions leaving at most kAutoMaxCold expected shared
// cold dimensions per pair); otherwise the hybrid hot set is chosen and
// every item tile of this first build is probed: when more than
// kAutoOverflowShare of them hold more cold entries than a shared-memory
// image takes (rows too long or too spread for item tiles), posting lists,
// else item tiles.  Reading the sample statistics (and the probe)
// synchronises the stream once per item matrix.
ss_status build_chunk(ss_handle *h, const ss_csr &items, int64_t rb, int64_t re, cudaStream_t s) {
  ss_status st = SS_OK;
  if (h->mode == MODE_POSTING) return build_algo(h, ALGO_POSTING, items, rb, re, s);
  if (h->mode == MODE_TILES) return build_algo(h, ALGO_HYBRID, items, rb, re, s);
  if (h->mode == MODE_TENSOR) return build_algo(h, ALGO_TENSOR, items, rb, re, s);
  if (!same_auto_source(h, items)) {
    int queued = 0;
    SS_CUDA(h, launch_tc_hot_select(h, items, s, &queued));
    h->launches += queued;
    if (h->tc_H >= tcp::kAutoMinHot && h->tc_est_cold <= tcp::kAutoMaxCold) {
      h->auto_algo = ALGO_TENSOR;
    } else {
      SS_CUDA(h, launch_hot_select(h, items, s, &queued));
      SS_CUDA(h, launch_auto_probe(h, items, rb, re, h->probe, s));
      h->launches += queued + 1;
      int32_t counts[2] = {0, 0};
      SS_CUDA(h, cudaMemcpyAsync(counts, h->probe, sizeof(counts), cudaMemcpyDeviceToHost, s));
      SS_CUDA(h, cudaStreamSynchronize(s));
      h->auto_algo = ((double)counts[1] > kAutoOverflowShare * (double)counts[0]) ? ALGO_POSTING : ALGO_HYBRID;
    }
    h->auto_src[0] = items.indptr;
    h->auto_src[1] = items.indices;
    h->auto_src[2] = items.values;
    h->auto_src_rows = items.n_rows;
    h->auto_src_nnz = items.nnz;
  }
  return build_algo(h, h->auto_algo, items, rb, re, s);
}

cudaError_t score(ss_handle *h, const ss_csr &q, const float *inv_q, const ss_index &idx,
                  const float *inv_i, float *out, int64_t ld_out, cudaStream_t s,
                  const ss_topk *topk = nullptr) {
  int queued = 0;
  if (idx.algo == ALGO_POSTING) {
    const cudaError_t e = launch_score_lists(h, q, inv_q, idx, inv_i, out, ld_out, s, &queued, topk);
    h->launches += queued;
    return e;
  }
  if (idx.algo == ALGO_TENSOR) {
    const cudaError_t e = launch_score_tc(h, q, inv_q, idx, inv_i, out, ld_out, s, &queued, topk);
    h->launches += queued;
    return e;
  }
  const cudaError_t e = launch_score_hybrid(h, q, inv_q, idx, inv_i, out, ld_out, s, &queued, topk);
  h->launches += queued;
  return e;
}

// Top-k candidate workspace for n_q rows of `cap` entries; synchronises the
// device when it has to grow.
ss_status ensure_topk_space(ss_handle *h, int64_t n_q, int64_t cap) {
  const int64_t elems = std::max<int64_t>(1, n_q * cap);
  if (elems <= h->cand_elems && n_q <= h->cand_rows) return SS_OK;
  SS_CUDA(h, cudaDeviceSynchronize());
  cudaFree(h->cand_val);
  cudaFree(h->cand_item);
  cudaFree(h->cand_n);
  h->cand_val = nullptr;
  h->cand_item = nullptr;
  h->cand_n = nullptr;
  h->cand_elems = h->cand_rows = 0;
  SS_CUDA(h, dev_alloc(&h->cand_val, sizeof(float) * (size_t)elems));
  SS_CUDA(h, dev_alloc(&h->cand_item, sizeof(int32_t) * (size_t)elems));
  SS_CUDA(h, dev_alloc(&h->cand_n, sizeof(int32_t) * (size_t)std::max<int64_t>(1, n_q)));
  SS_CUDA(h, cudaMemset(h->cand_n, 0, sizeof(int32_t) * (size_t)std::max<int64_t>(1, n_q)));
  h->cand_elems = elems;
  h->cand_rows = n_q;
  return SS_OK;
}

ss_status check_topk_args(ss_handle *h, int32_t k, const float *best_val, const int64_t *best_item,
                          int64_t n_q, const char *what) {
  if (k < 1 || k > kTopkMax) return fail(h, SS_ERR_LIMIT, "%s: k = %d outside [1, %d]", what, k, kTopkMax);
  if ((int64_t)k * (h->chunk_tiles + 1) > kTopkEntries)
    return fail(h, SS_ERR_LIMIT, "%s: k = %d too large for chunks of %d rows (k * (chunk_rows / 256 + 1) <= %d)",
                what, k, h->chunk_rows, kTopkEntries);
  if (n_q > 0 && (!best_val || !best_item)) return fail(h, SS_ERR_INVALID_ARG, "%s: null output", what);
  return SS_OK;
}

// Whether idx is one of the handle's current chunk indexes.
bool owns_index(const ss_handle *h, const ss_index *idx) {
  for (int k = 0; k < h->n_views; ++k)
    if (idx == &h->views[k]) return true;
  return false;
}

}  // namespace

cudaError_t dev_alloc(void **p, size_t bytes) {
  if (injected_failure()) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes);
}

cudaError_t host_alloc(void **p, size_t bytes) {
  if (injected_failure()) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaHostAlloc(p, bytes, cudaHostAllocDefault);
}

void reset_after_oom(ss_handle *h) {
  cudaDeviceSynchronize();
  cudaGetLastError();
  free_lazy_buffers(h);
  ss_invalidate(h);
}

cudaError_t ensure_dyn_smem(const void *kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void *, int>, size_t> raised;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t &have = raised[{kernel, dev}];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

void prof_mark(ss_handle *h, cudaStream_t s) {
  if (!h->prof_on) return;
  if (h->prof_used == h->prof_ev.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) {
      h->prof_on = false;
      return;
    }
    h->prof_ev.push_back(e);
  }
  cudaEventRecord(h->prof_ev[h->prof_used++], s);
}

extern "C" {

const char *ss_status_string(ss_status s) {
  switch (s) {
    case SS_OK: return "ok";
    case SS_ERR_INVALID_ARG: return "invalid argument";
    case SS_ERR_UNSORTED: return "indices not strictly increasing within a row";
    case SS_ERR_OUT_OF_RANGE: return "index out of range";
    case SS_ERR_OOM: return "out of memory";
    case SS_ERR_CUDA: return "CUDA error";
    case SS_ERR_DEVICE_CHECK: return "device-side check failed";
    case SS_ERR_TIMEOUT: return "timed out waiting for the GPU";
    case SS_ERR_LIMIT: return "size beyond a documented limit";
    default: return "unknown status";
  }
}

const char *ss_last_error(const ss_handle *h) { return h ? h->last_error.c_str() : ""; }

uint64_t ss_kernel_launches(const ss_handle *h) { return h ? h->launches : 0; }

int64_t ss_inject_alloc_failure(int64_t nth) { return g_alloc_countdown.exchange(nth > 0 ? nth : 0); }

ss_status ss_profile_scorer(ss_handle *h, int32_t on) {
  if (!h) return SS_ERR_INVALID_ARG;
  h->prof_on = on != 0;  // the pairs recorded so far stay until ss_scorer_time reads them
  return SS_OK;
}

ss_status ss_scorer_time(ss_handle *h, double *total_ms, int64_t *launches) {
  if (!h || !total_ms || !launches) return SS_ERR_INVALID_ARG;
  *total_ms = 0.0;
  *launches = 0;
  ss_status st = set_device(h);
  if (st != SS_OK) return st;
  const size_t pairs = h->prof_used / 2;
  if (pairs > 0) SS_CUDA(h, cudaEventSynchronize(h->prof_ev[2 * pairs - 1]));
  for (size_t k = 0; k < pairs; ++k) {
    float ms = 0.f;
    SS_CUDA(h, cudaEventElapsedTime(&ms, h->prof_ev[2 * k], h->prof_ev[2 * k + 1]));
    *total_ms += ms;
  }
  *launches = (int64_t)pairs;
  h->prof_used = 0;
  return SS_OK;
}

ss_status ss_create(ss_handle **out, int device, int64_t dim, int32_t chunk_rows, int32_t flags) {
  if (!out) return SS_ERR_INVALID_ARG;
  *out = nullptr;
  if (dim <= 0 || chunk_rows <= 0) return SS_ERR_INVALID_ARG;
  if (chunk_rows > SS_MAX_CHUNK_ROWS || dim >= ((int64_t)1 << 31) - 1) return SS_ERR_LIMIT;
  ss_handle *h = new (std::nothrow) ss_handle();
  if (!h) return SS_ERR_OOM;
  h->device = device;
  h->dim = dim;
  h->chunk_rows = chunk_rows;
  h->flags = flags;
  const int n_algo_flags = ((flags & SS_ALGO_POSTING_LISTS) != 0) + ((flags & SS_ALGO_TILES) != 0) +
                           ((flags & SS_ALGO_TENSOR) != 0);
  if (n_algo_flags > 1) {
    delete h;
    return SS_ERR_INVALID_ARG;
  }
  h->mode = (flags & SS_ALGO_POSTING_LISTS) ? MODE_POSTING
            : (flags & SS_ALGO_TILES)       ? MODE_TILES
            : (flags & SS_ALGO_TENSOR)      ? MODE_TENSOR
                                            : MODE_AUTO;
  h->algo = (h->mode == MODE_POSTING) ? ALGO_POSTING : (h->mode == MODE_TENSOR) ? ALGO_TENSOR : ALGO_HYBRID;
  cudaError_t e = cudaSetDevice(device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device);
  if (e == cudaSuccess) e = dev_alloc(&h->d_status, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = dev_alloc(&h->row_next, 2 * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->row_next, 0, 2 * sizeof(int32_t));
  if (e == cudaSuccess) e = dev_alloc(&h->probe, 2 * sizeof(int32_t));
  if (e == cudaSuccess) e = dev_alloc(&h->hot, sizeof(int32_t) * (1 + hyb::kHotMax));
  if (e == cudaSuccess) e = cudaMemset(h->hot, 0, sizeof(int32_t) * (1 + hyb::kHotMax));
  {
    using namespace hyb;
    // One build covers enough chunks to give every SM a tile (a chunk alone
    // has only chunk_rows / 256 tiles, one block each).
    h->chunk_tiles = (chunk_rows + kTI - 1) / kTI;
    const int sms = h->sm_count > 0 ? h->sm_count : 1;
    h->build_batch = std::max(1, std::min(kMaxBuildBatch, (sms + h->chunk_tiles - 1) / h->chunk_tiles));
    h->max_tiles = h->build_batch * h->chunk_tiles;
  }
  // The posting-list workspace is allocated by the first posting build; the
  // tile workspace unless the handle only ever builds posting lists.
  if (e == cudaSuccess && h->mode != MODE_POSTING && h->mode != MODE_TENSOR) {
    using namespace hyb;
    const size_t tiles = (size_t)h->max_tiles;
    if (e == cudaSuccess) e = dev_alloc(&h->slab, sizeof(float) * tiles * kHotMax * kTI);
    if (e == cudaSuccess) e = dev_alloc(&h->ell, sizeof(int2) * tiles * kEllMaxW * kTI);
    if (e == cudaSuccess) e = dev_alloc(&h->meta, sizeof(int32_t) * tiles * kMetaInts);
    if (e == cudaSuccess) e = dev_alloc(&h->heavy_tbl, sizeof(int4) * tiles * kTI);
    const size_t n_counters = 1 + (size_t)h->build_batch * (1 + h->chunk_tiles);
    if (e == cudaSuccess) e = dev_alloc(&h->counters, sizeof(int32_t) * n_counters);
    if (e == cudaSuccess) e = cudaMemset(h->counters, 0, sizeof(int32_t) * n_counters);
    if (e == cudaSuccess) e = dev_alloc(&h->image, (size_t)kImgBytes * tiles);
  }
  if (e != cudaSuccess) {
    const ss_status st = (e == cudaErrorMemoryAllocation) ? SS_ERR_OOM : SS_ERR_CUDA;
    free_workspace(h);
    delete h;
    return st;
  }
  *out = h;
  return SS_OK;
}

ss_status ss_destroy(ss_handle *h) {
  if (!h) return SS_ERR_INVALID_ARG;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  free_workspace(h);
  delete h;
  return SS_OK;
}

ss_status ss_validate_csr(ss_handle *h, const ss_csr *m, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  ss_status st = check_csr_args(h, m, "ss_validate_csr");
  if (st != SS_OK) return st;
  if ((st = set_device(h)) != SS_OK) return st;
  return validate(h, *m, as_stream(stream), "ss_validate_csr");
}

ss_status ss_invalidate(ss_handle *h) {
  if (!h) return SS_ERR_INVALID_ARG;
  invalidate_queries(h);
  for (int j = 0; j < 3; ++j) h->hot_src[j] = h->auto_src[j] = h->tc_hot_src[j] = nullptr;
  h->tc_hot_rows = h->tc_hot_nnz = h->hot_src_rows = h->hot_src_nnz = -1;
  h->auto_src_rows = h->auto_src_nnz = -1;
  return SS_OK;
}

ss_status ss_index_stats(ss_handle *h, const ss_index *idx, int64_t *stats, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  if (!idx || !owns_index(h, idx) || !stats)
    return fail(h, SS_ERR_INVALID_ARG, "ss_index_stats: bad index or output");
  ss_status st = set_device(h);
  if (st != SS_OK) return st;
  for (int j = 0; j < 8; ++j) stats[j] = 0;
  stats[0] = idx->algo;
  stats[1] = idx->n_items;
  SS_CUDA(h, cudaStreamSynchronize(as_stream(stream)));
  if (idx->algo == ALGO_TENSOR) {
    std::vector<int2> rng((size_t)idx->n_items);
    SS_CUDA(h, cudaMemcpy(rng.data(), idx->icold_rng, sizeof(int2) * rng.size(), cudaMemcpyDeviceToHost));
    for (const int2 &r : rng) stats[6] += r.y;
    int32_t hcount = 0;
    SS_CUDA(h, cudaMemcpy(&hcount, idx->hot, sizeof(int32_t), cudaMemcpyDeviceToHost));
    stats[3] = hcount;
    return SS_OK;
  }
  if (idx->algo == ALGO_POSTING) {
    int32_t ends[2] = {0, 0};
    SS_CUDA(h, cudaMemcpy(&ends[0], idx->col_ptr, sizeof(int32_t), cudaMemcpyDeviceToHost));
    SS_CUDA(h, cudaMemcpy(&ends[1], idx->col_ptr + idx->dim, sizeof(int32_t), cudaMemcpyDeviceToHost));
    stats[6] = ends[1] - ends[0];
    if (idx->hot) {  // hot dimensions split off into the dense slab (0 when too few)
      int32_t hcount = 0;
      SS_CUDA(h, cudaMemcpy(&hcount, idx->hot, sizeof(int32_t), cudaMemcpyDeviceToHost));
      stats[3] = hcount >= kSplitMinHot ? hcount : 0;
    }
    return SS_OK;
  }
  if (idx->n_tiles == 0) return SS_OK;
  stats[2] = idx->n_tiles;
  int32_t hcount = 0;
  SS_CUDA(h, cudaMemcpy(&hcount, idx->hot, sizeof(int32_t), cudaMemcpyDeviceToHost));
  stats[3] = hcount;
  int32_t n_ovf = 0;
  SS_CUDA(h, cudaMemcpy(&n_ovf, idx->counters + 1, sizeof(int32_t), cudaMemcpyDeviceToHost));
  stats[7] = n_ovf;
  std::vector<int32_t> meta((size_t)idx->n_tiles * hyb::kMetaInts);
  SS_CUDA(h, cudaMemcpy(meta.data(), idx->meta, sizeof(int32_t) * meta.size(), cudaMemcpyDeviceToHost));
  for (int32_t t = 0; t < idx->n_tiles; ++t) {
    const int32_t *m = meta.data() + (size_t)t * hyb::kMetaInts;
    stats[4] += m[9];
    for (int w = 0; w < 8; ++w) {
      stats[5] = std::max<int64_t>(stats[5], m[w]);
      stats[6] += (int64_t)m[w] * 32;
    }
  }
  return SS_OK;
}

static_assert(tcp::kHotMax <= SS_EXPORT_HOT_MAX && hyb::kHotMax <= SS_EXPORT_HOT_MAX,
              "every hot set fits the export's rows");

ss_status ss_index_export(ss_handle *h, const ss_index *idx, int32_t *n_hot, int32_t *hot,
                          float *hot_values, int32_t *col_ptr, int32_t *item, float *value,
                          int64_t capacity, int64_t *n_entries, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  if (!idx || !owns_index(h, idx))
    return fail(h, SS_ERR_INVALID_ARG, "ss_index_export: index does not belong to this handle");
  if (idx->algo != ALGO_POSTING && idx->algo != ALGO_TENSOR)
    return fail(h, SS_ERR_INVALID_ARG, "ss_index_export: item-tile indexes have no list form");
  if (capacity < 0) return fail(h, SS_ERR_INVALID_ARG, "ss_index_export: negative capacity");
  ss_status st = set_device(h);
  if (st != SS_OK) return st;
  SS_CUDA(h, cudaStreamSynchronize(as_stream(stream)));
  const int64_t n_items = idx->n_items, dim = idx->dim;

  // The dimensions held dense, and their values per item.
  std::vector<int32_t> hot_set;
  if (idx->hot) {
    const int hmax = idx->algo == ALGO_TENSOR ? tcp::kHotMax : hyb::kHotMax;
    std::vector<int32_t> raw(1 + (size_t)hmax);
    SS_CUDA(h, cudaMemcpy(raw.data(), idx->hot, sizeof(int32_t) * raw.size(), cudaMemcpyDeviceToHost));
    const int H = std::max(0, std::min(raw[0], hmax));
    // Posting lists keep every dimension in the lists below kSplitMinHot.
    if (idx->algo == ALGO_TENSOR || H >= kSplitMinHot) hot_set.assign(raw.begin() + 1, raw.begin() + 1 + H);
  }
  const int H = (int)hot_set.size();
  if (n_hot) *n_hot = H;
  if (hot) std::copy(hot_set.begin(), hot_set.end(), hot);
  if (hot_values) {
    std::fill(hot_values, hot_values + (size_t)n_items * SS_EXPORT_HOT_MAX, 0.f);
    if (H > 0) {
      if (idx->algo == ALGO_TENSOR) {  // slab [item][kHotMax]
        std::vector<float> slab((size_t)n_items * tcp::kHotMax);
        SS_CUDA(h, cudaMemcpy(slab.data(), idx->slab, sizeof(float) * slab.size(), cudaMemcpyDeviceToHost));
        for (int64_t i = 0; i < n_items; ++i)
          for (int j = 0; j < H; ++j) hot_values[i * SS_EXPORT_HOT_MAX + j] = slab[(size_t)i * tcp::kHotMax + j];
      } else {  // slab [hot dim][slab_ld]
        std::vector<float> slab((size_t)hyb::kHotMax * idx->slab_ld);
        SS_CUDA(h, cudaMemcpy(slab.data(), idx->slab, sizeof(float) * slab.size(), cudaMemcpyDeviceToHost));
        for (int64_t i = 0; i < n_items; ++i)
          for (int j = 0; j < H; ++j) hot_values[i * SS_EXPORT_HOT_MAX + j] = slab[(size_t)j * idx->slab_ld + i];
      }
    }
  }

  if (idx->algo == ALGO_TENSOR) {
    // The tensor path keeps each item's cold entries (CSR order); their
    // lists by dimension, items ascending, are made here.
    std::vector<int2> rng((size_t)n_items);
    SS_CUDA(h, cudaMemcpy(rng.data(), idx->icold_rng, sizeof(int2) * rng.size(), cudaMemcpyDeviceToHost));
    int64_t lo = INT64_MAX, hi = 0, n = 0;
    for (const int2 &r : rng) {
      if (r.x < 0 || r.y < 0) return fail(h, SS_ERR_DEVICE_CHECK, "ss_index_export: bad cold entry range");
      if (r.y > 0) {
        lo = std::min<int64_t>(lo, r.x);
        hi = std::max<int64_t>(hi, (int64_t)r.x + r.y);
      }
      n += r.y;
    }
    if (n > 0 && hi > idx->capacity) return fail(h, SS_ERR_DEVICE_CHECK, "ss_index_export: entries outside the index");
    if (n_entries) *n_entries = n;
    std::vector<int2> ent(n > 0 ? (size_t)(hi - lo) : 0);
    if (n > 0) SS_CUDA(h, cudaMemcpy(ent.data(), idx->icold + lo, sizeof(int2) * ent.size(), cudaMemcpyDeviceToHost));
    std::vector<int64_t> ptr((size_t)dim + 2, 0);
    for (int64_t i = 0; i < n_items; ++i)
      for (int j = 0; j < rng[(size_t)i].y; ++j) {
        const int32_t k = ent[(size_t)(rng[(size_t)i].x - lo + j)].x;
        if (k < 0 || k >= dim) return fail(h, SS_ERR_DEVICE_CHECK, "ss_index_export: dimension out of range");
        ++ptr[(size_t)k + 2];
      }
    for (int64_t k = 0; k < dim; ++k) ptr[(size_t)k + 2] += ptr[(size_t)k + 1];
    if (col_ptr)
      for (int64_t k = 0; k <= dim; ++k) col_ptr[k] = (int32_t)ptr[(size_t)k + 1];
    if (item || value) {
      if (capacity < n) return fail(h, SS_ERR_LIMIT, "ss_index_export: %lld entries exceed capacity %lld",
                                    (long long)n, (long long)capacity);
      for (int64_t i = 0; i < n_items; ++i)  // items in order: each list ascends
        for (int j = 0; j < rng[(size_t)i].y; ++j) {
          const int2 e = ent[(size_t)(rng[(size_t)i].x - lo + j)];
          const int64_t at = ptr[(size_t)e.x + 1]++;
          if (item) item[at] = (int32_t)i;
          if (value) memcpy(value + at, &e.y, sizeof(float));
        }
    }
    return SS_OK;
  }

  // The lists, positions made relative to the chunk's first entry and each
  // list put in ascending item order (the device leaves it unspecified).
  std::vector<int32_t> ptr((size_t)dim + 1);
  SS_CUDA(h, cudaMemcpy(ptr.data(), idx->col_ptr, sizeof(int32_t) * ptr.size(), cudaMemcpyDeviceToHost));
  const int64_t base = ptr[0], n = (int64_t)ptr[dim] - base;
  if (n < 0 || base < 0 || base + n > idx->capacity)
    return fail(h, SS_ERR_DEVICE_CHECK, "ss_index_export: list offsets outside the index");
  if (n_entries) *n_entries = n;
  if (col_ptr)
    for (int64_t k = 0; k <= dim; ++k) col_ptr[k] = (int32_t)(ptr[k] - base);
  if (item || value) {
    if (capacity < n) return fail(h, SS_ERR_LIMIT, "ss_index_export: %lld entries exceed capacity %lld",
                                  (long long)n, (long long)capacity);
    std::vector<uint16_t> it((size_t)n);
    std::vector<float> val((size_t)n);
    if (n > 0) {
      SS_CUDA(h, cudaMemcpy(it.data(), idx->post_item + base, sizeof(uint16_t) * (size_t)n, cudaMemcpyDeviceToHost));
      SS_CUDA(h, cudaMemcpy(val.data(), idx->post_val + base, sizeof(float) * (size_t)n, cudaMemcpyDeviceToHost));
    }
    std::vector<int64_t> order;
    for (int64_t k = 0; k < dim; ++k) {
      const int64_t b = ptr[k] - base, e = ptr[k + 1] - base;
      order.resize((size_t)(e - b));
      for (int64_t p = b; p < e; ++p) order[(size_t)(p - b)] = p;
      std::sort(order.begin(), order.end(), [&](int64_t x, int64_t y) { return it[(size_t)x] < it[(size_t)y]; });
      for (int64_t p = b; p < e; ++p) {
        if (item) item[p] = it[(size_t)order[(size_t)(p - b)]];
        if (value) value[p] = val[(size_t)order[(size_t)(p - b)]];
      }
    }
  }
  return SS_OK;
}

ss_status ss_lists_export(ss_handle *h, int64_t *n_dims, int32_t *dims, int32_t *col_ptr, int32_t *query,
                          float *value, int64_t capacity, int64_t *n_entries, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  if (!h->tc_qptr || !h->tc_qlist || h->tcq_rows < 0 || capacity < 0)
    return fail(h, SS_ERR_INVALID_ARG, "ss_lists_export: no tensor-path scoring call made yet");
  ss_status st = set_device(h);
  if (st != SS_OK) return st;
  SS_CUDA(h, cudaStreamSynchronize(as_stream(stream)));
  const int64_t dim = h->dim, S = h->tcq_slices, stride = dim + 1;
  std::vector<int32_t> off((size_t)(S * stride));
  SS_CUDA(h, cudaMemcpy(off.data(), h->tc_qptr, sizeof(int32_t) * off.size(), cudaMemcpyDeviceToHost));
  const int64_t n = S > 0 ? off[(size_t)(S * stride - 1)] : 0;
  if (S < 1 || off[0] != 0 || n < 0 || n > h->tc_qlist_cap)
    return fail(h, SS_ERR_DEVICE_CHECK, "ss_lists_export: offsets outside the lists");
  for (int64_t k = 1; k < S * stride; ++k)
    if (off[(size_t)k] < off[(size_t)k - 1]) return fail(h, SS_ERR_DEVICE_CHECK, "ss_lists_export: offsets not ascending");
  // The slices' lists of each dimension, merged.
  std::vector<int32_t> ptr(1, 0), held;
  for (int64_t d = 0; d < dim; ++d) {
    int64_t len = 0;
    for (int64_t sl = 0; sl < S; ++sl) len += off[(size_t)(sl * stride + d + 1)] - off[(size_t)(sl * stride + d)];
    if (len > 0) {
      held.push_back((int32_t)d);
      ptr.push_back(ptr.back() + (int32_t)len);
    }
  }
  const int64_t nd = (int64_t)held.size();
  if (ptr.back() != n) return fail(h, SS_ERR_DEVICE_CHECK, "ss_lists_export: slices inconsistent");
  if (n_dims) *n_dims = nd;
  if (n_entries) *n_entries = n;
  if (dims && nd > 0) memcpy(dims, held.data(), sizeof(int32_t) * held.size());
  if (col_ptr) memcpy(col_ptr, ptr.data(), sizeof(int32_t) * ptr.size());
  if (query || value) {
    if (capacity < n)
      return fail(h, SS_ERR_LIMIT, "ss_lists_export: %lld entries exceed capacity %lld", (long long)n,
                  (long long)capacity);
    std::vector<int2> raw((size_t)n), ent;
    ent.reserve((size_t)n);
    if (n > 0) SS_CUDA(h, cudaMemcpy(raw.data(), h->tc_qlist, sizeof(int2) * (size_t)n, cudaMemcpyDeviceToHost));
    for (int64_t k = 0; k < nd; ++k) {
      const int64_t d = held[(size_t)k];
      for (int64_t sl = 0; sl < S; ++sl)
        ent.insert(ent.end(), raw.begin() + off[(size_t)(sl * stride + d)], raw.begin() + off[(size_t)(sl * stride + d + 1)]);
      // each list by ascending query row (the device order is unspecified)
      std::sort(ent.begin() + ptr[(size_t)k], ent.end(), [](const int2 &x, const int2 &y) { return x.x < y.x; });
    }
    for (int64_t p = 0; p < n; ++p) {
      if (query) query[p] = ent[(size_t)p].x;
      if (value) memcpy(value + p, &ent[(size_t)p].y, sizeof(float));
    }
  }
  return SS_OK;
}

ss_status ss_check_device(ss_handle *h, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  ss_status st = set_device(h);
  if (st != SS_OK) return st;
  // Work of a host pass that returned early (a timeout, a stopped consumer)
  // may still be queued on the pass's own streams.
  for (cudaStream_t ps : {h->host.comp, h->host.copy, h->host.up})
    if (ps) SS_CUDA(h, cudaStreamSynchronize(ps));
  int32_t code = 0;
  if ((st = read_status(h, as_stream(stream), &code)) != SS_OK) return st;
  return status_from_device(h, code, "ss_check_device");
}

ss_status ss_row_norms(ss_handle *h, const ss_csr *m, float *inv_norms, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  ss_status st = check_csr_args(h, m, "ss_row_norms");
  if (st != SS_OK) return st;
  if (m->n_rows > 0 && !inv_norms) return fail(h, SS_ERR_INVALID_ARG, "ss_row_norms: null output");
  if ((st = set_device(h)) != SS_OK) return st;
  cudaStream_t s = as_stream(stream);
  if (h->flags & SS_VALIDATE) {
    if ((st = validate(h, *m, s, "ss_row_norms")) != SS_OK) return st;
  }
  SS_CUDA(h, launch_row_norms(*m, inv_norms, h->sm_count, s));
  if (m->n_rows > 0) h->launches += 1;
  return SS_OK;
}

ss_status ss_build_item_index(ss_handle *h, const ss_csr *items, int64_t row_begin,
                              int64_t row_end, ss_index **out, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  if (!out) return fail(h, SS_ERR_INVALID_ARG, "ss_build_item_index: null out");
  *out = nullptr;
  ss_status st = check_csr_args(h, items, "ss_build_item_index");
  if (st != SS_OK) return st;
  if (row_begin < 0 || row_end <= row_begin || row_end > items->n_rows)
    return fail(h, SS_ERR_INVALID_ARG, "ss_build_item_index: bad row range [%lld, %lld)",
                (long long)row_begin, (long long)row_end);
  if (row_end - row_begin > h->chunk_rows)
    return fail(h, SS_ERR_LIMIT, "ss_build_item_index: %lld rows exceed chunk_rows %d",
                (long long)(row_end - row_begin), h->chunk_rows);
  if ((st = set_device(h)) != SS_OK) return st;
  if ((st = build_chunk(h, *items, row_begin, row_end, as_stream(stream))) != SS_OK) return st;
  *out = &h->views[0];
  return SS_OK;
}

int32_t ss_build_batch(const ss_handle *h) { return h ? h->build_batch : 0; }

ss_status ss_build_item_indexes(ss_handle *h, const ss_csr *items, int64_t row_begin,
                                int64_t row_end, ss_index **out, int32_t *n_out, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  if (!out || !n_out) return fail(h, SS_ERR_INVALID_ARG, "ss_build_item_indexes: null out");
  *n_out = 0;
  ss_status st = check_csr_args(h, items, "ss_build_item_indexes");
  if (st != SS_OK) return st;
  if (row_begin < 0 || row_end <= row_begin || row_end > items->n_rows)
    return fail(h, SS_ERR_INVALID_ARG, "ss_build_item_indexes: bad row range [%lld, %lld)",
                (long long)row_begin, (long long)row_end);
  const int64_t n_chunks = (row_end - row_begin + h->chunk_rows - 1) / h->chunk_rows;
  if (n_chunks > h->build_batch)
    return fail(h, SS_ERR_LIMIT, "ss_build_item_indexes: %lld chunks exceed the build batch %d",
                (long long)n_chunks, h->build_batch);
  if ((st = set_device(h)) != SS_OK) return st;
  if ((st = build_chunk(h, *items, row_begin, row_end, as_stream(stream))) != SS_OK) return st;
  for (int k = 0; k < h->n_views; ++k) out[k] = &h->views[k];
  *n_out = h->n_views;
  return SS_OK;
}

ss_status ss_score_chunk(ss_handle *h, const ss_csr *queries, const float *inv_q,
                         const ss_index *idx, const float *inv_i, float *out, int64_t ld_out,
                         void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  ss_status st = check_csr_args(h, queries, "ss_score_chunk");
  if (st != SS_OK) return st;
  if (!idx || !owns_index(h, idx))
    return fail(h, SS_ERR_INVALID_ARG, "ss_score_chunk: index does not belong to this handle");
  if (queries->n_rows > 0 && (!inv_q || !inv_i || !out))
    return fail(h, SS_ERR_INVALID_ARG, "ss_score_chunk: null norms or output");
  if (ld_out < idx->n_items)
    return fail(h, SS_ERR_INVALID_ARG, "ss_score_chunk: ld_out %lld < chunk width %d",
                (long long)ld_out, idx->n_items);
  if ((st = set_device(h)) != SS_OK) return st;
  SS_CUDA(h, score(h, *queries, inv_q, *idx, inv_i, out, ld_out, as_stream(stream)));
  return SS_OK;
}

ss_status ss_score_all(ss_handle *h, const ss_csr *queries, const float *inv_q,
                       const ss_csr *items, const float *inv_i, float *out, int64_t ld_out,
                       void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  ss_status st = check_csr_args(h, queries, "ss_score_all");
  if (st == SS_OK) st = check_csr_args(h, items, "ss_score_all");
  if (st != SS_OK) return st;
  if (ld_out < items->n_rows)
    return fail(h, SS_ERR_INVALID_ARG, "ss_score_all: ld_out < number of items");
  if (queries->n_rows == 0 || items->n_rows == 0) return SS_OK;
  if (!inv_q || !inv_i || !out) return fail(h, SS_ERR_INVALID_ARG, "ss_score_all: null pointer");
  if ((st = set_device(h)) != SS_OK) return st;
  cudaStream_t s = as_stream(stream);
  // One build per batch of chunks, then each chunk scored on its own.
  const int64_t span = (int64_t)h->chunk_rows * h->build_batch;
  for (int64_t bb = 0; bb < items->n_rows; bb += span) {
    const int64_t be = std::min<int64_t>(bb + span, items->n_rows);
    if ((st = build_chunk(h, *items, bb, be, s)) != SS_OK) return st;
    for (int k = 0; k < h->n_views; ++k) {
      const ss_index &v = h->views[k];
      SS_CUDA(h, score(h, *queries, inv_q, v, inv_i + v.row_begin, out + v.row_begin, ld_out, s));
    }
  }
  return SS_OK;
}

ss_status ss_topk_reset(ss_handle *h, int64_t n_q, int32_t k, float *best_val, int64_t *best_item,
                        void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  if (n_q < 0) return fail(h, SS_ERR_INVALID_ARG, "ss_topk_reset: n_q < 0");
  ss_status st = check_topk_args(h, k, best_val, best_item, n_q, "ss_topk_reset");
  if (st != SS_OK) return st;
  if ((st = set_device(h)) != SS_OK) return st;
  if ((st = ensure_topk_space(h, n_q, (int64_t)h->chunk_tiles * k)) != SS_OK) return st;
  SS_CUDA(h, launch_topk_reset(n_q, k, best_val, best_item, h->cand_n, h->sm_count, as_stream(stream)));
  if (n_q > 0) h->launches += 1;
  return SS_OK;
}

ss_status ss_score_chunk_topk(ss_handle *h, const ss_csr *queries, const float *inv_q,
                              const ss_index *idx, const float *inv_i, int32_t k, float *best_val,
                              int64_t *best_item, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  ss_status st = check_csr_args(h, queries, "ss_score_chunk_topk");
  if (st != SS_OK) return st;
  if ((st = check_topk_args(h, k, best_val, best_item, queries->n_rows, "ss_score_chunk_topk")) != SS_OK)
    return st;
  if (!idx || !owns_index(h, idx))
    return fail(h, SS_ERR_INVALID_ARG, "ss_score_chunk_topk: index does not belong to this handle");
  if (queries->n_rows == 0 || idx->n_items == 0) return SS_OK;
  if (!inv_q || !inv_i) return fail(h, SS_ERR_INVALID_ARG, "ss_score_chunk_topk: null norms");
  if (queries->n_rows > h->cand_rows || (int64_t)h->chunk_tiles * k * queries->n_rows > h->cand_elems)
    return fail(h, SS_ERR_INVALID_ARG, "ss_score_chunk_topk: call ss_topk_reset for these rows and k first");
  if ((st = set_device(h)) != SS_OK) return st;
  cudaStream_t s = as_stream(stream);
  ss_topk t;
  t.k = k;
  t.best_val = best_val;
  t.cand_val = h->cand_val;
  t.cand_item = h->cand_item;
  t.cand_n = h->cand_n;
  t.cand_cap = h->chunk_tiles * k;
  SS_CUDA(h, score(h, *queries, inv_q, *idx, inv_i, nullptr, idx->n_items, s, &t));
  SS_CUDA(h, launch_topk_merge(t, queries->n_rows, idx->row_begin, best_val, best_item, h->sm_count, s));
  h->launches += 1;
  return SS_OK;
}

ss_status ss_tile_checksum(ss_handle *h, const float *tile, int64_t n_rows, int64_t n_cols,
                           int64_t ld, uint64_t *bits_sum, double *value_sum, void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  if (n_rows < 0 || n_cols < 0 || ld < n_cols || !bits_sum || !value_sum ||
      (n_rows > 0 && n_cols > 0 && !tile))
    return fail(h, SS_ERR_INVALID_ARG, "ss_tile_checksum: bad arguments");
  ss_status st = set_device(h);
  if (st != SS_OK) return st;
  SS_CUDA(h, launch_tile_checksum(tile, n_rows, n_cols, ld, bits_sum, value_sum, h->sm_count,
                                  as_stream(stream)));
  if (n_rows > 0 && n_cols > 0) h->launches += 1;
  return SS_OK;
}

ss_status ss_tile_checksum_host(const float *tile, int64_t n_rows, int64_t n_cols, int64_t ld,
                                uint64_t *bits_sum, double *value_sum) {
  if (n_rows < 0 || n_cols < 0 || ld < n_cols || !bits_sum || !value_sum ||
      (n_rows > 0 && n_cols > 0 && !tile))
    return SS_ERR_INVALID_ARG;
  tile_checksum_host(tile, n_rows, n_cols, ld, bits_sum, value_sum);
  return SS_OK;
}

ss_status ss_stream_checksum(const ss_handle *h, int64_t chunk, uint64_t *bits_sum,
                             double *value_sum) {
  if (!h || !bits_sum || !value_sum || chunk < 0 || chunk >= (int64_t)h->host.log_bits.size())
    return SS_ERR_INVALID_ARG;
  *bits_sum = h->host.log_bits[(size_t)chunk];
  *value_sum = h->host.log_values[(size_t)chunk];
  return SS_OK;
}

ss_status ss_topk_all(ss_handle *h, const ss_csr *queries, const float *inv_q, const ss_csr *items,
                      const float *inv_i, int32_t k, float *best_val, int64_t *best_item,
                      void *stream) {
  if (!h) return SS_ERR_INVALID_ARG;
  ss_status st = check_csr_args(h, queries, "ss_topk_all");
  if (st == SS_OK) st = check_csr_args(h, items, "ss_topk_all");
  if (st != SS_OK) return st;
  if ((st = ss_topk_reset(h, queries->n_rows, k, best_val, best_item, stream)) != SS_OK) return st;
  if (queries->n_rows == 0 || items->n_rows == 0) return SS_OK;
  if (!inv_q || !inv_i) return fail(h, SS_ERR_INVALID_ARG, "ss_topk_all: null norms");
  cudaStream_t s = as_stream(stream);
  const int64_t span = (int64_t)h->chunk_rows * h->build_batch;
  for (int64_t bb = 0; bb < items->n_rows; bb += span) {
    const int64_t be = std::min<int64_t>(bb + span, items->n_rows);
    if ((st = build_chunk(h, *items, bb, be, s)) != SS_OK) return st;
    for (int v = 0; v < h->n_views; ++v) {
      const ss_index *ix = &h->views[v];
      if ((st = ss_score_chunk_topk(h, queries, inv_q, ix, inv_i + ix->row_begin, k, best_val,
                                    best_item, stream)) != SS_OK)
        return st;
    }
  }
  return SS_OK;
}

}  // extern "C"
