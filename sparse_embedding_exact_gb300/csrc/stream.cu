// Host-buffer streaming pass: the "streaming batch" pipeline of the blog post
// ("Engineering practice for bulk similarity calculation over sparse
// embeddings", sections 2.2 and 4.4): items are scored chunk by chunk and
// each chunk's slice of the result reaches host memory.
//
// When the caller's output is page-locked host memory that the device can
// address, each chunk's scoring kernel stores its normalised tile straight
// into it (device stores cross to host memory at the same rate as the copy
// engines, and a pitched store costs no more than a contiguous one, while a
// pitched copy-engine transfer of the chunk's rows runs at about half that
// rate).  Otherwise two device output buffers alternate between chunks: the
// compute stream builds the index and scores chunk c into buffer c % 2, the
// copy stream then copies the buffer into slot c % R of a ring of
// page-locked buffers, from which the host copies rows out or hands the tile
// to the caller's consumer.  Events order buffer and slot reuse; every host
// wait polls its event with a deadline.  Streams, events and buffers stay
// with the handle between calls.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <string>
#include <thread>
#include <vector>

#include "internal.cuh"

namespace {

ss_status sfail(ss_handle *h, ss_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  h->last_error = buf;
  return st;
}

ss_status scuda(ss_handle *h, cudaError_t e, const char *what) {
  const ss_status st = (e == cudaErrorMemoryAllocation) ? SS_ERR_OOM : SS_ERR_CUDA;
  if (st == SS_ERR_OOM) reset_after_oom(h);
  return sfail(h, st, "%s: %s", what, cudaGetErrorString(e));
}

#define S_CUDA(call)                                    \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return scuda(h, e_, #call);  \
  } while (0)
#define SS_CUDA_LAUNCH(call)                            \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return scuda(h, e_, #call);  \
    h->launches += 1;                                   \
  } while (0)

ss_status wait_event(ss_handle *h, cudaEvent_t ev, int32_t timeout_ms, const char *what) {
  const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
  for (;;) {
    const cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return SS_OK;
    if (e != cudaErrorNotReady) return scuda(h, e, what);
    if (std::chrono::steady_clock::now() > deadline)
      return sfail(h, SS_ERR_TIMEOUT, "%s: no completion within %d ms", what, timeout_ms);
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

// Copies rows of a ring slot (ld = chunk width) into the caller's output.
void scatter_rows(float *out, int64_t ld_out, int64_t col0, const float *slot, int64_t ld_slot,
                  int64_t width, int64_t n_rows) {
  const unsigned hw = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
  const int64_t per = (n_rows + hw - 1) / hw;
  auto work = [&](int64_t r0, int64_t r1) {
    for (int64_t r = r0; r < r1; ++r)
      memcpy(out + r * ld_out + col0, slot + r * ld_slot, sizeof(float) * (size_t)width);
  };
  if (n_rows * width < (1 << 20) || hw == 1) {
    work(0, n_rows);
    return;
  }
  std::vector<std::thread> th;
  for (unsigned t = 0; t < hw; ++t) {
    const int64_t r0 = t * per, r1 = std::min(n_rows, r0 + per);
    if (r0 < r1) th.emplace_back(work, r0, r1);
  }
  for (auto &t : th) t.join();
}

ss_status check_host_csr(ss_handle *h, const ss_csr *m, const char *what) {
  if (!m || !m->indptr || m->n_rows < 0 || m->nnz < 0 || (m->nnz > 0 && (!m->indices || !m->values)))
    return sfail(h, SS_ERR_INVALID_ARG, "%s: bad host CSR", what);
  if (m->dim != h->dim) return sfail(h, SS_ERR_INVALID_ARG, "%s: dim mismatch", what);
  if (m->indptr[0] != 0 || m->indptr[m->n_rows] != m->nnz)
    return sfail(h, SS_ERR_OUT_OF_RANGE, "%s: indptr does not span [0, nnz]", what);
  // Under a device limit the pass copies row ranges of fewer than 2^31 nonzeros.
  if (h->host.device_limit == 0 && m->nnz >= ((int64_t)1 << 31))
    return sfail(h, SS_ERR_LIMIT, "%s: nnz too large", what);
  return SS_OK;
}

// Grows device buffer `role` of the pass to at least `bytes` (its contents
// are not kept).  The previous pass has finished: every call waits for its
// own work before returning, and drains the streams before starting.
ss_status ensure_buf(ss_handle *h, int role, size_t bytes) {
  ss_host_pass &hp = h->host;
  bytes = std::max<size_t>(bytes, 16);
  if (hp.cap[role] >= bytes) return SS_OK;
  cudaFree(hp.buf[role]);
  hp.buf[role] = nullptr;
  hp.cap[role] = 0;
  S_CUDA(dev_alloc(&hp.buf[role], bytes));
  hp.cap[role] = bytes;
  return SS_OK;
}

// indptr of a row range copied from the host, made to start at 0.
__global__ void k_rebase_indptr(int64_t *ptr, int64_t n, int64_t first) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    ptr[i] -= first;
}

// 16-bit values widened to float32 (both conversions are exact).
__global__ void k_widen_values(const uint16_t *__restrict__ src, float *__restrict__ dst, int64_t n,
                               int32_t type) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const uint16_t b = src[i];
    dst[i] = type == SS_VALUES_BF16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
  }
}

// Bytes the pass holds on the device for a row range of a CSR matrix: indptr
// (int64), indices and values (4 bytes each), inverse norms (float), and
// with 16-bit host values their 2-byte staging copy.
int64_t range_bytes(int64_t rows, int64_t nnz, bool half) {
  return 8 * (rows + 1) + (half ? 10 : 8) * nnz + 4 * rows;
}

// Copies rows [r0, r1) of the host CSR m into the buffers of roles
// base .. base + 2 (grown beforehand; 16-bit values through the staging
// buffer of role `stage`, then widened) on stream s, and describes the copy.
ss_status upload_rows(ss_handle *h, const ss_csr *m, int64_t r0, int64_t r1, int base, int stage,
                      cudaStream_t s, ss_csr *view) {
  ss_host_pass &hp = h->host;
  const int64_t n = r1 - r0, p0 = m->indptr[r0], nnz = m->indptr[r1] - p0;
  int64_t *ptr = static_cast<int64_t *>(hp.buf[base]);
  int32_t *idx = static_cast<int32_t *>(hp.buf[base + 1]);
  float *val = static_cast<float *>(hp.buf[base + 2]);
  S_CUDA(cudaMemcpyAsync(ptr, m->indptr + r0, sizeof(int64_t) * (size_t)(n + 1), cudaMemcpyHostToDevice, s));
  if (nnz > 0) {
    S_CUDA(cudaMemcpyAsync(idx, m->indices + p0, sizeof(int32_t) * (size_t)nnz, cudaMemcpyHostToDevice, s));
    if (hp.value_type == SS_VALUES_F32) {
      S_CUDA(cudaMemcpyAsync(val, m->values + p0, sizeof(float) * (size_t)nnz, cudaMemcpyHostToDevice, s));
    } else {
      uint16_t *half = static_cast<uint16_t *>(hp.buf[stage]);
      const uint16_t *src = reinterpret_cast<const uint16_t *>(m->values) + p0;
      S_CUDA(cudaMemcpyAsync(half, src, sizeof(uint16_t) * (size_t)nnz, cudaMemcpyHostToDevice, s));
      const int blocks = (int)std::min<int64_t>((nnz + 255) / 256, 8 * (int64_t)h->sm_count);
      k_widen_values<<<blocks, 256, 0, s>>>(half, val, nnz, hp.value_type);
      SS_CUDA_LAUNCH(cudaGetLastError());
    }
  }
  if (p0 != 0) {
    const int blocks = (int)std::min<int64_t>((n + 1 + 255) / 256, 4 * (int64_t)h->sm_count);
    k_rebase_indptr<<<blocks, 256, 0, s>>>(ptr, n + 1, p0);
    SS_CUDA_LAUNCH(cudaGetLastError());
  }
  *view = {ptr, idx, val, n, nnz, h->dim};
  return SS_OK;
}

// Largest row ranges from row 0 on whose device copy (range_bytes) stays
// within `cap`, with at most `max_rows` rows and fewer than 2^31 nonzeros;
// a range of `align` rows or more ends on a multiple of `align` rows after
// its start, the last one excepted.  bounds = {0, ..., n}.  False when one
// row alone does not fit.
bool split_rows(const int64_t *ptr, int64_t n, int64_t cap, int64_t max_rows, int64_t align, bool half,
                std::vector<int64_t> &bounds) {
  bounds.assign(1, 0);
  int64_t r0 = 0;
  auto fits = [&](int64_t r1) {
    const int64_t nnz = ptr[r1] - ptr[r0];
    return nnz < ((int64_t)1 << 31) && range_bytes(r1 - r0, nnz, half) <= cap;
  };
  while (r0 < n) {
    int64_t lo = r0, hi = std::min(n, r0 + max_rows);
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo + 1) / 2;
      if (fits(mid)) lo = mid;
      else hi = mid - 1;
    }
    if (lo == r0) return false;
    int64_t r1 = lo;
    if (r1 < n && r1 - r0 >= align) r1 = r0 + (r1 - r0) / align * align;
    bounds.push_back(r1);
    r0 = r1;
  }
  return true;
}

// The shape of a host pass under a device-memory limit: query tiles (row
// ranges of the queries, each scored against every item) and item batches
// (row ranges of the items, each copied to the device once).  Without a
// limit, or when everything fits it, one tile and one batch.  Otherwise the
// queries stay one tile if they and their output tiles take at most half the
// limit, else tiles of at most a quarter of it each, with output tiles of at
// most another quarter; the item batches share what is left in two slots
// (one being scored, the next being copied) and are whole multiples of the
// chunk when a chunk fits.  `why` says what did not fit.
ss_status plan_pass(const int64_t *qptr, int64_t n_q, const int64_t *iptr, int64_t n_i, int64_t C,
                    int64_t limit, bool direct, bool half, std::vector<int64_t> &qb, std::vector<int64_t> &ib,
                    std::string &why) {
  qb = {0, n_q};
  ib = {0, n_i};
  if (limit <= 0 || n_q == 0 || n_i == 0) return SS_OK;
  const int64_t W = std::min(C, n_i);
  auto out_bytes = [&](int64_t rows) { return direct ? (int64_t)0 : 2 * 4 * rows * W; };
  const int64_t nnz_q = qptr[n_q], nnz_i = iptr[n_i], big = (int64_t)1 << 31;
  const int64_t q_all = range_bytes(n_q, nnz_q, half) + out_bytes(n_q);
  if (nnz_q < big && nnz_i < big && q_all + range_bytes(n_i, nnz_i, half) <= limit) return SS_OK;
  int64_t q_used = q_all;
  if (nnz_q >= big || q_all > limit / 2) {
    const int64_t max_rows = direct ? n_q : (limit / 4) / (8 * W);
    if (max_rows < 1) {
      why = "the output tiles of one query row exceed a quarter of the device limit";
      return SS_ERR_LIMIT;
    }
    if (!split_rows(qptr, n_q, limit / 4, max_rows, 1, half, qb)) {
      why = "one query row exceeds a quarter of the device limit";
      return SS_ERR_LIMIT;
    }
    int64_t worst = 0, rows = 0;
    for (size_t t = 0; t + 1 < qb.size(); ++t) {
      worst = std::max(worst, range_bytes(qb[t + 1] - qb[t], qptr[qb[t + 1]] - qptr[qb[t]], half));
      rows = std::max(rows, qb[t + 1] - qb[t]);
    }
    q_used = worst + out_bytes(rows);
  }
  if (!split_rows(iptr, n_i, (limit - q_used) / 2, n_i, C, half, ib)) {
    why = "one item row exceeds half of what the query tiles leave of the device limit";
    return SS_ERR_LIMIT;
  }
  return SS_OK;
}

// Waits (with the deadline) until everything queued on the pass's streams has run.
ss_status drain(ss_handle *h, int32_t timeout_ms) {
  ss_host_pass &hp = h->host;
  for (cudaStream_t s : {hp.comp, hp.copy, hp.up}) {
    S_CUDA(cudaEventRecord(hp.finished, s));
    const ss_status st = wait_event(h, hp.finished, timeout_ms, "ss_bulk_cosine_host");
    if (st != SS_OK) return st;
  }
  return SS_OK;
}

ss_status ensure_sync_objects(ss_handle *h, int ring) {
  ss_host_pass &hp = h->host;
  if (!hp.comp) S_CUDA(cudaStreamCreateWithFlags(&hp.comp, cudaStreamNonBlocking));
  if (!hp.copy) S_CUDA(cudaStreamCreateWithFlags(&hp.copy, cudaStreamNonBlocking));
  if (!hp.up) S_CUDA(cudaStreamCreateWithFlags(&hp.up, cudaStreamNonBlocking));
  if (!hp.finished) S_CUDA(cudaEventCreateWithFlags(&hp.finished, cudaEventDisableTiming));
  for (int b = 0; b < 2; ++b) {
    if (!hp.done[b]) S_CUDA(cudaEventCreateWithFlags(&hp.done[b], cudaEventDisableTiming));
    if (!hp.out_free[b]) S_CUDA(cudaEventCreateWithFlags(&hp.out_free[b], cudaEventDisableTiming));
    if (!hp.batch_ready[b]) S_CUDA(cudaEventCreateWithFlags(&hp.batch_ready[b], cudaEventDisableTiming));
    if (!hp.batch_free[b]) S_CUDA(cudaEventCreateWithFlags(&hp.batch_free[b], cudaEventDisableTiming));
  }
  while ((int)hp.copied.size() < ring) {
    cudaEvent_t e = nullptr;
    S_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    hp.copied.push_back(e);
  }
  return SS_OK;
}

ss_status ensure_ring(ss_handle *h, int ring, size_t bytes) {
  ss_host_pass &hp = h->host;
  if (hp.slot_bytes < bytes) {
    for (float *p : hp.slots) cudaFreeHost(p);
    hp.slots.clear();
    hp.slot_bytes = bytes;
  }
  while ((int)hp.slots.size() < ring) {
    float *p = nullptr;
    S_CUDA(host_alloc(&p, hp.slot_bytes));
    hp.slots.push_back(p);
  }
  return SS_OK;
}

}  // namespace

void invalidate_queries(ss_handle *h) {
  for (int j = 0; j < 3; ++j) h->prep_src[j] = h->qd_src[j] = nullptr;
  for (int j = 0; j < 4; ++j) h->tcq_src[j] = nullptr;
  h->tcq_rows = h->tcq_nnz = h->prep_rows = h->prep_nnz = h->qd_rows = h->qd_nnz = -1;
  h->tcq_generation = h->qd_generation = h->prep_generation = ~0ull;
}

void free_host_pass(ss_host_pass &hp) {
  if (hp.comp) cudaStreamSynchronize(hp.comp);
  if (hp.copy) cudaStreamSynchronize(hp.copy);
  if (hp.up) cudaStreamSynchronize(hp.up);
  for (float *p : hp.slots) cudaFreeHost(p);
  hp.slots.clear();
  hp.slot_bytes = 0;
  for (cudaEvent_t e : hp.copied) cudaEventDestroy(e);
  hp.copied.clear();
  for (int b = 0; b < 2; ++b) {
    if (hp.done[b]) cudaEventDestroy(hp.done[b]);
    if (hp.out_free[b]) cudaEventDestroy(hp.out_free[b]);
    if (hp.batch_ready[b]) cudaEventDestroy(hp.batch_ready[b]);
    if (hp.batch_free[b]) cudaEventDestroy(hp.batch_free[b]);
    hp.done[b] = hp.out_free[b] = hp.batch_ready[b] = hp.batch_free[b] = nullptr;
  }
  if (hp.finished) cudaEventDestroy(hp.finished);
  hp.finished = nullptr;
  for (int r = 0; r < ss_host_pass::kBuffers; ++r) {
    cudaFree(hp.buf[r]);
    hp.buf[r] = nullptr;
    hp.cap[r] = 0;
  }
  cudaFree(hp.dev_sums);
  cudaFreeHost(hp.host_sums);
  hp.dev_sums = hp.host_sums = nullptr;
  hp.sums_slots = 0;
  if (hp.comp) cudaStreamDestroy(hp.comp);
  if (hp.copy) cudaStreamDestroy(hp.copy);
  if (hp.up) cudaStreamDestroy(hp.up);
  hp.comp = hp.copy = hp.up = nullptr;
}

extern "C" ss_status ss_set_device_limit(ss_handle *h, int64_t bytes) {
  if (!h || bytes < 0) return SS_ERR_INVALID_ARG;
  h->host.device_limit = bytes;
  return SS_OK;
}

extern "C" ss_status ss_set_host_values(ss_handle *h, int32_t value_type) {
  if (!h || (value_type != SS_VALUES_F32 && value_type != SS_VALUES_BF16 && value_type != SS_VALUES_F16))
    return SS_ERR_INVALID_ARG;
  h->host.value_type = value_type;
  return SS_OK;
}

extern "C" ss_status ss_plan_host_pass(const int64_t *q_indptr, int64_t n_q, const int64_t *i_indptr,
                                       int64_t n_i, int32_t chunk_rows, int64_t device_limit,
                                       int32_t direct_output, int32_t value_type, int64_t *q_bounds,
                                       int64_t q_cap, int64_t *n_q_tiles, int64_t *i_bounds, int64_t i_cap,
                                       int64_t *n_i_batches) {
  if (!q_indptr || !i_indptr || n_q < 0 || n_i < 0 || chunk_rows < 1 || device_limit < 0 ||
      !n_q_tiles || !n_i_batches ||
      (value_type != SS_VALUES_F32 && value_type != SS_VALUES_BF16 && value_type != SS_VALUES_F16))
    return SS_ERR_INVALID_ARG;
  std::vector<int64_t> qb, ib;
  std::string why;
  const ss_status st = plan_pass(q_indptr, n_q, i_indptr, n_i, chunk_rows, device_limit, direct_output != 0,
                                 value_type != SS_VALUES_F32, qb, ib, why);
  if (st != SS_OK) return st;
  *n_q_tiles = (int64_t)qb.size() - 1;
  *n_i_batches = (int64_t)ib.size() - 1;
  if ((q_bounds && q_cap < (int64_t)qb.size()) || (i_bounds && i_cap < (int64_t)ib.size()))
    return SS_ERR_INVALID_ARG;
  if (q_bounds) std::copy(qb.begin(), qb.end(), q_bounds);
  if (i_bounds) std::copy(ib.begin(), ib.end(), i_bounds);
  return SS_OK;
}

extern "C" ss_status ss_bulk_cosine_host(ss_handle *h, const ss_csr *qh, const ss_csr *ih,
                                         float *out_host, int64_t ld_out,
                                         ss_chunk_consumer consumer, void *user,
                                         int32_t ring_depth, int32_t timeout_ms) {
  if (!h) return SS_ERR_INVALID_ARG;
  ss_status st = check_host_csr(h, qh, "ss_bulk_cosine_host queries");
  if (st == SS_OK) st = check_host_csr(h, ih, "ss_bulk_cosine_host items");
  if (st != SS_OK) return st;
  if (!out_host && !consumer)
    return sfail(h, SS_ERR_INVALID_ARG, "ss_bulk_cosine_host: no output and no consumer");
  if (out_host && ld_out < ih->n_rows)
    return sfail(h, SS_ERR_INVALID_ARG, "ss_bulk_cosine_host: ld_out < number of items");
  if (ring_depth < 2) return sfail(h, SS_ERR_INVALID_ARG, "ss_bulk_cosine_host: ring_depth < 2");
  if (timeout_ms <= 0) timeout_ms = 60000;
  const int64_t n_q = qh->n_rows, n_i = ih->n_rows, C = h->chunk_rows;
  if (n_q == 0 || n_i == 0) return SS_OK;
  S_CUDA(cudaSetDevice(h->device));
  const int R = ring_depth;
  if ((st = ensure_sync_objects(h, R)) != SS_OK) return st;
  if ((st = drain(h, timeout_ms)) != SS_OK) return st;
  ss_host_pass &hp = h->host;

  // Direct stores when the caller's output is page-locked, the device can
  // address it, and nobody else needs the tile; otherwise the ring.
  const bool verify = (h->flags & SS_VERIFY_STREAM) != 0;
  hp.log_bits.clear();
  hp.log_values.clear();
  float *out_dev = nullptr;
  if (out_host && !consumer && !verify) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, out_host) == cudaSuccess && attr.type == cudaMemoryTypeHost &&
        attr.devicePointer)
      out_dev = static_cast<float *>(attr.devicePointer);
    cudaGetLastError();
  }

  // Query tiles x item batches (one of each unless the device limit says otherwise).
  const bool half = hp.value_type != SS_VALUES_F32;
  std::vector<int64_t> qb, ib;
  {
    std::string why;
    st = plan_pass(qh->indptr, n_q, ih->indptr, n_i, C, hp.device_limit, out_dev != nullptr, half, qb, ib, why);
    if (st != SS_OK)
      return sfail(h, st, "ss_bulk_cosine_host: device limit of %lld bytes: %s", (long long)hp.device_limit,
                   why.c_str());
  }
  const int64_t n_tiles = (int64_t)qb.size() - 1, n_batches = (int64_t)ib.size() - 1;
  if (consumer && n_tiles > 1)
    return sfail(h, SS_ERR_LIMIT,
                 "ss_bulk_cosine_host: the device limit splits the queries into %lld tiles; a consumer "
                 "receives whole columns of the result, so pass out_host instead",
                 (long long)n_tiles);

  // Buffers at their largest size over the tiles and batches, allocated
  // before anything is queued (growing one later would synchronise).
  using HP = ss_host_pass;
  auto grow_for = [&](const ss_csr *m, const std::vector<int64_t> &bnd, int base, int inv, int stage) -> ss_status {
    int64_t rows = 0, nnz = 0;
    for (size_t t = 0; t + 1 < bnd.size(); ++t) {
      rows = std::max(rows, bnd[t + 1] - bnd[t]);
      nnz = std::max(nnz, m->indptr[bnd[t + 1]] - m->indptr[bnd[t]]);
    }
    ss_status s2 = ensure_buf(h, base, sizeof(int64_t) * (size_t)(rows + 1));
    if (s2 == SS_OK) s2 = ensure_buf(h, base + 1, sizeof(int32_t) * (size_t)nnz);
    if (s2 == SS_OK) s2 = ensure_buf(h, base + 2, sizeof(float) * (size_t)nnz);
    if (s2 == SS_OK) s2 = ensure_buf(h, inv, sizeof(float) * (size_t)rows);
    if (s2 == SS_OK && half) s2 = ensure_buf(h, stage, sizeof(uint16_t) * (size_t)nnz);
    return s2;
  };
  if ((st = grow_for(qh, qb, HP::kQPtr, HP::kInvQ, HP::kQHalf)) != SS_OK) return st;
  for (int s = 0; s < (n_batches > 1 ? 2 : 1); ++s)
    if ((st = grow_for(ih, ib, HP::kIPtr0 + s * HP::kSlotRoles, HP::kInvI0 + s * HP::kSlotRoles,
                       HP::kIHalf0 + s)) != SS_OK)
      return st;
  int64_t tile_rows = 0;
  for (int64_t t = 0; t < n_tiles; ++t) tile_rows = std::max(tile_rows, qb[t + 1] - qb[t]);
  const int64_t width_max = std::min<int64_t>(C, n_i);
  float *dbuf[2] = {nullptr, nullptr};
  if (!out_dev) {
    const size_t tile_bytes = sizeof(float) * (size_t)(tile_rows * width_max);
    if ((st = ensure_buf(h, HP::kOut0, tile_bytes)) != SS_OK) return st;
    if ((st = ensure_buf(h, HP::kOut1, tile_bytes)) != SS_OK) return st;
    if ((st = ensure_ring(h, R, tile_bytes)) != SS_OK) return st;
    dbuf[0] = static_cast<float *>(hp.buf[HP::kOut0]);
    dbuf[1] = static_cast<float *>(hp.buf[HP::kOut1]);
    if (verify && hp.sums_slots < R) {
      cudaFree(hp.dev_sums);
      cudaFreeHost(hp.host_sums);
      hp.dev_sums = hp.host_sums = nullptr;
      hp.sums_slots = 0;
      S_CUDA(dev_alloc(&hp.dev_sums, 16 * (size_t)R));
      S_CUDA(host_alloc(&hp.host_sums, 16 * (size_t)R));
      hp.sums_slots = R;
    }
  }
  // Slot r of the checksum buffers: {bits_sum (u64), value_sum (double)}.
  auto dev_sum_slot = [&](int64_t u) { return static_cast<unsigned char *>(hp.dev_sums) + 16 * (u % R); };
  auto host_sum_slot = [&](int64_t u) { return static_cast<unsigned char *>(hp.host_sums) + 16 * (u % R); };
  void *vs = reinterpret_cast<void *>(hp.comp);
  float *inv_q = static_cast<float *>(hp.buf[HP::kInvQ]);

  // A unit is one chunk of items scored against one query tile; through the
  // ring, unit u uses device buffer u % 2 and ring slot u % R.
  struct Unit {
    int64_t chunk, rb, re, q0, q1;
  };
  std::vector<Unit> units;
  int64_t delivered = 0;
  auto deliver = [&](int64_t u) -> ss_status {
    const Unit &un = units[(size_t)u];
    const int64_t w = un.re - un.rb, rows = un.q1 - un.q0;
    ss_status s2 = wait_event(h, hp.copied[u % R], timeout_ms, "ss_bulk_cosine_host copy");
    if (s2 != SS_OK) return s2;
    const float *slot = hp.slots[u % R];
    if (verify) {
      uint64_t hb = 0, db = 0;
      double hv = 0.0;
      tile_checksum_host(slot, rows, w, w, &hb, &hv);
      memcpy(&db, host_sum_slot(u), sizeof(db));
      if (hb != db)
        return sfail(h, SS_ERR_DEVICE_CHECK,
                     "ss_bulk_cosine_host: chunk %lld (query rows %lld..%lld) checksum differs between device "
                     "(%llu) and host copy (%llu)",
                     (long long)un.chunk, (long long)un.q0, (long long)un.q1, (unsigned long long)db,
                     (unsigned long long)hb);
      hp.log_bits.push_back(hb);
      hp.log_values.push_back(hv);
    }
    if (out_host) scatter_rows(out_host + un.q0 * ld_out, ld_out, un.rb, slot, w, w, rows);
    if (consumer && consumer(user, un.chunk, un.rb, un.re, slot, w, rows) != 0)
      return sfail(h, SS_ERR_INVALID_ARG, "ss_bulk_cosine_host: consumer stopped the pass");
    return SS_OK;
  };
  // Scores one chunk index against the current query tile.
  auto score = [&](const Unit &un, const ss_csr &qv, const ss_index *idx, const float *inv_i_chunk) -> ss_status {
    ss_status s2;
    if (out_dev) return ss_score_chunk(h, &qv, inv_q, idx, inv_i_chunk, out_dev + un.q0 * ld_out + un.rb, ld_out, vs);
    const int64_t u = (int64_t)units.size(), w = un.re - un.rb, rows = un.q1 - un.q0;
    units.push_back(un);
    const int b = (int)(u & 1);
    if (u >= 2) S_CUDA(cudaStreamWaitEvent(hp.comp, hp.out_free[b], 0));
    if ((s2 = ss_score_chunk(h, &qv, inv_q, idx, inv_i_chunk, dbuf[b], w, vs)) != SS_OK) return s2;
    if (verify) {
      // The checksum slot of unit u - R was copied out before this unit's
      // buffer became free (same copy stream, earlier).
      S_CUDA(cudaMemsetAsync(dev_sum_slot(u), 0, 16, hp.comp));
      unsigned char *ds = dev_sum_slot(u);
      SS_CUDA_LAUNCH(launch_tile_checksum(dbuf[b], rows, w, w, reinterpret_cast<uint64_t *>(ds),
                                          reinterpret_cast<double *>(ds + 8), h->sm_count, hp.comp));
    }
    S_CUDA(cudaEventRecord(hp.done[b], hp.comp));
    S_CUDA(cudaStreamWaitEvent(hp.copy, hp.done[b], 0));
    // Slot u % R was last used by unit u - R, delivered before this point.
    S_CUDA(cudaMemcpyAsync(hp.slots[u % R], dbuf[b], sizeof(float) * (size_t)(rows * w),
                           cudaMemcpyDeviceToHost, hp.copy));
    if (verify)
      S_CUDA(cudaMemcpyAsync(host_sum_slot(u), dev_sum_slot(u), 16, cudaMemcpyDeviceToHost, hp.copy));
    S_CUDA(cudaEventRecord(hp.copied[u % R], hp.copy));
    S_CUDA(cudaEventRecord(hp.out_free[b], hp.copy));
    // Keep R - 1 units in flight; deliver the oldest.
    while (delivered <= u - (R - 1)) {
      if ((s2 = deliver(delivered)) != SS_OK) return s2;
      ++delivered;
    }
    return SS_OK;
  };

  // Item batch k goes to slot k % 2 on the upload stream, once the slot's
  // previous batch (k - 2) has been scored.
  ss_csr iv[2];
  auto upload_batch = [&](int64_t k) -> ss_status {
    const int s = (int)(k & 1);
    if (k >= 2) S_CUDA(cudaStreamWaitEvent(hp.up, hp.batch_free[s], 0));
    ss_status s2 = upload_rows(h, ih, ib[k], ib[k + 1], HP::kIPtr0 + s * HP::kSlotRoles, HP::kIHalf0 + s, hp.up,
                               &iv[s]);
    if (s2 != SS_OK) return s2;
    S_CUDA(cudaEventRecord(hp.batch_ready[s], hp.up));
    return SS_OK;
  };
  if ((st = upload_batch(0)) != SS_OK) return st;
  const int64_t span = C * h->build_batch;
  ss_index *views[kMaxBuildBatch];
  int32_t n_views = 0;
  int64_t chunk = 0;
  ss_csr qv{};
  for (int64_t k = 0; k < n_batches; ++k) {
    const int s = (int)(k & 1);
    if (k + 1 < n_batches && (st = upload_batch(k + 1)) != SS_OK) return st;
    S_CUDA(cudaStreamWaitEvent(hp.comp, hp.batch_ready[s], 0));
    // The pass's buffers hold new contents at addresses the handle may have
    // prepared other matrices from.
    ss_invalidate(h);
    float *inv_i = static_cast<float *>(hp.buf[HP::kInvI0 + s * HP::kSlotRoles]);
    if ((st = ss_row_norms(h, &iv[s], inv_i, vs)) != SS_OK) return st;
    const int64_t nb = ib[k + 1] - ib[k], chunk0 = chunk;
    for (int64_t t = 0; t < n_tiles; ++t) {
      if (k == 0 || n_tiles > 1) {
        // The tile's buffers were last read by scoring calls queued earlier on comp.
        if ((st = upload_rows(h, qh, qb[t], qb[t + 1], HP::kQPtr, HP::kQHalf, hp.comp, &qv)) != SS_OK) return st;
        invalidate_queries(h);
        if ((st = ss_row_norms(h, &qv, inv_q, vs)) != SS_OK) return st;
      }
      chunk = chunk0;
      for (int64_t g0 = 0; g0 < nb; g0 += span) {
        if ((st = ss_build_item_indexes(h, &iv[s], g0, std::min(g0 + span, nb), views, &n_views, vs)) != SS_OK)
          return st;
        for (int v = 0; v < n_views; ++v) {
          const int64_t r0 = views[v]->row_begin, r1 = views[v]->row_end;
          const Unit un = {chunk++, ib[k] + r0, ib[k] + r1, qb[t], qb[t + 1]};
          if ((st = score(un, qv, views[v], inv_i + r0)) != SS_OK) return st;
        }
      }
    }
    S_CUDA(cudaEventRecord(hp.batch_free[s], hp.comp));
  }
  while (delivered < (int64_t)units.size()) {
    if ((st = deliver(delivered)) != SS_OK) return st;
    ++delivered;
  }
  if ((st = drain(h, timeout_ms)) != SS_OK) return st;
  return ss_check_device(h, vs);
}
