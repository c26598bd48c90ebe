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
  if (m->nnz >= ((int64_t)1 << 31)) return sfail(h, SS_ERR_LIMIT, "%s: nnz too large", what);
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
  S_CUDA(cudaMalloc(&hp.buf[role], bytes));
  hp.cap[role] = bytes;
  return SS_OK;
}

template <typename T>
ss_status upload(ss_handle *h, int role, const T *src, int64_t n) {
  ss_status st = ensure_buf(h, role, sizeof(T) * (size_t)n);
  if (st != SS_OK) return st;
  if (n > 0)
    S_CUDA(cudaMemcpyAsync(h->host.buf[role], src, sizeof(T) * (size_t)n, cudaMemcpyHostToDevice,
                           h->host.comp));
  return SS_OK;
}

// Waits (with the deadline) until everything queued on the pass's streams has run.
ss_status drain(ss_handle *h, int32_t timeout_ms) {
  ss_host_pass &hp = h->host;
  for (cudaStream_t s : {hp.comp, hp.copy}) {
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
  if (!hp.finished) S_CUDA(cudaEventCreateWithFlags(&hp.finished, cudaEventDisableTiming));
  for (int b = 0; b < 2; ++b) {
    if (!hp.done[b]) S_CUDA(cudaEventCreateWithFlags(&hp.done[b], cudaEventDisableTiming));
    if (!hp.out_free[b]) S_CUDA(cudaEventCreateWithFlags(&hp.out_free[b], cudaEventDisableTiming));
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
    S_CUDA(cudaHostAlloc(&p, hp.slot_bytes, cudaHostAllocDefault));
    hp.slots.push_back(p);
  }
  return SS_OK;
}

}  // namespace

void free_host_pass(ss_host_pass &hp) {
  if (hp.comp) cudaStreamSynchronize(hp.comp);
  if (hp.copy) cudaStreamSynchronize(hp.copy);
  for (float *p : hp.slots) cudaFreeHost(p);
  hp.slots.clear();
  hp.slot_bytes = 0;
  for (cudaEvent_t e : hp.copied) cudaEventDestroy(e);
  hp.copied.clear();
  for (int b = 0; b < 2; ++b) {
    if (hp.done[b]) cudaEventDestroy(hp.done[b]);
    if (hp.out_free[b]) cudaEventDestroy(hp.out_free[b]);
    hp.done[b] = hp.out_free[b] = nullptr;
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
  hp.comp = hp.copy = nullptr;
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

  using HP = ss_host_pass;
  if ((st = upload(h, HP::kQPtr, qh->indptr, n_q + 1)) != SS_OK) return st;
  if ((st = upload(h, HP::kQIdx, qh->indices, qh->nnz)) != SS_OK) return st;
  if ((st = upload(h, HP::kQVal, qh->values, qh->nnz)) != SS_OK) return st;
  if ((st = upload(h, HP::kIPtr, ih->indptr, n_i + 1)) != SS_OK) return st;
  if ((st = upload(h, HP::kIIdx, ih->indices, ih->nnz)) != SS_OK) return st;
  if ((st = upload(h, HP::kIVal, ih->values, ih->nnz)) != SS_OK) return st;
  if ((st = ensure_buf(h, HP::kInvQ, sizeof(float) * (size_t)n_q)) != SS_OK) return st;
  if ((st = ensure_buf(h, HP::kInvI, sizeof(float) * (size_t)n_i)) != SS_OK) return st;
  float *inv_q = static_cast<float *>(hp.buf[HP::kInvQ]);
  float *inv_i = static_cast<float *>(hp.buf[HP::kInvI]);
  const ss_csr qd = {static_cast<const int64_t *>(hp.buf[HP::kQPtr]),
                     static_cast<const int32_t *>(hp.buf[HP::kQIdx]),
                     static_cast<const float *>(hp.buf[HP::kQVal]), n_q, qh->nnz, h->dim};
  const ss_csr id = {static_cast<const int64_t *>(hp.buf[HP::kIPtr]),
                     static_cast<const int32_t *>(hp.buf[HP::kIIdx]),
                     static_cast<const float *>(hp.buf[HP::kIVal]), n_i, ih->nnz, h->dim};
  void *vs = reinterpret_cast<void *>(hp.comp);
  // The device copies above reuse the pass's buffers: whatever the handle
  // prepared from an earlier pass's matrices at these addresses is stale.
  ss_invalidate(h);
  if ((st = ss_row_norms(h, &qd, inv_q, vs)) != SS_OK) return st;
  if ((st = ss_row_norms(h, &id, inv_i, vs)) != SS_OK) return st;
  const int64_t n_chunks = (n_i + C - 1) / C;

  // The chunks' indexes are built h->build_batch at a time (one launch).
  const int64_t span = C * h->build_batch;
  ss_index *views[kMaxBuildBatch];
  int32_t n_views = 0;
  if (out_dev) {
    for (int64_t bb = 0; bb < n_i; bb += span) {
      if ((st = ss_build_item_indexes(h, &id, bb, std::min(bb + span, n_i), views, &n_views, vs)) != SS_OK)
        return st;
      for (int k = 0; k < n_views; ++k) {
        const int64_t rb = views[k]->row_begin;
        if ((st = ss_score_chunk(h, &qd, inv_q, views[k], inv_i + rb, out_dev + rb, ld_out, vs)) != SS_OK)
          return st;
      }
    }
    if ((st = drain(h, timeout_ms)) != SS_OK) return st;
    return ss_check_device(h, vs);
  }

  const int64_t width_max = std::min<int64_t>(C, n_i);
  const size_t tile_bytes = sizeof(float) * (size_t)(n_q * width_max);
  if ((st = ensure_buf(h, HP::kOut0, tile_bytes)) != SS_OK) return st;
  if ((st = ensure_buf(h, HP::kOut1, tile_bytes)) != SS_OK) return st;
  if ((st = ensure_ring(h, R, tile_bytes)) != SS_OK) return st;
  float *dbuf[2] = {static_cast<float *>(hp.buf[HP::kOut0]), static_cast<float *>(hp.buf[HP::kOut1])};
  if (verify && hp.sums_slots < R) {
    cudaFree(hp.dev_sums);
    cudaFreeHost(hp.host_sums);
    hp.dev_sums = hp.host_sums = nullptr;
    hp.sums_slots = 0;
    S_CUDA(cudaMalloc(&hp.dev_sums, 16 * (size_t)R));
    S_CUDA(cudaHostAlloc(&hp.host_sums, 16 * (size_t)R, cudaHostAllocDefault));
    hp.sums_slots = R;
  }
  // Slot r of the checksum buffers: {bits_sum (u64), value_sum (double)}.
  auto dev_sum_slot = [&](int64_t c) { return static_cast<unsigned char *>(hp.dev_sums) + 16 * (c % R); };
  auto host_sum_slot = [&](int64_t c) { return static_cast<unsigned char *>(hp.host_sums) + 16 * (c % R); };

  int64_t delivered = 0;
  auto deliver = [&](int64_t c) -> ss_status {
    const int64_t rb = c * C, re = std::min(rb + C, n_i), w = re - rb;
    ss_status s2 = wait_event(h, hp.copied[c % R], timeout_ms, "ss_bulk_cosine_host copy");
    if (s2 != SS_OK) return s2;
    const float *slot = hp.slots[c % R];
    if (verify) {
      uint64_t hb = 0, db = 0;
      double hv = 0.0;
      tile_checksum_host(slot, n_q, w, w, &hb, &hv);
      memcpy(&db, host_sum_slot(c), sizeof(db));
      if (hb != db)
        return sfail(h, SS_ERR_DEVICE_CHECK,
                     "ss_bulk_cosine_host: chunk %lld checksum differs between device (%llu) and host copy (%llu)",
                     (long long)c, (unsigned long long)db, (unsigned long long)hb);
      hp.log_bits.push_back(hb);
      hp.log_values.push_back(hv);
    }
    if (out_host) scatter_rows(out_host, ld_out, rb, slot, w, w, n_q);
    if (consumer && consumer(user, c, rb, re, slot, w, n_q) != 0)
      return sfail(h, SS_ERR_INVALID_ARG, "ss_bulk_cosine_host: consumer stopped the pass");
    return SS_OK;
  };

  for (int64_t c = 0; c < n_chunks; ++c) {
    const int b = (int)(c & 1);
    const int64_t rb = c * C, re = std::min(rb + C, n_i), w = re - rb;
    if (rb % span == 0) {  // first chunk of a build batch
      if ((st = ss_build_item_indexes(h, &id, rb, std::min(rb + span, n_i), views, &n_views, vs)) != SS_OK)
        return st;
    }
    if (c >= 2) S_CUDA(cudaStreamWaitEvent(hp.comp, hp.out_free[b], 0));
    ss_index *idx = views[(rb % span) / C];
    if ((st = ss_score_chunk(h, &qd, inv_q, idx, inv_i + rb, dbuf[b], w, vs)) != SS_OK) return st;
    if (verify) {
      // The checksum slot of chunk c - R was copied out before this chunk's
      // buffer became free (same copy stream, earlier).
      S_CUDA(cudaMemsetAsync(dev_sum_slot(c), 0, 16, hp.comp));
      unsigned char *ds = dev_sum_slot(c);
      SS_CUDA_LAUNCH(launch_tile_checksum(dbuf[b], n_q, w, w, reinterpret_cast<uint64_t *>(ds),
                                          reinterpret_cast<double *>(ds + 8), h->sm_count, hp.comp));
    }
    S_CUDA(cudaEventRecord(hp.done[b], hp.comp));
    S_CUDA(cudaStreamWaitEvent(hp.copy, hp.done[b], 0));
    // Slot c % R was last used by chunk c - R, delivered before this point.
    S_CUDA(cudaMemcpyAsync(hp.slots[c % R], dbuf[b], sizeof(float) * (size_t)(n_q * w),
                           cudaMemcpyDeviceToHost, hp.copy));
    if (verify)
      S_CUDA(cudaMemcpyAsync(host_sum_slot(c), dev_sum_slot(c), 16, cudaMemcpyDeviceToHost, hp.copy));
    S_CUDA(cudaEventRecord(hp.copied[c % R], hp.copy));
    S_CUDA(cudaEventRecord(hp.out_free[b], hp.copy));
    // Keep R - 1 chunks in flight; deliver the oldest.
    while (delivered <= c - (R - 1)) {
      if ((st = deliver(delivered)) != SS_OK) return st;
      ++delivered;
    }
  }
  while (delivered < n_chunks) {
    if ((st = deliver(delivered)) != SS_OK) return st;
    ++delivered;
  }
  return ss_check_device(h, vs);
}
