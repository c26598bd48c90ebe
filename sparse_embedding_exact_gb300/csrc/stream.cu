// Host-buffer streaming pass: the "streaming batch" pipeline of the blog post
// ("Engineering practice for bulk similarity calculation over sparse
// embeddings", sections 2.2 and 4.4): items are scored chunk by chunk and each
// chunk's slice of the result goes back to host memory while the next chunk
// is computed.
//
// Two device output buffers alternate between chunks.  The compute stream
// builds the index and scores chunk c into buffer c % 2; the copy stream
// waits for that, then copies the buffer to the host: straight into the
// caller's output when that is page-locked, otherwise into slot c % R of a
// ring of page-locked buffers, from which the host thread copies rows out or
// hands the tile to the caller's consumer.  Events order buffer and slot
// reuse; every host wait polls its event with a deadline.
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

// Everything the pass allocates; the destructor drains the streams and frees.
struct Pass {
  cudaStream_t comp = nullptr, copy = nullptr;
  int64_t *q_indptr = nullptr, *i_indptr = nullptr;
  int32_t *q_idx = nullptr, *i_idx = nullptr;
  float *q_val = nullptr, *i_val = nullptr, *inv_q = nullptr, *inv_i = nullptr;
  float *dbuf[2] = {nullptr, nullptr};
  std::vector<float *> slots;
  cudaEvent_t done[2] = {nullptr, nullptr}, dbuf_free[2] = {nullptr, nullptr};
  std::vector<cudaEvent_t> copied;
  ~Pass() {
    if (comp) cudaStreamSynchronize(comp);
    if (copy) cudaStreamSynchronize(copy);
    for (float *p : slots) cudaFreeHost(p);
    for (cudaEvent_t e : copied) cudaEventDestroy(e);
    for (int b = 0; b < 2; ++b) {
      if (done[b]) cudaEventDestroy(done[b]);
      if (dbuf_free[b]) cudaEventDestroy(dbuf_free[b]);
      cudaFree(dbuf[b]);
    }
    cudaFree(q_indptr); cudaFree(i_indptr); cudaFree(q_idx); cudaFree(i_idx);
    cudaFree(q_val); cudaFree(i_val); cudaFree(inv_q); cudaFree(inv_i);
    if (comp) cudaStreamDestroy(comp);
    if (copy) cudaStreamDestroy(copy);
  }
};

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

template <typename T>
ss_status upload(ss_handle *h, T **dst, const T *src, int64_t n, cudaStream_t s) {
  S_CUDA(cudaMalloc(dst, sizeof(T) * (size_t)std::max<int64_t>(n, 1)));
  if (n > 0) S_CUDA(cudaMemcpyAsync(*dst, src, sizeof(T) * (size_t)n, cudaMemcpyHostToDevice, s));
  return SS_OK;
}

}  // namespace

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

  Pass p;
  S_CUDA(cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking));
  S_CUDA(cudaStreamCreateWithFlags(&p.copy, cudaStreamNonBlocking));
  if ((st = upload(h, &p.q_indptr, qh->indptr, n_q + 1, p.comp)) != SS_OK) return st;
  if ((st = upload(h, &p.q_idx, qh->indices, qh->nnz, p.comp)) != SS_OK) return st;
  if ((st = upload(h, &p.q_val, qh->values, qh->nnz, p.comp)) != SS_OK) return st;
  if ((st = upload(h, &p.i_indptr, ih->indptr, n_i + 1, p.comp)) != SS_OK) return st;
  if ((st = upload(h, &p.i_idx, ih->indices, ih->nnz, p.comp)) != SS_OK) return st;
  if ((st = upload(h, &p.i_val, ih->values, ih->nnz, p.comp)) != SS_OK) return st;
  S_CUDA(cudaMalloc(&p.inv_q, sizeof(float) * (size_t)n_q));
  S_CUDA(cudaMalloc(&p.inv_i, sizeof(float) * (size_t)n_i));
  const ss_csr qd = {p.q_indptr, p.q_idx, p.q_val, n_q, qh->nnz, h->dim};
  const ss_csr id = {p.i_indptr, p.i_idx, p.i_val, n_i, ih->nnz, h->dim};
  void *vs = reinterpret_cast<void *>(p.comp);
  if ((st = ss_row_norms(h, &qd, p.inv_q, vs)) != SS_OK) return st;
  if ((st = ss_row_norms(h, &id, p.inv_i, vs)) != SS_OK) return st;

  // Direct copies when the caller's output is page-locked and nobody else
  // needs the tile; otherwise go through the pinned ring.
  bool direct = false;
  if (out_host && !consumer) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, out_host) == cudaSuccess && attr.type == cudaMemoryTypeHost)
      direct = true;
    cudaGetLastError();
  }
  const int64_t width_max = std::min<int64_t>(C, n_i);
  const int R = ring_depth;
  for (int b = 0; b < 2; ++b) {
    S_CUDA(cudaMalloc(&p.dbuf[b], sizeof(float) * (size_t)(n_q * width_max)));
    S_CUDA(cudaEventCreateWithFlags(&p.done[b], cudaEventDisableTiming));
    S_CUDA(cudaEventCreateWithFlags(&p.dbuf_free[b], cudaEventDisableTiming));
  }
  p.copied.assign(R, nullptr);
  for (int r = 0; r < R; ++r) S_CUDA(cudaEventCreateWithFlags(&p.copied[r], cudaEventDisableTiming));
  if (!direct) {
    p.slots.assign(R, nullptr);
    for (int r = 0; r < R; ++r)
      S_CUDA(cudaHostAlloc(&p.slots[r], sizeof(float) * (size_t)(n_q * width_max), cudaHostAllocDefault));
  }

  const int64_t n_chunks = (n_i + C - 1) / C;
  int64_t delivered = 0;
  auto deliver = [&](int64_t c) -> ss_status {
    const int64_t rb = c * C, re = std::min(rb + C, n_i), w = re - rb;
    ss_status s2 = wait_event(h, p.copied[c % R], timeout_ms, "ss_bulk_cosine_host copy");
    if (s2 != SS_OK) return s2;
    if (!direct) {
      const float *slot = p.slots[c % R];
      if (out_host) scatter_rows(out_host, ld_out, rb, slot, w, w, n_q);
      if (consumer && consumer(user, c, rb, re, slot, w, n_q) != 0)
        return sfail(h, SS_ERR_INVALID_ARG, "ss_bulk_cosine_host: consumer stopped the pass");
    }
    return SS_OK;
  };

  for (int64_t c = 0; c < n_chunks; ++c) {
    const int b = (int)(c & 1);
    const int64_t rb = c * C, re = std::min(rb + C, n_i), w = re - rb;
    if (c >= 2) S_CUDA(cudaStreamWaitEvent(p.comp, p.dbuf_free[b], 0));
    ss_index *idx = nullptr;
    if ((st = ss_build_item_index(h, &id, rb, re, &idx, vs)) != SS_OK) return st;
    if ((st = ss_score_chunk(h, &qd, p.inv_q, idx, p.inv_i + rb, p.dbuf[b], w, vs)) != SS_OK)
      return st;
    S_CUDA(cudaEventRecord(p.done[b], p.comp));
    S_CUDA(cudaStreamWaitEvent(p.copy, p.done[b], 0));
    // Slot c % R was last used by chunk c - R, delivered before this point.
    float *dst = direct ? out_host + rb : p.slots[c % R];
    const int64_t dld = direct ? ld_out : w;
    S_CUDA(cudaMemcpy2DAsync(dst, sizeof(float) * (size_t)dld, p.dbuf[b], sizeof(float) * (size_t)w,
                             sizeof(float) * (size_t)w, (size_t)n_q, cudaMemcpyDeviceToHost, p.copy));
    S_CUDA(cudaEventRecord(p.copied[c % R], p.copy));
    S_CUDA(cudaEventRecord(p.dbuf_free[b], p.copy));
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
