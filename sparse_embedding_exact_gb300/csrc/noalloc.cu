// An entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running inside a host that owns
// all device memory through its own pool (a serving runtime or a framework
// allocator that forbids foreign allocations), code called while a CUDA
// graph is being captured where allocation is not allowed, or plug-ins whose
// memory budget is fixed up front.  ss_cosine_chunk_noalloc serves them: it
// scores one item chunk against all queries with the posting-list kernels
// and takes every byte of scratch from one file-scope device array of fixed
// size, so it never allocates.  The caller still provides the inputs and the
// output.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.cuh"

namespace {

// The scratch array: SS_NOALLOC_SCRATCH_BYTES on every GPU that loads the
// library, held until the process exits.  Every call shares it.
__device__ __align__(256) unsigned char g_noalloc_scratch[SS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// Device address of the scratch array on `device` (which must be current),
// looked up once per device and kept for the life of the process.  In host
// code the array's name is only a stand-in for the symbol, never an address
// a kernel may use.  The address kept is the one of the context current at
// the first call (the device's primary context, as the runtime uses); after
// cudaDeviceReset, or from another context on the same device, it is stale.
ss_status scratch_for_device(int device, void **addr, int *sm_count) {
  if (device < 0 || device >= kMaxDevices) return SS_ERR_LIMIT;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[device]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SS_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
      return SS_ERR_CUDA;
    g_scratch_addr[device] = p;
    g_sm_count[device] = sms;
  }
  *addr = g_scratch_addr[device];
  *sm_count = g_sm_count[device];
  return SS_OK;
}

bool csr_ok(const ss_csr *m) {
  return m && m->indptr && m->n_rows >= 0 && m->nnz >= 0 && m->dim > 0 &&
         (m->nnz == 0 || (m->indices && m->values));
}

}  // namespace

extern "C" ss_status ss_cosine_chunk_noalloc(const ss_csr *queries, const ss_csr *items,
                                             int64_t row_begin, int64_t row_end,
                                             int64_t chunk_nnz, float *out, int64_t ld_out,
                                             int32_t *device_status, void *stream) {
  if (!csr_ok(queries) || !csr_ok(items) || queries->dim != items->dim) return SS_ERR_INVALID_ARG;
  if (row_begin < 0 || row_end <= row_begin || row_end > items->n_rows) return SS_ERR_INVALID_ARG;
  if (chunk_nnz < 0 || chunk_nnz > items->nnz) return SS_ERR_INVALID_ARG;
  const int64_t width = row_end - row_begin;
  if (ld_out < width || (queries->n_rows > 0 && !out)) return SS_ERR_INVALID_ARG;
  if (width > SS_MAX_CHUNK_ROWS || items->dim >= ((int64_t)1 << 31) - 1) return SS_ERR_LIMIT;

  // Carve the scratch: status word, two norm vectors, the per-dimension
  // counters and list offsets, the scan's tile sums, the posting lists.
  const int64_t dim = items->dim;
  const int64_t tiles = scan_tile_count(dim + 1);
  size_t off = 0;
  const size_t o_status = off; off = align256(off + sizeof(int32_t));
  const size_t o_inv_q = off;  off = align256(off + sizeof(float) * (size_t)queries->n_rows);
  const size_t o_inv_i = off;  off = align256(off + sizeof(float) * (size_t)width);
  const size_t o_cnt = off;    off = align256(off + sizeof(int32_t) * (size_t)(dim + 1));
  const size_t o_ptr = off;    off = align256(off + sizeof(int32_t) * (size_t)(dim + 1));
  const size_t o_part = off;   off = align256(off + sizeof(int32_t) * (size_t)(tiles + 1));
  const size_t o_item = off;   off = align256(off + sizeof(uint16_t) * (size_t)chunk_nnz);
  const size_t o_val = off;    off = align256(off + sizeof(float) * (size_t)chunk_nnz);
  const size_t o_hat = off;    off = align256(off + sizeof(int2) * (size_t)chunk_nnz);
  const size_t o_rows = off;   off = align256(off + 2 * sizeof(int32_t));
  if (off > (size_t)SS_NOALLOC_SCRATCH_BYTES) return SS_ERR_LIMIT;

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SS_ERR_CUDA;
  void *base = nullptr;
  int sm_count = 0;
  ss_status st = scratch_for_device(device, &base, &sm_count);
  if (st != SS_OK) return st;
  unsigned char *b = static_cast<unsigned char *>(base);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // A handle-shaped view of the scratch, so the existing launchers run
  // unchanged on it.  It lives on the host stack; nothing is allocated.
  ss_handle view;
  view.device = device;
  view.dim = dim;
  view.chunk_rows = (int32_t)width;
  view.algo = ALGO_POSTING;
  view.mode = MODE_POSTING;
  view.build_batch = 1;
  view.sm_count = sm_count;
  // The kernels report what they find in the caller's status word when one
  // is given, else in the scratch's own (which nobody reads).
  view.d_status = device_status ? device_status : reinterpret_cast<int32_t *>(b + o_status);
  view.col_cnt = reinterpret_cast<int32_t *>(b + o_cnt);
  view.col_ptr = reinterpret_cast<int32_t *>(b + o_ptr);
  view.scan_part = reinterpret_cast<int32_t *>(b + o_part);
  view.scan_tiles = tiles;
  view.post_item = reinterpret_cast<uint16_t *>(b + o_item);
  view.post_val = reinterpret_cast<float *>(b + o_val);
  view.post_hat = reinterpret_cast<int2 *>(b + o_hat);
  view.post_cap = chunk_nnz;
  view.row_next = reinterpret_cast<int32_t *>(b + o_rows);
  float *inv_q = reinterpret_cast<float *>(b + o_inv_q);
  float *inv_i = reinterpret_cast<float *>(b + o_inv_i);

  // The scratch keeps the previous call's contents: the status word and the
  // scorer's row counter start at zero here, and the index builder clears
  // its own counters.
  if (cudaMemsetAsync(view.d_status, 0, sizeof(int32_t), s) != cudaSuccess) return SS_ERR_CUDA;
  if (cudaMemsetAsync(view.row_next, 0, 2 * sizeof(int32_t), s) != cudaSuccess) return SS_ERR_CUDA;
  if (launch_row_norms(*queries, inv_q, sm_count, s) != cudaSuccess) return SS_ERR_CUDA;
  ss_csr chunk_rows = *items;
  chunk_rows.indptr = items->indptr + row_begin;
  chunk_rows.n_rows = width;
  if (launch_row_norms(chunk_rows, inv_i, sm_count, s) != cudaSuccess) return SS_ERR_CUDA;
  if (launch_build_index(&view, *items, row_begin, row_end, s) != cudaSuccess) return SS_ERR_CUDA;
  int queued = 0;
  if (launch_score_lists(&view, *queries, inv_q, view.views[0], inv_i, out, ld_out, s, &queued) !=
      cudaSuccess)
    return SS_ERR_CUDA;
  return SS_OK;
}
