// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "sparsecos.h"

// Device status word codes (first error wins; 0 = none).
enum : int32_t {
  DEV_OK = 0,
  DEV_UNSORTED = 1,
  DEV_OUT_OF_RANGE = 2,
  DEV_CAPACITY = 3,
};

// The per-chunk inverted index: for each dimension k of the chunk, the
// posting list of (item number within the chunk, value), laid out CSC-style
// by dimension.
struct ss_index {
  int64_t row_begin = 0;
  int64_t row_end = 0;
  int32_t n_items = 0;
  int64_t dim = 0;
  const int32_t *col_ptr = nullptr;    // [dim + 1], posting list k = [col_ptr[k], col_ptr[k+1])
  const uint16_t *post_item = nullptr; // [capacity]
  const float *post_val = nullptr;     // [capacity]
  int64_t capacity = 0;
};

struct ss_handle {
  int device = 0;
  int64_t dim = 0;
  int32_t chunk_rows = 0;
  int32_t flags = 0;
  int sm_count = 0;
  std::string last_error;
  uint64_t launches = 0;  // kernels queued by this handle

  // Device workspace, owned by the handle.
  int32_t *d_status = nullptr;   // one status word
  int32_t *col_cnt = nullptr;    // [dim + 1]: histogram, then scatter cursors
  int32_t *col_ptr = nullptr;    // [dim + 1]
  int32_t *scan_part = nullptr;  // [scan tiles + 1]
  int64_t scan_tiles = 0;
  uint16_t *post_item = nullptr; // [post_cap]
  float *post_val = nullptr;     // [post_cap]
  int64_t post_cap = 0;

  ss_index index;
};

// Launchers (all asynchronous on `s`).
cudaError_t launch_row_norms(const ss_csr &m, float *inv_norms, int sm_count, cudaStream_t s);
cudaError_t launch_validate_csr(const ss_csr &m, int32_t *d_status, int sm_count, cudaStream_t s);
cudaError_t launch_build_index(ss_handle *h, const ss_csr &items, int64_t row_begin,
                               int64_t row_end, cudaStream_t s);
cudaError_t launch_score_chunk(const ss_handle *h, const ss_csr &queries, const float *inv_q,
                               const ss_index &idx, const float *inv_i, float *out,
                               int64_t ld_out, cudaStream_t s);

// Kernels queued by one launch_build_index call.
constexpr int kIndexKernels = 5;

// Number of scan tiles needed for n counters.
int64_t scan_tile_count(int64_t n);
