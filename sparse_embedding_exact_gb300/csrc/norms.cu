// Row norms and CSR validation.
//
// Row norms follow section 5.2 of the blog post ("Engineering practice for
// bulk similarity calculation over sparse embeddings"): the Euclidean norm of
// a row is taken over its stored nonzeros only, never over a densified row.
// The product path needs 1/|row|, so that is what is stored.
#include <cuda_runtime.h>
#include <math.h>

#include "internal.cuh"

namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per row.  Squares are summed in double (a float squared is exact
// in double), so the only roundings are the double sum and the final
// reciprocal square root; inv = 0 for a row whose sum is 0.
__global__ void __launch_bounds__(kNormThreads)
    k_row_inv_norms(const int64_t *__restrict__ indptr, const float *__restrict__ values,
                    int64_t n_rows, float *__restrict__ inv) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kNormThreads / 32);
  for (int64_t r = (int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5); r < n_rows;
       r += warps) {
    const int64_t b = indptr[r], e = indptr[r + 1];
    double s = 0.0;
    for (int64_t j = b + lane; j < e; j += 32) {
      const double v = (double)__ldg(values + j);
      s = fma(v, v, s);
    }
    s = warp_sum(s);
    if (lane == 0) inv[r] = (s > 0.0) ? (float)(1.0 / sqrt(s)) : 0.0f;
  }
}

__device__ __forceinline__ void flag(int32_t *status, int32_t code) {
  atomicCAS(status, DEV_OK, code);
}

// One warp per row: indptr monotone and inside [0, nnz], indices strictly
// increasing and inside [0, dim).
__global__ void __launch_bounds__(kNormThreads)
    k_validate_csr(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                   int64_t n_rows, int64_t nnz, int64_t dim, int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kNormThreads / 32);
  const int64_t first = (int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
  if (first == 0 && lane == 0) {
    if (indptr[0] != 0 || indptr[n_rows] != nnz) flag(status, DEV_OUT_OF_RANGE);
  }
  for (int64_t r = first; r < n_rows; r += warps) {
    const int64_t b = indptr[r], e = indptr[r + 1];
    if (b < 0 || e < b || e > nnz) {
      if (lane == 0) flag(status, DEV_OUT_OF_RANGE);
      continue;
    }
    bool bad_range = false, bad_order = false;
    for (int64_t j = b + lane; j < e; j += 32) {
      const int32_t k = indices[j];
      if (k < 0 || (int64_t)k >= dim) bad_range = true;
      if (j > b && indices[j - 1] >= k) bad_order = true;
    }
    if (__any_sync(0xffffffffu, bad_range)) {
      if (lane == 0) flag(status, DEV_OUT_OF_RANGE);
    } else if (__any_sync(0xffffffffu, bad_order)) {
      if (lane == 0) flag(status, DEV_UNSORTED);
    }
  }
}

int grid_for_rows(int64_t n_rows, int sm_count) {
  const int64_t need = (n_rows + (kNormThreads / 32) - 1) / (kNormThreads / 32);
  const int64_t cap = (int64_t)(sm_count > 0 ? sm_count : 148) * 16;
  return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace

cudaError_t launch_row_norms(const ss_csr &m, float *inv_norms, int sm_count, cudaStream_t s) {
  if (m.n_rows == 0) return cudaSuccess;
  k_row_inv_norms<<<grid_for_rows(m.n_rows, sm_count), kNormThreads, 0, s>>>(
      m.indptr, m.values, m.n_rows, inv_norms);
  return cudaGetLastError();
}

cudaError_t launch_validate_csr(const ss_csr &m, int32_t *d_status, int sm_count, cudaStream_t s) {
  k_validate_csr<<<grid_for_rows(m.n_rows, sm_count), kNormThreads, 0, s>>>(
      m.indptr, m.indices, m.n_rows, m.nnz, m.dim, d_status);
  return cudaGetLastError();
}
