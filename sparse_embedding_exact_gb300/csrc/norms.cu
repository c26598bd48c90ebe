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

constexpr int kNormLanes = 8;  // lanes per row: a warp takes 4 rows at a time

// Float-float arithmetic (Knuth's two-sum; products split exactly with an
// fma).  The rounded intrinsics keep the compiler from fusing the steps.
// Adds x^2 to the pair (s, c), whose value is s + c.
__device__ __forceinline__ void ff_add_square(float x, float &s, float &c) {
  const float p = __fmul_rn(x, x);
  const float pe = __fmaf_rn(x, x, -p);  // p + pe == x^2 exactly (x^2 not subnormal)
  const float t = __fadd_rn(s, p);
  const float bp = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp));  // s + p == t + err
  s = t;
  c = __fadd_rn(c, __fadd_rn(err, pe));
}
__device__ __forceinline__ void ff_add(float &s, float &c, float s2, float c2) {
  const float t = __fadd_rn(s, s2);
  const float bp = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(s2, bp));
  s = t;
  c = __fadd_rn(c, __fadd_rn(err, c2));
}

// Sum of squares of row [b, e) over the kNormLanes lanes of a group, each
// value multiplied by 2^-scale_exp first (exact for normal results).  Every
// lane of the group gets (hi, lo) with hi = fl(hi + lo).
__device__ __forceinline__ void group_sum_squares(const float *values, int64_t b, int64_t e, int li,
                                                  int scale_exp, float &hi, float &lo) {
  float s = 0.f, c = 0.f;
  for (int64_t j = b + li; j < e; j += kNormLanes) {
    const float v = __ldg(values + j);
    ff_add_square(scale_exp == 0 ? v : ldexpf(v, -scale_exp), s, c);
  }
#pragma unroll
  for (int o = kNormLanes / 2; o > 0; o >>= 1)
    ff_add(s, c, __shfl_xor_sync(0xffffffffu, s, o), __shfl_xor_sync(0xffffffffu, c, o));
  hi = __fadd_rn(s, c);
  lo = __fsub_rn(c, __fsub_rn(hi, s));
}

// 1 / sqrt(hi + lo) for hi + lo > 0 in the normal range: one Newton step from
// rsqrtf with the residual 1 - (hi + lo) y^2 formed with fmas, which puts the
// result within one unit in the last place of the exact value.
__device__ __forceinline__ float ff_rsqrt(float hi, float lo) {
  const float y0 = rsqrtf(hi);
  const float th = __fmul_rn(y0, y0);
  const float tl = __fmaf_rn(y0, y0, -th);
  float r = __fmaf_rn(-hi, th, 1.0f);
  r = __fmaf_rn(-hi, tl, r);
  r = __fmaf_rn(-lo, th, r);
  return __fmaf_rn(__fmul_rn(0.5f, y0), r, y0);
}

// Groups of kNormLanes lanes per row.  The squares are summed in float-float
// (about 48 significant bits, far beyond what the rounded float result
// needs), so the only rounding that matters is the last one; inv = 0 for a
// row whose sum is 0.  A row whose plain sum leaves the comfortable float
// range (all values tiny, or squares overflowing) is summed again scaled by a
// power of two near its largest magnitude, and the result scaled back.
__global__ void __launch_bounds__(kNormThreads)
    k_row_inv_norms(const int64_t *__restrict__ indptr, const float *__restrict__ values,
                    int64_t n_rows, float *__restrict__ inv) {
  const int lane = threadIdx.x & 31;
  const int li = lane % kNormLanes;
  constexpr int kRowsPerWarp = 32 / kNormLanes;
  const int64_t warps = (int64_t)gridDim.x * (kNormThreads / 32);
  const int64_t quads = (n_rows + kRowsPerWarp - 1) / kRowsPerWarp;
  for (int64_t w = (int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5); w < quads;
       w += warps) {
    const int64_t r = w * kRowsPerWarp + lane / kNormLanes;
    const bool live = r < n_rows;
    const int64_t b = live ? indptr[r] : 0, e = live ? indptr[r + 1] : 0;
    float hi, lo;
    group_sum_squares(values, b, e, li, 0, hi, lo);
    float out = 0.f;
    const bool plain = hi >= 0x1p-60f && hi <= 0x1p+100f;
    if (plain) out = ff_rsqrt(hi, lo);
    // The rare rows outside that range (the condition is the same on all the
    // group's lanes, and every group of the warp takes the shuffles below).
    if (__any_sync(0xffffffffu, !plain)) {
      float m = 0.f;
      for (int64_t j = b + li; j < e; j += kNormLanes) m = fmaxf(m, fabsf(__ldg(values + j)));
#pragma unroll
      for (int o = kNormLanes / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int ex = m > 0.f ? ilogbf(m) : 0;
      float shi, slo;
      group_sum_squares(values, plain ? e : b, e, li, ex, shi, slo);
      if (!plain) out = (m > 0.f && shi > 0.f) ? ldexpf(ff_rsqrt(shi, slo), -ex) : 0.f;
    }
    if (live && li == 0) inv[r] = out;
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
