// Device helpers of the top-k epilogue, shared by the scoring kernels.
//
// Each scorer offers, per query row and per slice of 256 items of a chunk,
// the scores not below the row's current k-th best (at most k of them, the
// best in the top-k order when more pass) as candidates; a merge kernel then
// folds a chunk's candidates into the running best k.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.cuh"

namespace topk_dev {

__device__ __forceinline__ void flag_status(int32_t *status, int32_t code) {
  atomicCAS(status, DEV_OK, code);
}

// Order of the top-k epilogue: larger score first, equal scores by smaller
// item number.
__device__ __forceinline__ bool topk_before(float v, int64_t i, float w, int64_t j) {
  return v > w || (v == w && i < j);
}

// How many of query row q's scores in one item tile (8 per lane) are >= thr
// (the row's current k-th best score).
__device__ __forceinline__ int topk_count(float thr, const float (&v)[8], const bool (&valid)[8]) {
  int count = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) count += __popc(__ballot_sync(0xffffffffu, valid[j] && v[j] >= thr));
  return count;
}

// Writes a tile's offer for query row q at slots [base, base + min(count,
// k)) of the row's candidates: the scores >= thr, or when more than k pass,
// the k best in the top-k order (k rounds of warp arg-best).  Items are
// chunk-relative.
__device__ __forceinline__ void topk_emit(const ss_topk &t, int64_t q, float thr, const float (&v)[8],
                                          const int (&item)[8], const bool (&valid)[8], int base,
                                          int count, int lane) {
  bool pass[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) pass[j] = valid[j] && v[j] >= thr;
  float *cv = t.cand_val + q * t.cand_cap + base;
  int32_t *ci = t.cand_item + q * t.cand_cap + base;
  if (count <= t.k) {
    const unsigned lt = (1u << lane) - 1u;
    int off = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const unsigned m = __ballot_sync(0xffffffffu, pass[j]);
      if (pass[j]) {
        const int pos = off + __popc(m & lt);
        cv[pos] = v[j];
        ci[pos] = item[j];
      }
      off += __popc(m);
    }
    return;
  }
  for (int r = 0; r < t.k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff, bj = -1;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (pass[j] && topk_before(v[j], item[j], bv, bi)) {
        bv = v[j];
        bi = item[j];
        bj = j;
      }
    float wv = bv;
    int wi = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
      if (topk_before(ov, oi, wv, wi)) {
        wv = ov;
        wi = oi;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)  // items are distinct: one lane holds the winner
      if (j == bj && bi == wi) pass[j] = false;
    if (lane == 0) {
      cv[r] = wv;
      ci[r] = wi;
    }
  }
}

// Offers query row q's scores of one item tile to the row's candidates
// (reserving the slots with one atomic).
__device__ __forceinline__ void topk_offer(const ss_topk &t, int64_t q, float thr, const float (&v)[8],
                                           const int (&item)[8], const bool (&valid)[8], int lane,
                                           int32_t *status) {
  const int count = topk_count(thr, v, valid);
  if (count == 0) return;
  const int n_emit = count < t.k ? count : t.k;
  int base = 0;
  if (lane == 0) base = atomicAdd(t.cand_n + q, n_emit);
  base = __shfl_sync(0xffffffffu, base, 0);
  if (base + n_emit > t.cand_cap) {  // cannot happen: a chunk's tiles offer at most k each
    if (lane == 0) flag_status(status, DEV_CAPACITY);
    return;
  }
  topk_emit(t, q, thr, v, item, valid, base, count, lane);
}

}  // namespace topk_dev
