// The hot set in shared memory: a small open-addressing table of the item
// matrix's hot dimensions (<= kHotMax keys in kHotSlots slots), dimension ->
// position in the ascending hot list.  Shared by the builders and scorers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"

namespace hotset {

constexpr int kHotSlots = 128;

__device__ __forceinline__ uint32_t hash_a(int32_t k, int bits) {
  return ((uint32_t)k * 0x9E3779B1u) >> (32 - bits);
}
__device__ __forceinline__ uint32_t hash_b(int32_t k, int bits) {
  return ((uint32_t)k * 0x85EBCA77u) >> (32 - bits);
}

__device__ __forceinline__ void hot_insert(int *keys, int8_t *vals, int32_t k, int h) {
  uint32_t s = hash_a(k, 7);
  for (int n = 0; n < kHotSlots; ++n) {
    if (atomicCAS(&keys[s], -1, k) == -1) {
      vals[s] = (int8_t)h;
      return;
    }
    s = (s + 1) & (kHotSlots - 1);
  }
}
__device__ __forceinline__ int hot_find(const int *keys, const int8_t *vals, int32_t k) {
  if (k < 0) return -1;  // empty slots hold -1; no hot dimension is negative
  uint32_t s = hash_a(k, 7);
  for (int n = 0; n < kHotSlots; ++n) {
    const int key = keys[s];
    if (key == k) return vals[s];
    if (key == -1) return -1;
    s = (s + 1) & (kHotSlots - 1);
  }
  return -1;
}

// Fills the table from hot[0] = H, hot[1..H] (all threads of the block take
// part; ends with a barrier).  Returns H; a null hot set is an empty one.
__device__ __forceinline__ int load_hot_set(const int32_t *hot, int *keys, int8_t *vals) {
  for (int j = threadIdx.x; j < kHotSlots; j += blockDim.x) keys[j] = -1;
  __syncthreads();
  const int H = hot ? hot[0] : 0;
  for (int j = threadIdx.x; j < H; j += blockDim.x) hot_insert(keys, vals, hot[1 + j], j);
  __syncthreads();
  return H;
}

}  // namespace hotset
