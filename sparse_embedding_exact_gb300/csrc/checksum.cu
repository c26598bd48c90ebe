// Per-chunk checksums of a result tile: the integrity check of a streamed
// result (a copy that changed a single bit changes the checksum).
//
// bits_sum  = sum over the tile of the float32 bit patterns read as unsigned
//             32-bit integers, modulo 2^64: exact and independent of the
//             order of summation, so a device tile and its host copy agree
//             exactly when, and as a rule only when, they are bit-identical;
// value_sum = sum of the values in double, for reporting (its last bits
//             depend on the summation order).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <thread>
#include <vector>

#include "internal.cuh"

namespace {

constexpr int kSumThreads = 256;

__global__ void __launch_bounds__(kSumThreads)
    k_tile_checksum(const float *__restrict__ tile, int64_t n_rows, int64_t n_cols, int64_t ld,
                    unsigned long long *bits_sum, double *value_sum) {
  __shared__ unsigned long long part_b[kSumThreads / 32];
  __shared__ double part_v[kSumThreads / 32];
  unsigned long long b = 0;
  double v = 0.0;
  const int64_t n = n_rows * n_cols;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / n_cols, c = e - r * n_cols;
    const float x = __ldg(tile + r * ld + c);
    b += (unsigned long long)__float_as_uint(x);
    v += (double)x;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    b += __shfl_xor_sync(0xffffffffu, b, o);
    v += __shfl_xor_sync(0xffffffffu, v, o);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    part_b[warp] = b;
    part_v[warp] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long tb = 0;
    double tv = 0.0;
    for (int w = 0; w < kSumThreads / 32; ++w) {
      tb += part_b[w];
      tv += part_v[w];
    }
    atomicAdd(bits_sum, tb);
    atomicAdd(value_sum, tv);
  }
}

}  // namespace

cudaError_t launch_tile_checksum(const float *tile, int64_t n_rows, int64_t n_cols, int64_t ld,
                                 uint64_t *bits_sum, double *value_sum, int sm_count,
                                 cudaStream_t s) {
  const int64_t n = n_rows * n_cols;
  if (n <= 0) return cudaSuccess;
  const int64_t need = (n + kSumThreads - 1) / kSumThreads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count * 8));
  k_tile_checksum<<<grid, kSumThreads, 0, s>>>(tile, n_rows, n_cols, ld,
                                               reinterpret_cast<unsigned long long *>(bits_sum),
                                               value_sum);
  return cudaGetLastError();
}

void tile_checksum_host(const float *tile, int64_t n_rows, int64_t n_cols, int64_t ld,
                        uint64_t *bits_sum, double *value_sum) {
  const unsigned hw = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
  const unsigned nt = (n_rows * n_cols < (1 << 20)) ? 1u : hw;
  std::vector<uint64_t> b(nt, 0);
  std::vector<double> v(nt, 0.0);
  auto work = [&](unsigned t) {
    uint64_t sb = 0;
    double sv = 0.0;
    for (int64_t r = t; r < n_rows; r += nt) {
      const float *row = tile + r * ld;
      for (int64_t c = 0; c < n_cols; ++c) {
        uint32_t u;
        memcpy(&u, row + c, sizeof(u));
        sb += u;
        sv += (double)row[c];
      }
    }
    b[t] = sb;
    v[t] = sv;
  };
  if (nt == 1) {
    work(0);
  } else {
    std::vector<std::thread> th;
    for (unsigned t = 0; t < nt; ++t) th.emplace_back(work, t);
    for (auto &x : th) x.join();
  }
  uint64_t tb = 0;
  double tv = 0.0;
  for (unsigned t = 0; t < nt; ++t) {
    tb += b[t];
    tv += v[t];
  }
  *bits_sum = tb;
  *value_sum = tv;
}
