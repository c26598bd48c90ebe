// Scoring kernel: sparse dot products of every query row with every item of
// one indexed chunk, normalised in the store.
//
// Blog post "Engineering practice for bulk similarity calculation over sparse
// embeddings": section 3.1 (u.v summed over supp(u) and supp(v)) and
// section 4.4 (normalise by the two norms right after the product).
//
// One warp owns one query row and an item tile of kTileItems items, held as
// float32 accumulators in shared memory.  For each nonzero (k, q_k) of the
// row, in ascending k, the warp walks the posting list of k and adds
// q_k * v_ik into the accumulator of item i.  A posting list names each item
// at most once, so the 32 lanes never touch the same accumulator inside one
// list, and a __syncwarp between lists orders the lists: the sum for each
// (q, i) is formed in ascending dimension order, the same order as a merge of
// the two sorted index lists.  The store multiplies by inv_q[q] * inv_i[i]
// and writes 16-byte vectors when the output is aligned.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "internal.cuh"

namespace {

constexpr int kRowsPerBlock = 8;   // warps per block, one query row each
constexpr int kTileItems = 2048;   // items per block (shared: 8 x 2048 x 4 B = 64 KB)

__global__ void __launch_bounds__(kRowsPerBlock * 32)
    k_score_rows(const int64_t *__restrict__ q_indptr, const int32_t *__restrict__ q_idx,
                 const float *__restrict__ q_val, int64_t n_q, const float *__restrict__ inv_q,
                 const int32_t *__restrict__ col_ptr, const uint16_t *__restrict__ post_item,
                 const float *__restrict__ post_val, const float *__restrict__ inv_i,
                 int32_t n_items, int32_t dim, int32_t capacity, float *__restrict__ out,
                 int64_t ld_out, int vec_ok) {
  extern __shared__ float4 smem4[];
  float *acc_all = reinterpret_cast<float *>(smem4);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t q = (int64_t)blockIdx.x * kRowsPerBlock + warp;
  const int32_t i0 = (int32_t)blockIdx.y * kTileItems;
  const int32_t width = min(kTileItems, n_items - i0);
  float *acc = acc_all + warp * kTileItems;
  float4 *acc4 = reinterpret_cast<float4 *>(acc);
  for (int c = lane; c < kTileItems / 4; c += 32) acc4[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncwarp();
  if (q >= n_q) return;

  const int64_t jb = q_indptr[q], je = q_indptr[q + 1];
  for (int64_t j = jb; j < je; ++j) {
    const int32_t k = __ldg(q_idx + j);
    if ((uint32_t)k >= (uint32_t)dim) continue;  // invalid input: never read outside col_ptr
    const float qk = __ldg(q_val + j);
    const int32_t lo = __ldg(col_ptr + k), hi = min(__ldg(col_ptr + k + 1), capacity);
    for (int32_t p = lo + lane; p < hi; p += 32) {
      const int32_t it = (int32_t)__ldg(post_item + p) - i0;
      if ((unsigned)it < (unsigned)kTileItems) acc[it] = fmaf(qk, __ldg(post_val + p), acc[it]);
    }
    __syncwarp();
  }

  const float iq = __ldg(inv_q + q);
  float *orow = out + q * ld_out + i0;
  const float *ii = inv_i + i0;
  if (vec_ok) {
    const int w4 = width & ~3;
    for (int c = lane * 4; c < w4; c += 128) {
      const float4 a = acc4[c >> 2];
      const float4 n = *reinterpret_cast<const float4 *>(ii + c);
      float4 o;
      o.x = a.x * iq * n.x;
      o.y = a.y * iq * n.y;
      o.z = a.z * iq * n.z;
      o.w = a.w * iq * n.w;
      *reinterpret_cast<float4 *>(orow + c) = o;
    }
    for (int c = w4 + lane; c < width; c += 32) orow[c] = acc[c] * iq * ii[c];
  } else {
    for (int c = lane; c < width; c += 32) orow[c] = acc[c] * iq * ii[c];
  }
}

}  // namespace

cudaError_t launch_score_chunk(const ss_handle *h, const ss_csr &queries, const float *inv_q,
                               const ss_index &idx, const float *inv_i, float *out,
                               int64_t ld_out, cudaStream_t s) {
  (void)h;
  if (queries.n_rows == 0 || idx.n_items == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * kRowsPerBlock * kTileItems;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_score_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int vec_ok = ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(inv_i)) % 16 == 0) &&
                     (ld_out % 4 == 0);
  dim3 grid((unsigned)((queries.n_rows + kRowsPerBlock - 1) / kRowsPerBlock),
            (unsigned)((idx.n_items + kTileItems - 1) / kTileItems));
  k_score_rows<<<grid, kRowsPerBlock * 32, smem, s>>>(
      queries.indptr, queries.indices, queries.values, queries.n_rows, inv_q, idx.col_ptr,
      idx.post_item, idx.post_val, inv_i, idx.n_items, (int32_t)idx.dim,
      (int32_t)std::min<int64_t>(idx.capacity, INT32_MAX), out, ld_out, vec_ok);
  return cudaGetLastError();
}
