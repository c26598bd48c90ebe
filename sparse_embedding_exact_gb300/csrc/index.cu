// Per-chunk inverted index: the chunk's CSR rows turned into one posting list
// per dimension (CSR -> CSC by dimension).
//
// The blog post ("Engineering practice for bulk similarity calculation over
// sparse embeddings", section 3.1) computes u.v over supp(u) and supp(v);
// the posting list of dimension k names every item of the chunk whose support
// holds k, so a query nonzero at k meets exactly the items it multiplies.
//
// One build covers up to B chunks of C rows (B counter arrays of dim + 1 laid
// end to end).  Steps (all on the device, queued on one stream):
//   1. histogram: count[c][k] = number of rows of chunk c holding dimension k;
//   2. exclusive scan of the B * (dim + 1) counters as one array -> col_ptr
//      (tile sums, a scan of the tile sums, then the tiles again with
//      warp-shuffle scans).  Chunk c's lists thus follow chunk c-1's, and
//      col_ptr[c][k] is an absolute position in the build's entry arrays;
//   3. scatter: every nonzero (row r of chunk c, dim k, value v) takes the
//      next slot of list (c, k) and stores (item r - first row of c, v).
// A list's entries are in no particular order; the scorer does not need one.
//
// Hot dimensions.  When the item matrix has at least kSplitMinHot hot
// dimensions (a Zipf-like head held by a large share of the rows), their
// values go to a dense slab per chunk, slab[c][h][item], and not into the
// lists: the scorer multiplies them as a small dense product and walks the
// lists of the other ("cold") dimensions only.
#include <cuda_runtime.h>

#include <algorithm>

#include "hotset.cuh"
#include "internal.cuh"

namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 16;  // per thread
constexpr int kScanTile = kScanThreads * kScanItems;
constexpr int kHistThreads = 256;

__device__ __forceinline__ void flag(int32_t *status, int32_t code) {
  atomicCAS(status, DEV_OK, code);
}

__global__ void __launch_bounds__(kHistThreads)
    k_histogram(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                int64_t row_begin, int64_t row_end, int64_t chunk_rows, int n_chunks, int64_t dim,
                const int32_t *__restrict__ hot, int32_t *__restrict__ count, int32_t *status) {
  // First entry of each chunk of the build, then the build's end.
  __shared__ int64_t bound[kMaxBuildBatch + 1];
  __shared__ int hkeys[hotset::kHotSlots];
  __shared__ int8_t hvals[hotset::kHotSlots];
  const bool split = hotset::load_hot_set(hot, hkeys, hvals) >= kSplitMinHot;
  if (threadIdx.x <= n_chunks) {
    const int64_t r = min(row_begin + (int64_t)threadIdx.x * chunk_rows, row_end);
    bound[threadIdx.x] = indptr[r];
  }
  __syncthreads();
  const int64_t p0 = bound[0], p1 = bound[n_chunks];
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t p = p0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < p1; p += stride) {
    const int32_t k = __ldg(indices + p);
    int c = 0;
    while (c + 1 < n_chunks && p >= bound[c + 1]) ++c;
    if (k >= 0 && (int64_t)k < dim) {
      if (split && hotset::hot_find(hkeys, hvals, k) >= 0) continue;  // goes to the slab
      atomicAdd(count + (int64_t)c * (dim + 1) + k, 1);
    } else {
      flag(status, DEV_OUT_OF_RANGE);
    }
  }
}

// Inclusive warp scan with shuffles.
__device__ __forceinline__ int32_t warp_inclusive_scan(int32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive block scan of one value per thread (warp-shuffle scans inside
// each warp, then one warp scans the warp totals).  *total gets the sum.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t *total) {
  constexpr int kWarps = kScanThreads / 32;
  __shared__ int32_t warp_off[kWarps];
  __shared__ int32_t block_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t inc = warp_inclusive_scan(v);
  if (lane == 31) warp_off[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int32_t w = (lane < kWarps) ? warp_off[lane] : 0;
    const int32_t winc = warp_inclusive_scan(w);
    if (lane < kWarps) warp_off[lane] = winc - w;
    if (lane == kWarps - 1) block_total = winc;
  }
  __syncthreads();
  const int32_t r = warp_off[warp] + inc - v;
  *total = block_total;
  __syncthreads();  // warp_off and block_total are reused by the next call
  return r;
}

// A tile of kScanTile counters is read as kScanItems / 4 slices of
// kScanThreads int4 vectors: thread t holds counters [4 t, 4 t + 4) of each
// slice, so every warp access covers 512 contiguous bytes.  Vectors that
// run past n are read and written element by element.
__device__ __forceinline__ int4 load4(const int32_t *a, int64_t i, int64_t n) {
  if (i + 4 <= n) return *reinterpret_cast<const int4 *>(a + i);
  int4 v = make_int4(0, 0, 0, 0);
  if (i < n) v.x = a[i];
  if (i + 1 < n) v.y = a[i + 1];
  if (i + 2 < n) v.z = a[i + 2];
  return v;
}
__device__ __forceinline__ void store4(int32_t *a, int64_t i, int64_t n, int4 v) {
  if (i + 4 <= n) {
    *reinterpret_cast<int4 *>(a + i) = v;
    return;
  }
  if (i < n) a[i] = v.x;
  if (i + 1 < n) a[i + 1] = v.y;
  if (i + 2 < n) a[i + 2] = v.z;
}
constexpr int kScanSlices = kScanItems / 4;

// Phase 1: sum of each tile of kScanTile counters.
__global__ void __launch_bounds__(kScanThreads)
    k_scan_tile_sums(const int32_t *__restrict__ count, int64_t n, int32_t *__restrict__ part) {
  const int64_t tile = (int64_t)blockIdx.x * kScanTile;
  int4 v[kScanSlices];
#pragma unroll
  for (int sl = 0; sl < kScanSlices; ++sl) v[sl] = load4(count, tile + 4 * ((int64_t)sl * kScanThreads + threadIdx.x), n);
  int32_t s = 0;
#pragma unroll
  for (int sl = 0; sl < kScanSlices; ++sl) s += v[sl].x + v[sl].y + v[sl].z + v[sl].w;
  int32_t total;
  block_exclusive_scan(s, &total);
  if (threadIdx.x == 0) part[blockIdx.x] = total;
}

// Phase 2: one block scans the tile sums (exclusive), carrying across passes.
__global__ void __launch_bounds__(kScanThreads)
    k_scan_partials(int32_t *__restrict__ part, int64_t n_tiles) {
  int32_t carry = 0;
  for (int64_t b = 0; b < n_tiles; b += kScanThreads) {
    const int64_t i = b + threadIdx.x;
    const int32_t v = (i < n_tiles) ? part[i] : 0;
    int32_t total;
    const int32_t ex = block_exclusive_scan(v, &total);
    if (i < n_tiles) part[i] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) part[n_tiles] = carry;
}

// Phase 3: exclusive scan inside each tile plus the tile offset, slice by
// slice; writes col_ptr and resets the counters to the same values (scatter
// cursors).
__global__ void __launch_bounds__(kScanThreads)
    k_scan_apply(int32_t *__restrict__ count, int64_t n, const int32_t *__restrict__ part,
                 int32_t *__restrict__ col_ptr) {
  const int64_t tile = (int64_t)blockIdx.x * kScanTile;
  int4 v[kScanSlices];
#pragma unroll
  for (int sl = 0; sl < kScanSlices; ++sl) v[sl] = load4(count, tile + 4 * ((int64_t)sl * kScanThreads + threadIdx.x), n);
  int32_t carry = part[blockIdx.x];
#pragma unroll
  for (int sl = 0; sl < kScanSlices; ++sl) {
    const int32_t s = v[sl].x + v[sl].y + v[sl].z + v[sl].w;
    int32_t total;
    const int32_t run = block_exclusive_scan(s, &total) + carry;
    const int4 o = make_int4(run, run + v[sl].x, run + v[sl].x + v[sl].y, run + v[sl].x + v[sl].y + v[sl].z);
    const int64_t i = tile + 4 * ((int64_t)sl * kScanThreads + threadIdx.x);
    store4(col_ptr, i, n, o);
    store4(count, i, n, o);
    carry += total;
  }
}

// One warp per row: each nonzero claims the next slot of its list.
__global__ void __launch_bounds__(kHistThreads)
    k_scatter(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
              const float *__restrict__ values, int64_t row_begin, int64_t row_end,
              int64_t chunk_rows, int64_t dim, const int32_t *__restrict__ hot,
              int32_t *__restrict__ cursor, uint16_t *__restrict__ post_item,
              float *__restrict__ post_val, float *__restrict__ slab, int64_t capacity,
              int32_t *status) {
  __shared__ int hkeys[hotset::kHotSlots];
  __shared__ int8_t hvals[hotset::kHotSlots];
  const bool split = hotset::load_hot_set(hot, hkeys, hvals) >= kSplitMinHot;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kHistThreads / 32);
  for (int64_t r = row_begin + (int64_t)blockIdx.x * (kHistThreads / 32) + (threadIdx.x >> 5);
       r < row_end; r += warps) {
    const int64_t b = indptr[r], e = indptr[r + 1];
    const int64_t c = (r - row_begin) / chunk_rows;
    int32_t *cur = cursor + c * (dim + 1);
    const uint16_t item = (uint16_t)(r - row_begin - c * chunk_rows);
    for (int64_t j = b + lane; j < e; j += 32) {
      const int32_t k = __ldg(indices + j);
      if (k < 0 || (int64_t)k >= dim) continue;  // flagged by the histogram
      if (split) {
        const int hh = hotset::hot_find(hkeys, hvals, k);
        if (hh >= 0) {
          slab[(c * hyb::kHotMax + hh) * chunk_rows + item] = __ldg(values + j);
          continue;
        }
      }
      const int32_t pos = atomicAdd(cur + k, 1);
      if (pos >= 0 && (int64_t)pos < capacity) {
        post_item[pos] = item;
        post_val[pos] = __ldg(values + j);
      } else {
        flag(status, DEV_CAPACITY);
      }
    }
  }
}

}  // namespace

int64_t scan_tile_count(int64_t n) { return (n + kScanTile - 1) / kScanTile; }

cudaError_t launch_count_scan(int32_t *count, int64_t n, int32_t *part, int32_t *col_ptr,
                              cudaStream_t s) {
  const int64_t tiles = scan_tile_count(n);
  k_scan_tile_sums<<<(unsigned)tiles, kScanThreads, 0, s>>>(count, n, part);
  k_scan_partials<<<1, kScanThreads, 0, s>>>(part, tiles);
  k_scan_apply<<<(unsigned)tiles, kScanThreads, 0, s>>>(count, n, part, col_ptr);
  return cudaGetLastError();
}

cudaError_t launch_build_index(ss_handle *h, const ss_csr &items, int64_t row_begin,
                               int64_t row_end, cudaStream_t s) {
  const int64_t C = h->chunk_rows;
  const int n_chunks = (int)((row_end - row_begin + C - 1) / C);
  h->n_views = 0;
  if (n_chunks < 1 || n_chunks > h->build_batch) return cudaErrorInvalidValue;
  const int64_t stride = h->dim + 1;
  const int64_t n = stride * n_chunks;
  cudaError_t e = cudaMemsetAsync(h->col_cnt, 0, sizeof(int32_t) * (size_t)n, s);
  if (e != cudaSuccess) return e;
  // The hot slab (used only when the hot set is large enough to split off).
  const int32_t *hot = h->slab_post ? h->hot : nullptr;
  if (hot) {
    e = cudaMemsetAsync(h->slab_post, 0, sizeof(float) * (size_t)n_chunks * hyb::kHotMax * (size_t)C, s);
    if (e != cudaSuccess) return e;
  }
  const int grid = h->sm_count * 8;
  k_histogram<<<grid, kHistThreads, 0, s>>>(items.indptr, items.indices, row_begin, row_end, C,
                                            n_chunks, h->dim, hot, h->col_cnt, h->d_status);
  const int64_t tiles = scan_tile_count(n);
  k_scan_tile_sums<<<(unsigned)tiles, kScanThreads, 0, s>>>(h->col_cnt, n, h->scan_part);
  k_scan_partials<<<1, kScanThreads, 0, s>>>(h->scan_part, tiles);
  k_scan_apply<<<(unsigned)tiles, kScanThreads, 0, s>>>(h->col_cnt, n, h->scan_part, h->col_ptr);
  k_scatter<<<grid, kHistThreads, 0, s>>>(items.indptr, items.indices, items.values, row_begin,
                                          row_end, C, h->dim, hot, h->col_cnt, h->post_item,
                                          h->post_val, h->slab_post, h->post_cap, h->d_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  for (int k = 0; k < n_chunks; ++k) {
    ss_index &ix = h->views[k];
    ix = ss_index();
    ix.algo = ALGO_POSTING;
    ix.row_begin = row_begin + (int64_t)k * C;
    ix.row_end = std::min<int64_t>(ix.row_begin + C, row_end);
    ix.n_items = (int32_t)(ix.row_end - ix.row_begin);
    ix.dim = h->dim;
    ix.col_ptr = h->col_ptr + (size_t)k * stride;
    ix.post_item = h->post_item;
    ix.post_val = h->post_val;
    ix.capacity = h->post_cap;
    ix.hot = hot;
    ix.slab = hot ? h->slab_post + (size_t)k * hyb::kHotMax * (size_t)C : nullptr;
    ix.slab_ld = (int32_t)C;
  }
  h->n_views = n_chunks;
  return cudaSuccess;
}
