// Hybrid scoring path: dense "hot" dimensions on the FP32 pipes, sparse
// "cold" dimensions through hashed posting lists in shared memory.
//
// What is computed is the sparse dot product of the blog post "Engineering
// practice for bulk similarity calculation over sparse embeddings", section
// 3.1 (u.v summed over supp(u) and supp(v)), normalised in the store
// (section 4.4).  How it is computed is a GB300 design of our own:
//
// In BM25/TF-IDF data a few dimensions (the head of the dictionary, section
// 3.2) sit in a large share of all rows, and they carry most of the
// multiply-adds: a dimension held by a fraction p of the rows costs p*p
// multiply-adds per (query, item) pair.  Those "hot" dimensions, chosen
// once per item matrix from a row sample, are stored dense and multiplied
// as a small dense product with register tiles (no tensor cores: the sums
// stay FP32 FMA).  Every other ("cold") dimension goes through lists: the
// query tile's cold nonzeros are grouped by dimension into a hash table in
// shared memory (dimension -> list of (query row, value)), and each item
// walks its own cold nonzeros, looks each one up, and adds value products
// into a shared-memory accumulator tile.
//
// Per chunk, the index builder writes, for each tile of kTI items:
//   slab[h][i]  value of hot dimension h in item i (0 if absent);
//   ell[s][i]   the s-th cold nonzero of item i (dimension, value), dims
//               ascending, padded with dimension -1 to the warp's longest;
//   a heavy list for items with far more cold nonzeros than the tile's
//   mean (processed cooperatively with shared-memory atomics).
//
// The scoring kernel is persistent: each block owns a contiguous range of
// (query tile, item tile) units.  Per unit:
//   1. hot:  acc[q][i] = sum_h Qhot[h][q] * slab[h][i]    (8x8 register tile
//            per thread, packed FP32x2 FMAs), stored to shared memory;
//   2. cold: thread i walks item i's ELL entries; a hit on dimension k walks
//            the query list of k and does acc[q][i] += q_k * v_ik.  Thread i
//            alone owns column i, so no two threads touch one accumulator;
//   3. store: S = acc * inv_q * inv_i, 16-byte streaming stores.
// For each (q, i) the sum runs over hot dims ascending, then cold dims
// ascending (heavy items excepted: their cold adds are atomic).
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "internal.cuh"

namespace {

using namespace hyb;

constexpr int kSelThreads = 1024;
constexpr int kSelSlotsBits = 14;
constexpr int kSelSlots = 1 << kSelSlotsBits;
constexpr int kSelCand = 1024;
constexpr int kHotSlots = 128;

__device__ __forceinline__ void flag(int32_t *status, int32_t code) {
  atomicCAS(status, DEV_OK, code);
}

__device__ __forceinline__ uint32_t hash_a(int32_t k, int bits) {
  return ((uint32_t)k * 0x9E3779B1u) >> (32 - bits);
}
__device__ __forceinline__ uint32_t hash_b(int32_t k, int bits) {
  return ((uint32_t)k * 0x85EBCA77u) >> (32 - bits);
}

// ---------------------------------------------------------------- hot set
// Small open-addressing table of the hot dimensions (<= kHotMax keys in
// kHotSlots slots): dimension -> position in the ascending hot list.
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
  uint32_t s = hash_a(k, 7);
  for (int n = 0; n < kHotSlots; ++n) {
    const int key = keys[s];
    if (key == k) return vals[s];
    if (key == -1) return -1;
    s = (s + 1) & (kHotSlots - 1);
  }
  return -1;
}

// One block: counts the dimensions of `n_sample` evenly spaced rows in a
// shared hash table, keeps those held by >= kHotMinPercent of the sampled
// rows, the kHotMax most frequent of them (ties to the lower dimension), and
// writes hot[0] = H, hot[1..H] = those dimensions ascending.
__global__ void __launch_bounds__(kSelThreads)
    k_hot_select(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                 int64_t n_rows, int64_t n_sample, int32_t *__restrict__ hot) {
  extern __shared__ int sel_smem[];
  int *keys = sel_smem;
  int *cnts = sel_smem + kSelSlots;
  __shared__ int cand_dim[kSelCand], cand_cnt[kSelCand], cand_sel[kSelCand];
  __shared__ int n_cand;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int s = tid; s < kSelSlots; s += kSelThreads) {
    keys[s] = -1;
    cnts[s] = 0;
  }
  if (tid == 0) n_cand = 0;
  __syncthreads();
  for (int64_t j = warp; j < n_sample; j += kSelThreads / 32) {
    const int64_t r = j * n_rows / n_sample;
    for (int64_t p = indptr[r] + lane; p < indptr[r + 1]; p += 32) {
      const int32_t k = indices[p];
      uint32_t s = hash_a(k, kSelSlotsBits);
      for (int n = 0; n < kSelSlots; ++n) {
        const int prev = atomicCAS(&keys[s], -1, k);
        if (prev == -1 || prev == k) {
          atomicAdd(&cnts[s], 1);
          break;
        }
        s = (s + 1) & (kSelSlots - 1);
      }
    }
  }
  __syncthreads();
  const int thr = max(2, (int)((n_sample * kHotMinPercent + 99) / 100));
  for (int s = tid; s < kSelSlots; s += kSelThreads) {
    if (keys[s] >= 0 && cnts[s] >= thr) {
      const int c = atomicAdd(&n_cand, 1);
      if (c < kSelCand) {
        cand_dim[c] = keys[s];
        cand_cnt[c] = cnts[s];
      }
    }
  }
  __syncthreads();
  const int n = min(n_cand, kSelCand);
  for (int c = tid; c < n; c += kSelThreads) {
    int rank = 0;
    for (int j = 0; j < n; ++j)
      rank += (cand_cnt[j] > cand_cnt[c]) || (cand_cnt[j] == cand_cnt[c] && cand_dim[j] < cand_dim[c]);
    cand_sel[c] = rank < kHotMax;
  }
  __syncthreads();
  for (int c = tid; c < n; c += kSelThreads) {
    if (!cand_sel[c]) continue;
    int pos = 0;
    for (int j = 0; j < n; ++j) pos += cand_sel[j] && cand_dim[j] < cand_dim[c];
    hot[1 + pos] = cand_dim[c];
  }
  if (tid == 0) hot[0] = min(n, kHotMax);
}

// ---------------------------------------------------------------- builder
__device__ __forceinline__ int block_sum(int v, int *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ int block_exclusive_scan(int v, int *red, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  int off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    off += (w < warp) ? red[w] : 0;
    tot += red[w];
  }
  __syncthreads();
  *total = tot;
  return off + inc - v;
}

// One block per tile of kTI items, one thread per item.
__global__ void __launch_bounds__(kThreads)
    k_build_tiles(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                  const float *__restrict__ values, int64_t row_begin, int64_t row_end,
                  const int32_t *__restrict__ hot, float *__restrict__ slab,
                  int2 *__restrict__ ell, int32_t *__restrict__ meta,
                  int32_t *__restrict__ heavy_k, float *__restrict__ heavy_v,
                  uint8_t *__restrict__ heavy_item, int32_t *__restrict__ heavy_cursor,
                  int64_t heavy_cap, int32_t *status) {
  extern __shared__ float slab_s[];  // [kHotMax][kTI]
  __shared__ int hkeys[kHotSlots];
  __shared__ int8_t hvals[kHotSlots];
  __shared__ int red[kThreads / 32];
  __shared__ int heavy_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x;
  const int64_t item = row_begin + (int64_t)t * kTI + tid;
  const bool valid = item < row_end;
  const int H = hot[0];
  for (int s = tid; s < kHotSlots; s += kThreads) hkeys[s] = -1;
  __syncthreads();
  if (tid < H) hot_insert(hkeys, hvals, hot[1 + tid], tid);
  for (int h = 0; h < H; ++h) slab_s[h * kTI + tid] = 0.0f;
  __syncthreads();

  int64_t pb = 0, pe = 0;
  if (valid) {
    pb = indptr[item];
    pe = indptr[item + 1];
  }
  int cold = 0;
  for (int64_t p = pb; p < pe; ++p) {
    const int h = hot_find(hkeys, hvals, indices[p]);
    if (h >= 0) slab_s[h * kTI + tid] = values[p];
    else ++cold;
  }
  const int n_valid = block_sum(valid ? 1 : 0, red);
  const int sum_cold = block_sum(cold, red);
  const int mean = n_valid > 0 ? sum_cold / n_valid : 0;
  const int thr = min(kEllMaxW, 2 * mean + 32);
  const bool heavy = cold > thr;
  const int reg_len = heavy ? 0 : cold;
  int len_w = reg_len;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) len_w = max(len_w, __shfl_xor_sync(0xffffffffu, len_w, o));
  int heavy_total = 0;
  const int my_off = block_exclusive_scan(heavy ? cold : 0, red, &heavy_total);
  if (tid == 0) heavy_base = heavy_total > 0 ? atomicAdd(heavy_cursor, heavy_total) : 0;
  __syncthreads();
  const int64_t hbase = heavy_base;
  const bool heavy_ok = hbase + heavy_total <= heavy_cap;
  if (tid == 0 && !heavy_ok) flag(status, DEV_CAPACITY);

  int2 *col = ell + (size_t)t * kEllMaxW * kTI + tid;
  int s = 0;
  for (int64_t p = pb; p < pe; ++p) {
    const int32_t k = indices[p];
    if (hot_find(hkeys, hvals, k) >= 0) continue;
    const float v = values[p];
    if (!heavy) {
      col[(size_t)s * kTI] = make_int2(k, __float_as_int(v));
    } else if (heavy_ok) {
      const int64_t e = hbase + my_off + s;
      heavy_k[e] = k;
      heavy_v[e] = v;
      heavy_item[e] = (uint8_t)tid;
    }
    ++s;
  }
  for (int j = reg_len; j < len_w; ++j) col[(size_t)j * kTI] = make_int2(-1, 0);
  float *dst = slab + (size_t)t * kHotMax * kTI + tid;
  for (int h = 0; h < H; ++h) dst[(size_t)h * kTI] = slab_s[h * kTI + tid];
  int32_t *m = meta + (size_t)t * kMetaInts;
  if (lane == 0) m[warp] = len_w;
  if (tid == 0) {
    m[8] = (int32_t)hbase;
    m[9] = heavy_ok ? heavy_total : 0;
  }
}

// ---------------------------------------------------------------- scorer
struct HybridArgs {
  const int64_t *q_indptr;
  const int32_t *q_idx;
  const float *q_val;
  int64_t n_q;
  const float *inv_q;
  const int32_t *hot;
  const float *slab;
  const int2 *ell;
  const int32_t *meta;
  const int32_t *heavy_k;
  const float *heavy_v;
  const uint8_t *heavy_item;
  const float *inv_i;
  int32_t n_items;
  int32_t n_tiles;
  int64_t n_units;
  float *out;
  int64_t ld_out;
  int32_t vec_ok;
  int32_t dim;
};

// Shared-memory layout of the scoring block (bytes).
constexpr int kOffAcc = 0;
constexpr int kOffSlab = kOffAcc + kTQ * kTI * 4;
constexpr int kOffQhot = kOffSlab + kHotMax * kTI * 4;
constexpr int kOffKeys = kOffQhot + kHotMax * kTQ * 4;
constexpr int kOffMeta = kOffKeys + kHashSlots * 4;
constexpr int kOffLv = kOffMeta + kHashSlots * 4;
constexpr int kOffBits = kOffLv + kBatchEntries * 4;
constexpr int kOffHist = kOffBits + kBitmapWords * 4;
constexpr int kOffHotK = kOffHist + 256 * 4;
constexpr int kOffMisc = kOffHotK + kHotSlots * 4;
constexpr int kOffLq = kOffMisc + 64 * 4;
constexpr int kOffHotV = kOffLq + kBatchEntries;
constexpr int kScoreSmem = kOffHotV + kHotSlots;

struct Smem {
  float *acc, *slab, *qhot, *lv;
  int *keys, *hist, *hotk, *misc;
  uint32_t *hmeta, *bits;
  uint8_t *lq;
  int8_t *hotv;
};

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Queues the copy of one item tile's hot slab (H rows of kTI floats).
__device__ __forceinline__ void slab_prefetch(const Smem &sm, const HybridArgs &a, int t, int H) {
  const float4 *src = reinterpret_cast<const float4 *>(a.slab + (size_t)t * kHotMax * kTI);
  float4 *dst = reinterpret_cast<float4 *>(sm.slab);
  const int n4 = H * kTI / 4;
  for (int j = threadIdx.x; j < n4; j += kThreads) cp_async16(dst + j, src + j);
  cp_async_commit();
}

__device__ __forceinline__ int batch_insert(int *keys, int32_t k) {
  uint32_t s = hash_a(k, kHashBits);
  for (int n = 0; n < kHashSlots; ++n) {
    const int prev = atomicCAS(&keys[s], -1, k);
    if (prev == -1 || prev == k) return (int)s;
    s = (s + 1) & (kHashSlots - 1);
  }
  return -1;
}

// Returns (start << 16 | count) of dimension k's query list, or 0 if k has
// no list in the current batch.
__device__ __forceinline__ uint32_t batch_find(const Smem &sm, int32_t k) {
  const uint32_t b = hash_b(k, kBitmapBits);
  if (!((sm.bits[b >> 5] >> (b & 31)) & 1u)) return 0;
  uint32_t s = hash_a(k, kHashBits);
  for (int n = 0; n < kHashSlots; ++n) {
    const int key = sm.keys[s];
    if (key == k) return sm.hmeta[s];
    if (key == -1) return 0;
    s = (s + 1) & (kHashSlots - 1);
  }
  return 0;
}

// Visits every nonzero of query tile rows [q0, q0 + nq) as f(row, k, v),
// one warp per row.
template <typename F>
__device__ __forceinline__ void for_tile_entries(const HybridArgs &a, int64_t q0, int nq, F f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = warp; r < nq; r += kThreads / 32) {
    const int64_t b = a.q_indptr[q0 + r], e = a.q_indptr[q0 + r + 1];
    for (int64_t p = b + lane; p < e; p += 32) f(r, __ldg(a.q_idx + p), __ldg(a.q_val + p));
  }
}

// Hashes the query tile's cold nonzeros with dims in [lo, hi) (at most
// kBatchEntries of them): dimension -> list of (row, value).
__device__ void build_batch(const Smem &sm, const HybridArgs &a, int64_t q0, int nq, int32_t lo,
                            int32_t hi) {
  for (int s = threadIdx.x; s < kHashSlots; s += kThreads) {
    sm.keys[s] = -1;
    sm.hmeta[s] = 0;
  }
  for (int w = threadIdx.x; w < kBitmapWords; w += kThreads) sm.bits[w] = 0;
  __syncthreads();
  for_tile_entries(a, q0, nq, [&](int, int32_t k, float) {
    if (k < lo || k >= hi || hot_find(sm.hotk, sm.hotv, k) >= 0) return;
    const int s = batch_insert(sm.keys, k);
    if (s < 0) return;
    atomicAdd(&sm.hmeta[s], 1u);
    const uint32_t b = hash_b(k, kBitmapBits);
    atomicOr(&sm.bits[b >> 5], 1u << (b & 31));
  });
  __syncthreads();
  // Exclusive scan of the list lengths: kHashSlots / kThreads slots each.
  constexpr int kPer = kHashSlots / kThreads;
  uint32_t c[kPer];
  int local = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    c[j] = sm.hmeta[threadIdx.x * kPer + j] & 0xffffu;
    local += (int)c[j];
  }
  int total;
  int start = block_exclusive_scan(local, sm.misc + 16, &total);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    sm.hmeta[threadIdx.x * kPer + j] = ((uint32_t)start << 16) | c[j];
    start += (int)c[j];
  }
  __syncthreads();
  for_tile_entries(a, q0, nq, [&](int r, int32_t k, float v) {
    if (k < lo || k >= hi || hot_find(sm.hotk, sm.hotv, k) >= 0) return;
    uint32_t s = hash_a(k, kHashBits);
    bool found = false;
    for (int n = 0; n < kHashSlots && !found; ++n) {
      if (sm.keys[s] == k) found = true;
      else s = (s + 1) & (kHashSlots - 1);
    }
    if (!found) return;
    const uint32_t pos = atomicAdd(&sm.hmeta[s], 1u << 16) >> 16;
    if (pos < (uint32_t)kBatchEntries) {
      sm.lq[pos] = (uint8_t)r;
      sm.lv[pos] = v;
    }
  });
  __syncthreads();
  // The fill advanced each start by its count: move it back.
  for (int s = threadIdx.x; s < kHashSlots; s += kThreads) {
    const uint32_t m = sm.hmeta[s], cnt = m & 0xffffu;
    if (cnt) sm.hmeta[s] = (((m >> 16) - cnt) << 16) | cnt;
  }
  __syncthreads();
}

// Largest hi such that the query tile has at most kBatchEntries cold
// nonzeros with dims in [lo, hi): histogram the remaining range into 256
// buckets, take the longest prefix that fits, else narrow to the first
// bucket and repeat (a single dim has at most kTQ nonzeros, so it ends).
__device__ int32_t plan_batch(const Smem &sm, const HybridArgs &a, int64_t q0, int nq, int32_t lo) {
  int64_t span = (int64_t)a.dim - lo;
  for (;;) {
    const int64_t w = (span + 255) / 256;
    for (int b = threadIdx.x; b < 256; b += kThreads) sm.hist[b] = 0;
    __syncthreads();
    for_tile_entries(a, q0, nq, [&](int, int32_t k, float) {
      if (k < lo || (int64_t)k >= lo + span || hot_find(sm.hotk, sm.hotv, k) >= 0) return;
      atomicAdd(&sm.hist[(k - lo) / w], 1);
    });
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0, b = 0;
      while (b < 256 && acc + sm.hist[b] <= kBatchEntries) acc += sm.hist[b++];
      if (b > 0) {
        sm.misc[0] = 1;
        const int64_t end = lo + (int64_t)b * w;
        sm.misc[1] = (int)(end < lo + span ? end : lo + span);
      } else {
        sm.misc[0] = 0;
        sm.misc[1] = (int)w;
      }
    }
    __syncthreads();
    const int done = sm.misc[0], val = sm.misc[1];
    __syncthreads();
    if (done) return val;
    span = val;
  }
}

// Dense product over the hot dims: thread (lq, li) of warp (wq, wi) owns
// queries wq*32 + lq*8 + [0, 8) and items wi*64 + li*8 + [0, 8).
__device__ __forceinline__ void hot_product(const Smem &sm, int H) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int qb = (warp & 1) * 32 + (lane >> 3) * 8;
  const int ib = (warp >> 1) * 64 + (lane & 7) * 8;
  float2 c[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int j = 0; j < 4; ++j) c[r][j] = make_float2(0.f, 0.f);
  for (int h = 0; h < H; ++h) {
    const float4 qa = *reinterpret_cast<const float4 *>(sm.qhot + h * kTQ + qb);
    const float4 qc = *reinterpret_cast<const float4 *>(sm.qhot + h * kTQ + qb + 4);
    const float4 ia = *reinterpret_cast<const float4 *>(sm.slab + h * kTI + ib);
    const float4 ic = *reinterpret_cast<const float4 *>(sm.slab + h * kTI + ib + 4);
    const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qc.x, qc.y, qc.z, qc.w};
    const float2 i0 = make_float2(ia.x, ia.y), i1 = make_float2(ia.z, ia.w);
    const float2 i2 = make_float2(ic.x, ic.y), i3 = make_float2(ic.z, ic.w);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float2 qq = make_float2(qv[r], qv[r]);
      c[r][0] = __ffma2_rn(qq, i0, c[r][0]);
      c[r][1] = __ffma2_rn(qq, i1, c[r][1]);
      c[r][2] = __ffma2_rn(qq, i2, c[r][2]);
      c[r][3] = __ffma2_rn(qq, i3, c[r][3]);
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float4 *d = reinterpret_cast<float4 *>(sm.acc + (qb + r) * kTI + ib);
    d[0] = make_float4(c[r][0].x, c[r][0].y, c[r][1].x, c[r][1].y);
    d[1] = make_float4(c[r][2].x, c[r][2].y, c[r][3].x, c[r][3].y);
  }
}

// Cold nonzeros of item tile t with dims in [lo, hi).  `cursor` is this
// thread's position in its item's ELL column (kept across batches).
__device__ __forceinline__ void cold_pass(const Smem &sm, const HybridArgs &a, int t, int32_t lo,
                                          int32_t hi, int &cursor) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int32_t *m = a.meta + (size_t)t * kMetaInts;
  const int len = m[warp];
  const int2 *col = a.ell + (size_t)t * kEllMaxW * kTI + tid;
  float *accc = sm.acc + tid;
  int s = cursor;
  while (s < len) {
    const int2 x = __ldg(col + (size_t)s * kTI);
    if (x.x < 0 || x.x >= hi) break;
    ++s;
    const uint32_t hm = batch_find(sm, x.x);
    const uint32_t cnt = hm & 0xffffu;
    if (!cnt) continue;
    const float v = __int_as_float(x.y);
    const uint32_t st = hm >> 16;
    for (uint32_t e = st; e < st + cnt; ++e) {
      float *dst = accc + sm.lq[e] * kTI;
      *dst = fmaf(sm.lv[e], v, *dst);
    }
  }
  cursor = s;
  // Heavy items: their nonzeros are spread over all threads; several
  // threads may add into one accumulator, hence the atomics.
  const int hb = m[8], hc = m[9];
  for (int e = hb + tid; e < hb + hc; e += kThreads) {
    const int32_t k = __ldg(a.heavy_k + e);
    if (k < lo || k >= hi) continue;
    const uint32_t hm = batch_find(sm, k);
    const uint32_t cnt = hm & 0xffffu;
    if (!cnt) continue;
    const float v = __ldg(a.heavy_v + e);
    const int it = __ldg(a.heavy_item + e);
    const uint32_t st = hm >> 16;
    for (uint32_t j = st; j < st + cnt; ++j) atomicAdd(sm.acc + sm.lq[j] * kTI + it, sm.lv[j] * v);
  }
}

__device__ __forceinline__ void store_tile(const Smem &sm, const HybridArgs &a, int64_t q0, int nq,
                                           int t) {
  const int tid = threadIdx.x;
  const int i0 = t * kTI;
  const int ni = min(kTI, a.n_items - i0);
  const int c = (tid & 63) * 4;
  if (c >= ni) return;
  float n[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) n[j] = (c + j < ni) ? __ldg(a.inv_i + i0 + c + j) : 0.f;
  const bool vec = a.vec_ok && (c + 4 <= ni);
  for (int r = tid >> 6; r < nq; r += kThreads / 64) {
    const float4 v = *reinterpret_cast<const float4 *>(sm.acc + r * kTI + c);
    const float iq = __ldg(a.inv_q + q0 + r);
    float *dst = a.out + (q0 + r) * a.ld_out + i0 + c;
    const float o0 = v.x * iq * n[0], o1 = v.y * iq * n[1], o2 = v.z * iq * n[2], o3 = v.w * iq * n[3];
    if (vec) {
      __stcs(reinterpret_cast<float4 *>(dst), make_float4(o0, o1, o2, o3));
    } else {
      const float o[4] = {o0, o1, o2, o3};
      for (int j = 0; j < 4 && c + j < ni; ++j) dst[j] = o[j];
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_score_hybrid(const HybridArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem sm;
  sm.acc = reinterpret_cast<float *>(smem_raw + kOffAcc);
  sm.slab = reinterpret_cast<float *>(smem_raw + kOffSlab);
  sm.qhot = reinterpret_cast<float *>(smem_raw + kOffQhot);
  sm.keys = reinterpret_cast<int *>(smem_raw + kOffKeys);
  sm.hmeta = reinterpret_cast<uint32_t *>(smem_raw + kOffMeta);
  sm.lv = reinterpret_cast<float *>(smem_raw + kOffLv);
  sm.bits = reinterpret_cast<uint32_t *>(smem_raw + kOffBits);
  sm.hist = reinterpret_cast<int *>(smem_raw + kOffHist);
  sm.hotk = reinterpret_cast<int *>(smem_raw + kOffHotK);
  sm.misc = reinterpret_cast<int *>(smem_raw + kOffMisc);
  sm.lq = smem_raw + kOffLq;
  sm.hotv = reinterpret_cast<int8_t *>(smem_raw + kOffHotV);
  const int tid = threadIdx.x;

  const int H = a.hot[0];
  for (int s = tid; s < kHotSlots; s += kThreads) sm.hotk[s] = -1;
  __syncthreads();
  if (tid < H) hot_insert(sm.hotk, sm.hotv, a.hot[1 + tid], tid);
  __syncthreads();

  const int64_t u0 = (int64_t)blockIdx.x * a.n_units / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * a.n_units / gridDim.x;
  int64_t cur_g = -1;
  bool single = false;
  if (H > 0 && u0 < u1) slab_prefetch(sm, a, (int)(u0 % a.n_tiles), H);
  for (int64_t u = u0; u < u1; ++u) {
    const int64_t g = u / a.n_tiles;
    const int t = (int)(u % a.n_tiles);
    const int64_t q0 = g * kTQ;
    const int nq = (int)(a.n_q - q0 < kTQ ? a.n_q - q0 : kTQ);
    if (g != cur_g) {
      cur_g = g;
      for (int j = tid; j < H * kTQ; j += kThreads) sm.qhot[j] = 0.f;
      if (tid == 0) sm.misc[2] = 0;
      __syncthreads();
      int n_cold = 0;
      for_tile_entries(a, q0, nq, [&](int r, int32_t k, float v) {
        const int h = hot_find(sm.hotk, sm.hotv, k);
        if (h >= 0) sm.qhot[h * kTQ + r] = v;
        else ++n_cold;
      });
      atomicAdd(&sm.misc[2], n_cold);
      __syncthreads();
      single = sm.misc[2] <= kBatchEntries;
      __syncthreads();
      if (single) build_batch(sm, a, q0, nq, 0, a.dim);
    }
    // 1. hot dims: dense product into the accumulator tile
    if (H > 0) {
      cp_async_wait_all();
      __syncthreads();
      hot_product(sm, H);
    } else {
      float4 *acc4 = reinterpret_cast<float4 *>(sm.acc);
      for (int j = tid; j < kTQ * kTI / 4; j += kThreads) acc4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    if (H > 0 && u + 1 < u1) slab_prefetch(sm, a, (int)((u + 1) % a.n_tiles), H);
    // 2. cold dims through the hashed query lists
    int cursor = 0;
    if (single) {
      cold_pass(sm, a, t, 0, a.dim, cursor);
    } else {
      for (int32_t lo = 0; lo < a.dim;) {
        const int32_t hi = plan_batch(sm, a, q0, nq, lo);
        build_batch(sm, a, q0, nq, lo, hi);
        cold_pass(sm, a, t, lo, hi, cursor);
        __syncthreads();
        lo = hi;
      }
    }
    __syncthreads();
    // 3. normalise and store
    store_tile(sm, a, q0, nq, t);
    __syncthreads();
  }
  cp_async_wait_all();
}

}  // namespace

cudaError_t launch_hot_select(ss_handle *h, const ss_csr &items, cudaStream_t s, int *queued) {
  *queued = 0;
  if (h->hot_src[0] == items.indptr && h->hot_src[1] == items.indices &&
      h->hot_src[2] == items.values && h->hot_src_rows == items.n_rows &&
      h->hot_src_nnz == items.nnz)
    return cudaSuccess;
  const int64_t n = items.n_rows;
  int64_t n_sample = 0;
  if (n > 0 && items.nnz > 0) {
    n_sample = (int64_t)((double)kHotSampleEntries * (double)n / (double)items.nnz);
    n_sample = std::max<int64_t>(16, std::min<int64_t>(n, n_sample));
  }
  if (n_sample == 0) {
    cudaError_t e = cudaMemsetAsync(h->hot, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
  } else {
    const size_t smem = sizeof(int) * 2 * kSelSlots;
    static bool configured = false;
    if (!configured) {
      cudaError_t e = cudaFuncSetAttribute(k_hot_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
      configured = true;
    }
    k_hot_select<<<1, kSelThreads, smem, s>>>(items.indptr, items.indices, n, n_sample, h->hot);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *queued = 1;
  }
  h->hot_src[0] = items.indptr;
  h->hot_src[1] = items.indices;
  h->hot_src[2] = items.values;
  h->hot_src_rows = items.n_rows;
  h->hot_src_nnz = items.nnz;
  return cudaSuccess;
}

cudaError_t launch_build_hybrid(ss_handle *h, const ss_csr &items, int64_t row_begin,
                                int64_t row_end, cudaStream_t s) {
  const int n_items = (int)(row_end - row_begin);
  const int n_tiles = (n_items + kTI - 1) / kTI;
  cudaError_t e = cudaMemsetAsync(h->heavy_cursor, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(float) * kHotMax * kTI;
  static bool configured = false;
  if (!configured) {
    e = cudaFuncSetAttribute(k_build_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k_build_tiles<<<n_tiles, kThreads, smem, s>>>(
      items.indptr, items.indices, items.values, row_begin, row_end, h->hot, h->slab, h->ell,
      h->meta, h->heavy_k, h->heavy_v, h->heavy_item, h->heavy_cursor, h->heavy_cap, h->d_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ss_index &ix = h->index;
  ix.algo = ALGO_HYBRID;
  ix.row_begin = row_begin;
  ix.row_end = row_end;
  ix.n_items = n_items;
  ix.dim = h->dim;
  ix.n_tiles = n_tiles;
  ix.hot = h->hot;
  ix.slab = h->slab;
  ix.ell = h->ell;
  ix.meta = h->meta;
  ix.heavy_k = h->heavy_k;
  ix.heavy_v = h->heavy_v;
  ix.heavy_item = h->heavy_item;
  return cudaSuccess;
}

cudaError_t launch_score_hybrid(const ss_handle *h, const ss_csr &queries, const float *inv_q,
                                const ss_index &idx, const float *inv_i, float *out,
                                int64_t ld_out, cudaStream_t s) {
  if (queries.n_rows == 0 || idx.n_items == 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_score_hybrid, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kScoreSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  HybridArgs a;
  a.q_indptr = queries.indptr;
  a.q_idx = queries.indices;
  a.q_val = queries.values;
  a.n_q = queries.n_rows;
  a.inv_q = inv_q;
  a.hot = idx.hot;
  a.slab = idx.slab;
  a.ell = idx.ell;
  a.meta = idx.meta;
  a.heavy_k = idx.heavy_k;
  a.heavy_v = idx.heavy_v;
  a.heavy_item = idx.heavy_item;
  a.inv_i = inv_i;
  a.n_items = idx.n_items;
  a.n_tiles = idx.n_tiles;
  const int64_t n_qtiles = (queries.n_rows + kTQ - 1) / kTQ;
  a.n_units = n_qtiles * idx.n_tiles;
  if (a.n_units == 0) return cudaSuccess;
  a.out = out;
  a.ld_out = ld_out;
  a.vec_ok = ((reinterpret_cast<uintptr_t>(out) % 16) == 0) && (ld_out % 4 == 0);
  a.dim = (int32_t)idx.dim;
  const int grid = (int)std::min<int64_t>(a.n_units, h->sm_count > 0 ? h->sm_count : 148);
  k_score_hybrid<<<grid, kThreads, kScoreSmem, s>>>(a);
  return cudaGetLastError();
}
