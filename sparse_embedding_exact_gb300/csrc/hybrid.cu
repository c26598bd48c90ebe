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

// Open-addressing insert / find in the image-building hash (kImgSlots).
__device__ __forceinline__ int img_insert(int *keys, int32_t k) {
  uint32_t s = hash_a(k, kImgSlotsBits);
  for (int n = 0; n < kImgSlots; ++n) {
    const int prev = atomicCAS(&keys[s], -1, k);
    if (prev == -1 || prev == k) return (int)s;
    s = (s + 1) & (kImgSlots - 1);
  }
  return -1;
}
__device__ __forceinline__ int img_find(const int *keys, int32_t k) {
  uint32_t s = hash_a(k, kImgSlotsBits);
  for (int n = 0; n < kImgSlots; ++n) {
    const int key = keys[s];
    if (key == k) return (int)s;
    if (key == -1) return -1;
    s = (s + 1) & (kImgSlots - 1);
  }
  return -1;
}

// Shared memory of the builder block (bytes).
constexpr int kBThreads = 1024;  // builder: 32 warps, one item row per warp at a time
constexpr int kBldOffSlab = 0;
constexpr int kBldOffKeys = kBldOffSlab + kHotMax * kTI * 4;
constexpr int kBldOffCnt = kBldOffKeys + kImgSlots * 4;
constexpr int kBldOffCold = kBldOffCnt + kImgSlots * 4;  // cold nonzeros per item
constexpr int kBuildSmem = kBldOffCold + kTI * 4;

__device__ __forceinline__ int bblock_sum(int v, int *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < kBThreads / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ int bblock_exclusive_scan(int v, int *red, int *total) {
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
  for (int w = 0; w < kBThreads / 32; ++w) {
    off += (w < warp) ? red[w] : 0;
    tot += red[w];
  }
  __syncthreads();
  *total = tot;
  return off + inc - v;
}

// One block per tile of kTI items; warp w handles items w, w + 32, ..., its
// lanes taking the row's nonzeros 32 at a time (coalesced).  Hot values go
// to the tile's slab.  The cold nonzeros become the tile's image (dimension
// -> segment of (item, value)) when they fit; otherwise they go to the ELL
// block and the heavy list, and the tile joins the overflow list.
__global__ void __launch_bounds__(kBThreads, 1)
    k_build_tiles(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                  const float *__restrict__ values, int64_t row_begin, int64_t row_end,
                  const int32_t *__restrict__ hot, float *__restrict__ slab,
                  int2 *__restrict__ ell, int32_t *__restrict__ meta,
                  int32_t *__restrict__ heavy_k, float *__restrict__ heavy_v,
                  uint8_t *__restrict__ heavy_item, int32_t *__restrict__ counters,
                  int64_t heavy_cap, unsigned char *__restrict__ image, int32_t *status) {
  extern __shared__ __align__(16) unsigned char bsm[];
  float *slab_s = reinterpret_cast<float *>(bsm + kBldOffSlab);  // [kHotMax][kTI]
  int *ikeys = reinterpret_cast<int *>(bsm + kBldOffKeys);
  int *icnt = reinterpret_cast<int *>(bsm + kBldOffCnt);
  int *cold_n = reinterpret_cast<int *>(bsm + kBldOffCold);
  __shared__ int hkeys[kHotSlots];
  __shared__ int8_t hvals[kHotSlots];
  __shared__ int red[kBThreads / 32];
  __shared__ int heavy_base, img_fail;
  __shared__ int heavy_off[kTI];
  __shared__ uint32_t bits_s[(1 << kImgBitsLog2) / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int w = tid; w < (1 << kImgBitsLog2) / 32; w += kBThreads) bits_s[w] = 0u;
  const int t = blockIdx.x;
  const int64_t item0 = row_begin + (int64_t)t * kTI;
  const int n_items = (int)min((int64_t)kTI, row_end - item0);
  const int H = hot[0];
  for (int s = tid; s < kHotSlots; s += kBThreads) hkeys[s] = -1;
  for (int s = tid; s < kImgSlots; s += kBThreads) {
    ikeys[s] = -1;
    icnt[s] = 0;
  }
  for (int j = tid; j < H * kTI; j += kBThreads) slab_s[j] = 0.0f;
  if (tid == 0) img_fail = 0;
  __syncthreads();
  if (tid < H) hot_insert(hkeys, hvals, hot[1 + tid], tid);
  __syncthreads();

  // Pass 1: hot values into the slab; cold dims into the image hash.
  for (int it = warp; it < kTI; it += kBThreads / 32) {
    int cold = 0;
    if (it < n_items) {
      const int64_t pb = indptr[item0 + it], pe = indptr[item0 + it + 1];
      for (int64_t p = pb + lane; p < pe; p += 32) {
        const int32_t k = __ldg(indices + p);
        const int h = hot_find(hkeys, hvals, k);
        if (h >= 0) {
          slab_s[h * kTI + it] = __ldg(values + p);
        } else {
          ++cold;
          const int slot = img_insert(ikeys, k);
          if (slot < 0) img_fail = 1;
          else atomicAdd(&icnt[slot], 1);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cold += __shfl_xor_sync(0xffffffffu, cold, o);
    if (lane == 0) cold_n[it] = cold;
  }
  __syncthreads();
  const int my_cold = tid < kTI ? cold_n[tid] : 0;
  const int sum_cold = bblock_sum(my_cold, red);
  unsigned char *img = image + (size_t)t * kImgBytes;
  int32_t *hdr = reinterpret_cast<int32_t *>(img);

  // ---- image path
  constexpr int kPer = kImgSlots / kBThreads;
  int occ = 0, ent = 0;
  for (int j = 0; j < kPer; ++j) {
    const int s = tid * kPer + j;
    occ += ikeys[s] >= 0;
    ent += icnt[s];
  }
  int D = 0, E = 0;
  (void)bblock_exclusive_scan(occ, red, &D);
  int e_run = bblock_exclusive_scan(ent, red, &E);
  const bool fits = !img_fail && sum_cold <= kImgECap && D <= kImgDCap && E == sum_cold;
  if (fits) {
    uint2 *gslot = reinterpret_cast<uint2 *>(img + kImgOffSlots);
    for (int j = 0; j < kPer; ++j) {
      const int s = tid * kPer + j;
      if (ikeys[s] >= 0) {
        const int c = icnt[s];
        gslot[s] = make_uint2((uint32_t)ikeys[s], (uint32_t)e_run | ((uint32_t)(e_run + c) << 16));
        icnt[s] = e_run;  // now the fill cursor of this segment
        e_run += c;
        const uint32_t bb = hash_b(ikeys[s], kImgBitsLog2);
        atomicOr(&bits_s[bb >> 5], 1u << (bb & 31));
      } else {
        gslot[s] = make_uint2(0xffffffffu, 0u);
      }
    }
    if (tid == 0) {
      hdr[0] = D;
      hdr[1] = E;
      hdr[2] = 1;
      hdr[3] = 0;
    }
    __syncthreads();
    uint32_t *gbits = reinterpret_cast<uint32_t *>(img + kImgOffBits);
    for (int w = tid; w < (1 << kImgBitsLog2) / 32; w += kBThreads) gbits[w] = bits_s[w];
    uint8_t *gitem = img + kImgOffItem;
    float *gval = reinterpret_cast<float *>(img + kImgOffVal);
    for (int it = warp; it < n_items; it += kBThreads / 32) {
      const int64_t pb = indptr[item0 + it], pe = indptr[item0 + it + 1];
      for (int64_t p = pb + lane; p < pe; p += 32) {
        const int32_t k = __ldg(indices + p);
        if (hot_find(hkeys, hvals, k) >= 0) continue;
        const int pos = atomicAdd(&icnt[img_find(ikeys, k)], 1);
        gitem[pos] = (uint8_t)it;
        gval[pos] = __ldg(values + p);
      }
    }
  }

  // ---- ELL path for tiles whose cold part does not fit an image
  int32_t *m = meta + (size_t)t * kMetaInts;
  int heavy_total = 0;
  bool heavy_ok = true;
  if (!fits) {
    // Items far above the tile's mean go to the heavy list.
    const int mean = n_items > 0 ? sum_cold / n_items : 0;
    const int thr = min(kEllMaxW, 2 * mean + 32);
    const bool my_heavy = tid < n_items && my_cold > thr;
    const int off = bblock_exclusive_scan(my_heavy ? my_cold : 0, red, &heavy_total);
    if (tid < kTI) heavy_off[tid] = my_heavy ? off : -1;
    if (tid == 0) {
      heavy_base = heavy_total > 0 ? atomicAdd(&counters[0], heavy_total) : 0;
      hdr[2] = 0;
      const int c = atomicAdd(&counters[1], 1);
      counters[2 + c] = t;
    }
    __syncthreads();
    const int64_t hbase = heavy_base;
    heavy_ok = hbase + heavy_total <= heavy_cap;
    if (tid == 0 && !heavy_ok) flag(status, DEV_CAPACITY);
    // ELL width of each warp group of 32 items: the longest regular row.
    if (tid < kTI) {
      int len = heavy_off[tid] < 0 ? cold_n[tid] : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) len = max(len, __shfl_xor_sync(0xffffffffu, len, o));
      if (lane == 0) m[warp] = len;
      if (lane == 0) red[warp] = len;
    }
    __syncthreads();
    for (int it = warp; it < kTI; it += kBThreads / 32) {
      const int hoff = heavy_off[it];
      const int len_w = red[it >> 5];
      int2 *col = ell + (size_t)t * kEllMaxW * kTI + it;
      int s = 0;
      if (it < n_items) {
        const int64_t pb = indptr[item0 + it], pe = indptr[item0 + it + 1];
        for (int64_t p = pb; p < pe; p += 32) {
          const int64_t pp = p + lane;
          int32_t k = -1;
          bool is_cold = false;
          if (pp < pe) {
            k = __ldg(indices + pp);
            is_cold = hot_find(hkeys, hvals, k) < 0;
          }
          const unsigned cm = __ballot_sync(0xffffffffu, is_cold);
          const int pos = s + __popc(cm & lt_mask);
          if (is_cold) {
            const float v = __ldg(values + pp);
            if (hoff < 0) {
              col[(size_t)pos * kTI] = make_int2(k, __float_as_int(v));
            } else if (heavy_ok) {
              const int64_t e = hbase + hoff + pos;
              heavy_k[e] = k;
              heavy_v[e] = v;
              heavy_item[e] = (uint8_t)it;
            }
          }
          s += __popc(cm);
        }
      }
      const int reg_len = hoff < 0 ? s : 0;
      for (int j = reg_len + lane; j < len_w; j += 32) col[(size_t)j * kTI] = make_int2(-1, 0);
    }
    if (tid == 0) m[8] = (int32_t)hbase;
  } else if (tid < 8) {
    m[tid] = 0;
  }
  __syncthreads();
  float *dst = slab + (size_t)t * kHotMax * kTI;
  for (int j = tid; j < H * kTI; j += kBThreads) dst[j] = slab_s[j];
  if (tid == 0) {
    if (fits) m[8] = 0;
    m[9] = (!fits && heavy_ok) ? heavy_total : 0;
    m[kMetaFits] = fits ? 1 : 0;
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
  int64_t n_qtiles;
  const int32_t *counters;  // [1] tiles without an image, [2..] their ids
  float *out;
  int64_t ld_out;
  int32_t vec_ok;
  int32_t dim;
};

constexpr int kQueue = 8;  // cold entries probed per step; their hits queue per thread

// Shared-memory layout of the scoring block (bytes).
constexpr int kOffAcc = 0;
constexpr int kOffSlab = kOffAcc + kTQ * kTI * 4;
constexpr int kOffQhot = kOffSlab + kHotMax * kTI * 4;
constexpr int kOffKeys = kOffQhot + kHotMax * kTQ * 4;
constexpr int kOffMeta = kOffKeys + kHashSlots * 4;
constexpr int kOffLists = kOffMeta + kHashSlots * 4;
constexpr int kOffQueue = kOffLists + kBatchEntries * 8;
constexpr int kOffBits = kOffQueue + kQueue * kThreads * 8;
constexpr int kOffHist = kOffBits + kBitmapWords * 4;
constexpr int kOffHotK = kOffHist + 256 * 4;
constexpr int kOffMisc = kOffHotK + kHotSlots * 4;
constexpr int kOffHotV = kOffMisc + 64 * 4;
constexpr int kScoreSmem = kOffHotV + kHotSlots;
static_assert(kScoreSmem <= 232448, "scoring block exceeds 227 KB of shared memory");

struct Smem {
  float *acc, *slab, *qhot;
  int *keys, *hist, *hotk, *misc;
  uint32_t *hmeta, *bits;
  uint2 *lists;  // query lists: {row * kTI, value bits}
  uint2 *queue;  // per-thread hit queue: entry j of thread t at [j * kThreads + t]
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
    if (pos < (uint32_t)kBatchEntries) sm.lists[pos] = make_uint2((uint32_t)(r * kTI), __float_as_uint(v));
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

// Slot of dimension k in the batch hash, resolved past the first probe.
__device__ __noinline__ uint32_t batch_find_slow(const Smem &sm, int32_t k, uint32_t s) {
  for (int n = 1; n < kHashSlots; ++n) {
    s = (s + 1) & (kHashSlots - 1);
    const int key = sm.keys[s];
    if (key == k) return sm.hmeta[s];
    if (key == -1) return 0;
  }
  return 0;
}

// Cold nonzeros of item tile t with dims in [lo, hi).  `cursor` is this
// thread's position in its item's ELL column (kept across batches).
//
// Thread i owns item i (column i of the accumulator tile).  It takes its
// ELL entries kQueue at a time: the loads of the next group are in flight
// while the current one is probed, the kQueue probes are independent, and
// the hits go into the thread's queue.  The thread then walks all queued
// query lists in one loop, so a warp waits for its busiest lane's total,
// not for the longest list at every step.  Hits are queued and walked in
// ascending dimension order, which fixes the order of each entry's sum.
__device__ __forceinline__ void cold_pass(const Smem &sm, const HybridArgs &a, int t, int32_t lo,
                                          int32_t hi, int &cursor) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int32_t *m = a.meta + (size_t)t * kMetaInts;
  const int len = m[warp];
  const int2 *col = a.ell + (size_t)t * kEllMaxW * kTI + tid;
  float *accc = sm.acc + tid;
  uint2 *queue = sm.queue + tid;
  int s = cursor;
  bool active = s < len;
  int2 x[kQueue];
#pragma unroll
  for (int j = 0; j < kQueue; ++j)
    x[j] = (active && s + j < len) ? __ldg(col + (size_t)(s + j) * kTI) : make_int2(-1, 0);
  while (__any_sync(0xffffffffu, active)) {
    // Probe: entries are a prefix of valid dims (< hi), then pads / later dims.
    bool in[kQueue];
    uint32_t bit[kQueue], slot[kQueue];
    int consumed = 0;
#pragma unroll
    for (int j = 0; j < kQueue; ++j) {
      in[j] = active && x[j].x >= 0 && x[j].x < hi;
      if (in[j]) consumed = j + 1;
      const uint32_t b = hash_b(x[j].x, kBitmapBits);
      bit[j] = in[j] ? ((sm.bits[b >> 5] >> (b & 31)) & 1u) : 0u;
      slot[j] = hash_a(x[j].x, kHashBits);
    }
    uint32_t hm[kQueue];
#pragma unroll
    for (int j = 0; j < kQueue; ++j) {
      hm[j] = 0;
      if (bit[j]) {
        const int key = sm.keys[slot[j]];
        if (key == x[j].x) hm[j] = sm.hmeta[slot[j]];
        else if (key != -1) hm[j] = batch_find_slow(sm, x[j].x, slot[j]);
      }
    }
    int nh = 0;
#pragma unroll
    for (int j = 0; j < kQueue; ++j) {
      if (hm[j] & 0xffffu) {
        queue[nh * kThreads] = make_uint2(hm[j], (uint32_t)x[j].y);
        ++nh;
      }
    }
    s += consumed;
    if (consumed < kQueue || s >= len) active = false;
#pragma unroll
    for (int j = 0; j < kQueue; ++j)
      x[j] = (active && s + j < len) ? __ldg(col + (size_t)(s + j) * kTI) : make_int2(-1, 0);
    // Walk the queued lists: acc[q][i] += q_k * v_ik.
    int h = 0;
    uint32_t st = 0, end = 0;
    float v = 0.f;
    if (nh > 0) {
      const uint2 e0 = queue[0];
      st = e0.x >> 16;
      end = st + (e0.x & 0xffffu);
      v = __uint_as_float(e0.y);
    }
    while (__any_sync(0xffffffffu, h < nh)) {
      if (h < nh) {
        const uint2 e = sm.lists[st];
        float *d = accc + e.x;
        *d = fmaf(__uint_as_float(e.y), v, *d);
        if (++st == end) {
          if (++h < nh) {
            const uint2 en = queue[h * kThreads];
            st = en.x >> 16;
            end = st + (en.x & 0xffffu);
            v = __uint_as_float(en.y);
          }
        }
      }
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
    for (uint32_t j = st; j < st + cnt; ++j) {
      const uint2 l = sm.lists[j];
      atomicAdd(sm.acc + l.x + it, __uint_as_float(l.y) * v);
    }
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
  sm.lists = reinterpret_cast<uint2 *>(smem_raw + kOffLists);
  sm.queue = reinterpret_cast<uint2 *>(smem_raw + kOffQueue);
  sm.bits = reinterpret_cast<uint32_t *>(smem_raw + kOffBits);
  sm.hist = reinterpret_cast<int *>(smem_raw + kOffHist);
  sm.hotk = reinterpret_cast<int *>(smem_raw + kOffHotK);
  sm.misc = reinterpret_cast<int *>(smem_raw + kOffMisc);
  sm.hotv = reinterpret_cast<int8_t *>(smem_raw + kOffHotV);
  const int tid = threadIdx.x;

  const int H = a.hot[0];
  for (int s = tid; s < kHotSlots; s += kThreads) sm.hotk[s] = -1;
  __syncthreads();
  if (tid < H) hot_insert(sm.hotk, sm.hotv, a.hot[1 + tid], tid);
  __syncthreads();

  // Only the item tiles that have no image (the builder's overflow list).
  const int n_ovf = a.counters[1];
  const int32_t *ovf = a.counters + 2;
  const int64_t n_units = a.n_qtiles * n_ovf;
  const int64_t u0 = (int64_t)blockIdx.x * n_units / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * n_units / gridDim.x;
  int64_t cur_g = -1;
  bool single = false;
  if (H > 0 && u0 < u1) slab_prefetch(sm, a, ovf[u0 % n_ovf], H);
  for (int64_t u = u0; u < u1; ++u) {
    const int64_t g = u / n_ovf;
    const int t = ovf[u % n_ovf];
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
    if (H > 0 && u + 1 < u1) slab_prefetch(sm, a, ovf[(u + 1) % n_ovf], H);
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

// ---------------------------------------------------------------- fast path
// One warp per query row: the row's hot values into its column of the query
// tile's hot block ([tile][kHotMax][kTQ], zero where absent), and the row's
// cold nonzeros as {dim, value bits}, in their original (ascending) order,
// moved to the front of the row's own range, with their count.  Rows past
// n_q in the last tile get a zero column.
__global__ void __launch_bounds__(kThreads)
    k_prep_queries(const int64_t *__restrict__ indptr, const int32_t *__restrict__ idx,
                   const float *__restrict__ val, int64_t n_q, int64_t n_rows_padded,
                   const int32_t *__restrict__ hot, float *__restrict__ qhot,
                   int2 *__restrict__ qcold, int32_t *__restrict__ qcold_n) {
  __shared__ int hkeys[kHotSlots];
  __shared__ int8_t hvals[kHotSlots];
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int H = hot[0];
  for (int s = threadIdx.x; s < kHotSlots; s += kThreads) hkeys[s] = -1;
  __syncthreads();
  if ((int)threadIdx.x < H) hot_insert(hkeys, hvals, hot[1 + threadIdx.x], threadIdx.x);
  __syncthreads();
  const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
  for (int64_t q = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); q < n_rows_padded;
       q += warps) {
    float *col = qhot + (q / kTQ) * kHotMax * kTQ + (q % kTQ);
    for (int h = lane; h < kHotMax; h += 32) col[h * kTQ] = 0.f;
    __syncwarp();
    if (q >= n_q) continue;
    const int64_t b = indptr[q], e = indptr[q + 1];
    int n = 0;
    for (int64_t p0 = b; p0 < e; p0 += 32) {
      const int64_t p = p0 + lane;
      int32_t k = -1;
      float v = 0.f;
      int h = -1;
      if (p < e) {
        k = idx[p];
        v = val[p];
        h = hot_find(hkeys, hvals, k);
        if (h >= 0) col[h * kTQ] = v;
      }
      const bool cold = p < e && h < 0;
      const unsigned m = __ballot_sync(0xffffffffu, cold);
      if (cold) qcold[b + n + __popc(m & lt_mask)] = make_int2(k, __float_as_int(v));
      n += __popc(m);
    }
    if (lane == 0) qcold_n[q] = n;
  }
}

struct TileArgs {
  const int64_t *q_indptr;
  const int2 *qcold;
  const int32_t *qcold_n;
  int64_t n_q;
  const float *inv_q;
  const float *qhot;
  const int32_t *hot;
  const float *slab;
  const int32_t *meta;
  const unsigned char *image;
  const float *inv_i;
  int32_t n_items;
  int32_t n_tiles;
  int64_t n_qtiles;
  int64_t n_units;
  float *out;
  int64_t ld_out;
  int32_t vec_ok;
  int32_t *status;
};

constexpr int kFThreads = 512;  // fast scorer: 16 warps, 4 query rows each
constexpr int kRowsPerWarp = kTQ / (kFThreads / 32);
constexpr int kGroup = 32 / kRowsPerWarp;  // lanes walking one row's segments
constexpr int kHitCap = 24;  // hits of one query row walked per round
constexpr int kMaxRounds = 1 << 20;  // far above any row's entry count
constexpr int kFOffAcc = 0;
constexpr int kFOffImg = kFOffAcc + kTQ * kTI * 4;
constexpr int kFOffSlab = kFOffImg + kImgBytes;
constexpr int kFOffQhot = kFOffSlab + kHotMax * kTI * 4;
constexpr int kFOffHits = kFOffQhot + kHotMax * kTQ * 4;
constexpr int kFOffInvQ = kFOffHits + kTQ * kHitCap * 8;
constexpr int kFOffInvI = kFOffInvQ + kTQ * 4;
constexpr int kFOffNh = kFOffInvI + kTI * 4;
constexpr int kFastSmem = kFOffNh + kTQ * 4;
static_assert(kFastSmem <= 232448, "fast scoring block exceeds 227 KB of shared memory");
static_assert(kFOffSlab % 16 == 0 && kFOffQhot % 16 == 0 && kFOffHits % 16 == 0 &&
                  kFOffInvI % 16 == 0,
              "fast scorer shared sections must stay 16-byte aligned");

// Read-only global loads kept where they are written: the compiler may move
// plain __ldg loads past barriers to their first use, which would defeat
// issuing them early so their latency hides behind other work.
__device__ __forceinline__ int32_t ld_early_s32(const int32_t *p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ int64_t ld_early_s64(const int64_t *p) {
  int64_t v;
  asm volatile("ld.global.nc.s64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ int2 ld_early_s64_as_int2(const int2 *p) {
  int2 v;
  asm volatile("ld.global.nc.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Copies n bytes (a multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void cp_bytes(unsigned char *dst, const unsigned char *src, int n) {
  for (int j = threadIdx.x * 16; j < n; j += kFThreads * 16) cp_async16(dst + j, src + j);
}

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

// Looks dimension k up in the item tile's image (linear probing from the
// home slot).  Reads the aligned group of four slots around the probe point
// with two 16-byte loads and checks the four at once, so a long probe
// sequence costs a quarter as many dependent loads.  Returns the segment
// [start, end) packed as start | end << 16 (0 if absent).
__device__ __forceinline__ uint32_t image_find(const uint2 *slots, const uint32_t *bits, int32_t k) {
  // About half of a query row's cold dims are absent from a given item tile;
  // the tile's membership bitmap turns most of those misses into one load.
  const uint32_t bb = hash_b(k, kImgBitsLog2);
  if (!((bits[bb >> 5] >> (bb & 31)) & 1u)) return 0;
  const uint32_t s = hash_a(k, kImgSlotsBits);
  uint32_t base = s & ~3u;
  const int first = (int)(s & 3u);
  const uint32_t ku = (uint32_t)k, empty = 0xffffffffu;
  uint32_t valid = 0xfu << first;  // slots of the first group before the home slot do not count
  for (int n = 0; n < kImgSlots / 4; ++n) {
    const uint4 a = *reinterpret_cast<const uint4 *>(slots + base);
    const uint4 b = *reinterpret_cast<const uint4 *>(slots + base + 2);
    const uint32_t eq = ((a.x == ku) | ((a.z == ku) << 1) | ((b.x == ku) << 2) | ((b.z == ku) << 3)) & valid;
    const uint32_t em =
        ((a.x == empty) | ((a.z == empty) << 1) | ((b.x == empty) << 2) | ((b.z == empty) << 3)) & valid;
    const uint32_t stop = eq | em;
    if (stop) {
      const uint32_t j = __ffs(stop) - 1;  // the first slot that is k or empty
      if (!((eq >> j) & 1u)) return 0;
      return j == 0 ? a.y : j == 1 ? a.w : j == 2 ? b.y : b.w;
    }
    valid = 0xfu;
    base = (base + 4) & (kImgSlots - 1);
  }
  return 0;
}

// Dense product over the hot dims for 512 threads: thread (lq, li) of warp
// (wq, wi) owns queries wq*16 + lq*4 + [0, 4) and items wi*64 + li*8 + [0, 8).
__device__ __forceinline__ void hot_product512(float *acc, const float *qhot, const float *slab,
                                               int H) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int qb = (warp & 3) * 16 + (lane >> 3) * 4;
  const int ib = (warp >> 2) * 64 + (lane & 7) * 8;
  float2 c[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < 4; ++j) c[r][j] = make_float2(0.f, 0.f);
  // Operands of dim h + 1 are loaded while dim h is multiplied.
  float4 qa = make_float4(0.f, 0.f, 0.f, 0.f), ia = qa, ic = qa;
  if (H > 0) {
    qa = *reinterpret_cast<const float4 *>(qhot + qb);
    ia = *reinterpret_cast<const float4 *>(slab + ib);
    ic = *reinterpret_cast<const float4 *>(slab + ib + 4);
  }
  for (int h = 0; h < H; ++h) {
    const int hn = h + 1 < H ? h + 1 : h;
    const float4 qn = *reinterpret_cast<const float4 *>(qhot + hn * kTQ + qb);
    const float4 in = *reinterpret_cast<const float4 *>(slab + hn * kTI + ib);
    const float4 cn = *reinterpret_cast<const float4 *>(slab + hn * kTI + ib + 4);
    const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
    const float2 i0 = make_float2(ia.x, ia.y), i1 = make_float2(ia.z, ia.w);
    const float2 i2 = make_float2(ic.x, ic.y), i3 = make_float2(ic.z, ic.w);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float2 qq = make_float2(qv[r], qv[r]);
      c[r][0] = __ffma2_rn(qq, i0, c[r][0]);
      c[r][1] = __ffma2_rn(qq, i1, c[r][1]);
      c[r][2] = __ffma2_rn(qq, i2, c[r][2]);
      c[r][3] = __ffma2_rn(qq, i3, c[r][3]);
    }
    qa = qn;
    ia = in;
    ic = cn;
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float4 *d = reinterpret_cast<float4 *>(acc + (qb + r) * kTI + ib);
    d[0] = make_float4(c[r][0].x, c[r][0].y, c[r][1].x, c[r][1].y);
    d[1] = make_float4(c[r][2].x, c[r][2].y, c[r][3].x, c[r][3].y);
  }
}

// The persistent fast scorer for item tiles that have an image.  Units are
// (item tile, query tile) pairs, item-tile major, so a block loads an item
// tile's image and slab once and runs every query tile of its range on it.
// Per unit: the hot product writes acc; then warp w takes query rows
// 4w..4w+3, looks up each row's cold nonzeros in the image, and walks the
// hit segments with one 8-lane group per row (a group only touches its own
// row, and within one segment every item is distinct, so no accumulator is
// shared); then the normalised tile is stored.
__global__ void __launch_bounds__(kFThreads, 1) k_score_tiles(const TileArgs a) {
  extern __shared__ __align__(16) unsigned char fsm[];
  float *acc = reinterpret_cast<float *>(fsm + kFOffAcc);
  unsigned char *img = fsm + kFOffImg;
  float *slab = reinterpret_cast<float *>(fsm + kFOffSlab);
  float *qhot = reinterpret_cast<float *>(fsm + kFOffQhot);
  uint2 *hits = reinterpret_cast<uint2 *>(fsm + kFOffHits);
  float *invq = reinterpret_cast<float *>(fsm + kFOffInvQ);
  float *invi = reinterpret_cast<float *>(fsm + kFOffInvI);
  int *nh = reinterpret_cast<int *>(fsm + kFOffNh);
  const uint2 *slots = reinterpret_cast<const uint2 *>(img + kImgOffSlots);
  const uint32_t *bits = reinterpret_cast<const uint32_t *>(img + kImgOffBits);
  const uint8_t *seg_item = img + kImgOffItem;
  const float *seg_val = reinterpret_cast<const float *>(img + kImgOffVal);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.hot[0];

  const int64_t u0 = (int64_t)blockIdx.x * a.n_units / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * a.n_units / gridDim.x;
  int cur_t = -1;
  bool tile_ok = false;
  for (int64_t u = u0; u < u1; ++u) {
    const int t = (int)(u / a.n_qtiles);
    const int64_t g = u % a.n_qtiles;
    if (t != cur_t) {
      cur_t = t;
      tile_ok = a.meta[(size_t)t * kMetaInts + kMetaFits] != 0;
      if (tile_ok) {
        const unsigned char *src = a.image + (size_t)t * kImgBytes;
        const int32_t E = reinterpret_cast<const int32_t *>(src)[1];
        cp_bytes(img, src, kImgOffItem);  // header + slots
        cp_bytes(img + kImgOffItem, src + kImgOffItem, round16(E));
        cp_bytes(img + kImgOffVal, src + kImgOffVal, round16(4 * E));
        cp_bytes(reinterpret_cast<unsigned char *>(slab),
                 reinterpret_cast<const unsigned char *>(a.slab + (size_t)t * kHotMax * kTI),
                 H * kTI * 4);
        if (tid < kTI) {
          const int i = t * kTI + tid;
          invi[tid] = i < a.n_items ? __ldg(a.inv_i + i) : 0.f;
        }
      }
    }
    if (!tile_ok) continue;
    const int64_t q0 = g * kTQ;
    const int nq = (int)(a.n_q - q0 < kTQ ? a.n_q - q0 : kTQ);
    cp_bytes(reinterpret_cast<unsigned char *>(qhot),
             reinterpret_cast<const unsigned char *>(a.qhot + (size_t)g * kHotMax * kTQ),
             H * kTQ * 4);
    cp_async_commit();
    if (tid < kTQ) invq[tid] = tid < nq ? __ldg(a.inv_q + q0 + tid) : 0.f;
    // This warp's query rows: their cold ranges [indptr[q], indptr[q] +
    // cold count) and the first 32 cold entries of each, loaded now so that
    // the wait hides behind the hot product.
    int32_t p[kRowsPerWarp], e[kRowsPerWarp], ch[kRowsPerWarp];
    int2 pk[kRowsPerWarp];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int r = warp * kRowsPerWarp + rr;
      const int rc = r < nq ? r : 0;  // rows past n_q read row 0's range, then drop it
      p[rr] = (int32_t)ld_early_s64(a.q_indptr + q0 + rc);
      e[rr] = p[rr] + ld_early_s32(a.qcold_n + q0 + rc);
      if (r >= nq) p[rr] = e[rr] = 0;
      ch[rr] = 0;
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int32_t p0 = p[rr] + lane;
      pk[rr] = make_int2(-1, 0);
      if (p[rr] < e[rr]) {  // warp-uniform; the load is clamped inside the range, masked after
        const int2 x = ld_early_s64_as_int2(a.qcold + (p0 < e[rr] ? p0 : e[rr] - 1));
        if (p0 < e[rr]) pk[rr] = x;
      }
    }
    cp_async_wait_all();
    __syncthreads();
    // 1. hot dims
    if (H > 0) {
      hot_product512(acc, qhot, slab, H);
    } else {
      float4 *acc4 = reinterpret_cast<float4 *>(acc);
      for (int j = tid; j < kTQ * kTI / 4; j += kFThreads) acc4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    // 2. cold dims: lookups row by row, then one lane group per row walks.
    // Every round consumes at least one entry of some row; the round count is
    // bounded anyway, and running out of rounds raises the status flag.
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int round = 0;; ++round) {
      if (round == kMaxRounds) {
        if (lane == 0) flag(a.status, DEV_STALL);
        break;
      }
      bool left = false;
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        uint2 *hrow = hits + (warp * kRowsPerWarp + rr) * kHitCap;
        int n = 0;
        while (p[rr] < e[rr]) {
          const int32_t pp = p[rr] + lane;
          int2 x = make_int2(-1, 0);
          if (ch[rr] == 0) x = pk[rr];
          else if (pp < e[rr]) x = __ldg(a.qcold + pp);
          const int32_t k = x.x;
          const float v = __int_as_float(x.y);
          const uint32_t se = k >= 0 ? image_find(slots, bits, k) : 0u;
          const bool hit = (se >> 16) > (se & 0xffffu);
          const unsigned mask = __ballot_sync(0xffffffffu, hit);
          const int c = __popc(mask);
          const int room = kHitCap - n;
          const int rank = __popc(mask & lt_mask);
          if (c <= room) {
            if (hit) hrow[n + rank] = make_uint2(se, __float_as_uint(v));
            n += c;
            p[rr] = pp - lane + 32 < e[rr] ? pp - lane + 32 : e[rr];
            ++ch[rr];
            continue;
          }
          // More hits than room: keep the first `room` (room >= 1 whenever
          // n == 0, since kHitCap >= 1, so every round makes progress) and
          // resume right after the last one kept.
          if (room > 0) {
            if (hit && rank < room) hrow[n + rank] = make_uint2(se, __float_as_uint(v));
            unsigned m = mask;
            for (int j = 1; j < room; ++j) m &= m - 1u;  // drop the lowest room-1 hits
            p[rr] = pp - lane + __ffs(m);                 // one past the room-th hit's lane
            ch[rr] = 1;  // later chunks no longer line up with the prefetched one
            n += room;
          }
          break;
        }
        if (lane == 0) nh[warp * kRowsPerWarp + rr] = n;
        left |= p[rr] < e[rr];
      }
      __syncwarp();
      const int grp = lane / kGroup, li = lane % kGroup;
      const int row = warp * kRowsPerWarp + grp;
      const int my_n = nh[row];
      const uint2 *hrow = hits + row * kHitCap;
      float *arow = acc + row * kTI;
      for (int h = 0; h < my_n; ++h) {
        const uint2 hh = hrow[h];
        const float qv = __uint_as_float(hh.y);
        const int end = (int)(hh.x >> 16);
        // Two entries of the segment per step (distinct items, so the two
        // read-modify-writes are independent).
        int j = (int)(hh.x & 0xffffu) + li;
        for (; j + kGroup < end; j += 2 * kGroup) {
          float *d0 = arow + seg_item[j];
          float *d1 = arow + seg_item[j + kGroup];
          const float v0 = seg_val[j], v1 = seg_val[j + kGroup];
          const float a0 = *d0, a1 = *d1;
          *d0 = fmaf(qv, v0, a0);
          *d1 = fmaf(qv, v1, a1);
        }
        if (j < end) {
          float *d = arow + seg_item[j];
          *d = fmaf(qv, seg_val[j], *d);
        }
      }
      __syncwarp();
      if (!__any_sync(0xffffffffu, left)) break;
    }
    __syncthreads();
    // 3. normalise and store
    {
      const int i0 = t * kTI;
      const int ni = min(kTI, a.n_items - i0);
      const int c = (tid & 63) * 4;
      if (c < ni) {
        const float4 n4 = *reinterpret_cast<const float4 *>(invi + c);
        const bool vec = a.vec_ok && (c + 4 <= ni);
        for (int r = tid >> 6; r < nq; r += kFThreads / 64) {
          const float4 v = *reinterpret_cast<const float4 *>(acc + r * kTI + c);
          const float iq = invq[r];
          float *dst = a.out + (q0 + r) * a.ld_out + i0 + c;
          const float o0 = v.x * iq * n4.x, o1 = v.y * iq * n4.y, o2 = v.z * iq * n4.z,
                      o3 = v.w * iq * n4.w;
          if (vec) {
            __stcs(reinterpret_cast<float4 *>(dst), make_float4(o0, o1, o2, o3));
          } else {
            const float o[4] = {o0, o1, o2, o3};
            for (int j = 0; j < 4 && c + j < ni; ++j) dst[j] = o[j];
          }
        }
      }
    }
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
  ++h->hot_generation;
  return cudaSuccess;
}

cudaError_t launch_build_hybrid(ss_handle *h, const ss_csr &items, int64_t row_begin,
                                int64_t row_end, cudaStream_t s) {
  const int n_items = (int)(row_end - row_begin);
  const int n_tiles = (n_items + kTI - 1) / kTI;
  cudaError_t e = cudaMemsetAsync(h->counters, 0, 2 * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  static bool configured = false;
  if (!configured) {
    e = cudaFuncSetAttribute(k_build_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize, kBuildSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k_build_tiles<<<n_tiles, kBThreads, kBuildSmem, s>>>(
      items.indptr, items.indices, items.values, row_begin, row_end, h->hot, h->slab, h->ell,
      h->meta, h->heavy_k, h->heavy_v, h->heavy_item, h->counters, h->heavy_cap, h->image,
      h->d_status);
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
  ix.image = h->image;
  ix.counters = h->counters;
  return cudaSuccess;
}

// Hot values per query tile and the cold index view, for the current hot
// set; redone when the query matrix or the hot set changes.
static cudaError_t prepare_queries(ss_handle *h, const ss_csr &q, cudaStream_t s, int *queued) {
  *queued = 0;
  if (h->prep_src[0] == q.indptr && h->prep_src[1] == q.indices && h->prep_src[2] == q.values &&
      h->prep_rows == q.n_rows && h->prep_nnz == q.nnz && h->prep_generation == h->hot_generation)
    return cudaSuccess;
  const int64_t n_qtiles = (q.n_rows + kTQ - 1) / kTQ;
  const int64_t need_hot = std::max<int64_t>(1, n_qtiles * kHotMax * kTQ);
  const int64_t need_cold = std::max<int64_t>(1, q.nnz);
  const int64_t need_n = std::max<int64_t>(1, q.n_rows);
  if (need_hot > h->qhot_cap || need_cold > h->qcold_cap || need_n > h->qcold_n_cap) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (need_hot > h->qhot_cap) {
      cudaFree(h->qhot);
      h->qhot = nullptr;
      h->qhot_cap = 0;
      e = cudaMalloc(&h->qhot, sizeof(float) * (size_t)need_hot);
      if (e != cudaSuccess) return e;
      h->qhot_cap = need_hot;
    }
    if (need_cold > h->qcold_cap) {
      cudaFree(h->qcold);
      h->qcold = nullptr;
      h->qcold_cap = 0;
      e = cudaMalloc(&h->qcold, sizeof(int2) * (size_t)need_cold);
      if (e != cudaSuccess) return e;
      h->qcold_cap = need_cold;
    }
    if (need_n > h->qcold_n_cap) {
      cudaFree(h->qcold_n);
      h->qcold_n = nullptr;
      h->qcold_n_cap = 0;
      e = cudaMalloc(&h->qcold_n, sizeof(int32_t) * (size_t)need_n);
      if (e != cudaSuccess) return e;
      h->qcold_n_cap = need_n;
    }
  }
  const int64_t rows_padded = n_qtiles * kTQ;
  const int64_t blocks_needed = (rows_padded + kThreads / 32 - 1) / (kThreads / 32);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(blocks_needed, (int64_t)h->sm_count * 8));
  k_prep_queries<<<grid, kThreads, 0, s>>>(q.indptr, q.indices, q.values, q.n_rows, rows_padded,
                                           h->hot, h->qhot, h->qcold, h->qcold_n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *queued = 1;
  h->prep_src[0] = q.indptr;
  h->prep_src[1] = q.indices;
  h->prep_src[2] = q.values;
  h->prep_rows = q.n_rows;
  h->prep_nnz = q.nnz;
  h->prep_generation = h->hot_generation;
  return cudaSuccess;
}

cudaError_t launch_score_hybrid(ss_handle *h, const ss_csr &queries, const float *inv_q,
                                const ss_index &idx, const float *inv_i, float *out,
                                int64_t ld_out, cudaStream_t s, int *queued) {
  *queued = 0;
  if (queries.n_rows == 0 || idx.n_items == 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_score_hybrid, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kScoreSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_score_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize, kFastSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  int prep = 0;
  cudaError_t e = prepare_queries(h, queries, s, &prep);
  if (e != cudaSuccess) return e;
  const int64_t n_qtiles = (queries.n_rows + kTQ - 1) / kTQ;
  const int vec_ok = ((reinterpret_cast<uintptr_t>(out) % 16) == 0) && (ld_out % 4 == 0);
  const int sms = h->sm_count > 0 ? h->sm_count : 148;

  TileArgs f;
  f.q_indptr = queries.indptr;
  f.qcold = h->qcold;
  f.qcold_n = h->qcold_n;
  f.n_q = queries.n_rows;
  f.inv_q = inv_q;
  f.qhot = h->qhot;
  f.hot = idx.hot;
  f.slab = idx.slab;
  f.meta = idx.meta;
  f.image = idx.image;
  f.inv_i = inv_i;
  f.n_items = idx.n_items;
  f.n_tiles = idx.n_tiles;
  f.n_qtiles = n_qtiles;
  f.n_units = n_qtiles * idx.n_tiles;
  f.out = out;
  f.ld_out = ld_out;
  f.vec_ok = vec_ok;
  f.status = h->d_status;
  const int grid_f = (int)std::min<int64_t>(f.n_units, sms);
  k_score_tiles<<<grid_f, kFThreads, kFastSmem, s>>>(f);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

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
  a.n_qtiles = n_qtiles;
  a.counters = idx.counters;
  a.out = out;
  a.ld_out = ld_out;
  a.vec_ok = vec_ok;
  a.dim = (int32_t)idx.dim;
  k_score_hybrid<<<sms, kThreads, kScoreSmem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *queued = prep + 2;
  return cudaSuccess;
}
