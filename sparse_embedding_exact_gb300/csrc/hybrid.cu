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
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "internal.cuh"
#include "hotset.cuh"
#include "topk.cuh"

namespace {

using namespace hyb;
using namespace topk_dev;
using namespace hotset;

constexpr int kSelThreads = 1024;
constexpr int kSelSlotsBits = 14;
constexpr int kSelSlots = 1 << kSelSlotsBits;
constexpr int kSelCand = 1024;
__device__ __forceinline__ void flag(int32_t *status, int32_t code) {
  atomicCAS(status, DEV_OK, code);
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
// Probing starts at the first slot of the key's aligned group of four, so a
// reader that loads whole groups finds most keys in the first one.  Insert
// claims slots with compare-and-swap; find reads a group with one 16-byte
// load.  Every slot between a key's home and the key is occupied (slots go
// from empty to a key once and never change again), so a group that lacks
// the key but has an empty slot ends a search.
__device__ __forceinline__ uint32_t img_home(int32_t k) { return hash_a(k, kImgSlotsBits) & ~3u; }
__device__ __forceinline__ int img_insert(int *keys, uint32_t *bits, int32_t k) {
  uint32_t s = img_home(k);
  for (int n = 0; n < kImgSlots; ++n) {
    const int prev = atomicCAS(&keys[s], -1, k);
    if (prev == -1) {  // this thread added k: mark it in the membership bitmap
      const uint32_t bb = hash_b(k, kImgBitsLog2);
      atomicOr(&bits[bb >> 5], 1u << (bb & 31));
      return (int)s;
    }
    if (prev == k) return (int)s;
    s = (s + 1) & (kImgSlots - 1);
  }
  return -1;
}
__device__ __forceinline__ int img_find(const int *keys, int32_t k) {
  uint32_t base = img_home(k);
  for (int n = 0; n < kImgSlots / 4; ++n) {
    const int4 g = *reinterpret_cast<const int4 *>(keys + base);
    if (g.x == k) return (int)base;
    if (g.y == k) return (int)base + 1;
    if (g.z == k) return (int)base + 2;
    if (g.w == k) return (int)base + 3;
    if (g.x == -1 || g.y == -1 || g.z == -1 || g.w == -1) return -1;
    base = (base + 4) & (kImgSlots - 1);
  }
  return -1;
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gmem_src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

// Copies elements [b, e) of a 4-byte array to dst[0, e - a), where a = b
// rounded down to a multiple of 4 (so dst[p - a] holds element p): 16-byte
// copies for whole aligned groups inside [a, e) when the array itself is
// 16-byte aligned, 4-byte copies for the rest.  Elements [a, b) are copied
// too; they lie inside the array.
__device__ __forceinline__ void stage_words(void *dst, const void *src_array, int64_t b, int64_t e,
                                            int nthreads) {
  const int64_t a = b & ~(int64_t)3;
  const bool vec = (reinterpret_cast<uintptr_t>(src_array) & 15u) == 0;
  const int64_t e4 = vec ? (e & ~(int64_t)3) : a;
  const uint32_t *src = reinterpret_cast<const uint32_t *>(src_array);
  uint32_t *d = reinterpret_cast<uint32_t *>(dst);
  for (int64_t p = a + 4 * (int64_t)threadIdx.x; p < e4; p += 4 * (int64_t)nthreads)
    cp_async16(d + (p - a), src + p);
  const int64_t tail0 = e4 > a ? e4 : a;
  for (int64_t p = tail0 + threadIdx.x; p < e; p += nthreads) cp_async4(d + (p - a), src + p);
}

// Shared memory of the builder block (bytes).
constexpr int kBThreads = 1024;  // builder: 32 warps, one item row per warp at a time
constexpr int kBldOffSlab = 0;
constexpr int kBldOffKeys = kBldOffSlab + kHotMax * kTI * 4;
constexpr int kBldOffCnt = kBldOffKeys + kImgSlots * 4;
constexpr int kBldOffCold = kBldOffCnt + kImgSlots * 4;  // cold nonzeros per item
constexpr int kBldOffPtr = kBldOffCold + kTI * 4;         // the tile's row offsets (int64)
constexpr int kBldStage = 12288;                          // nonzeros of a tile staged on chip
constexpr int kBldOffIdx = kBldOffPtr + ((kTI + 1) * 8 + 15) / 16 * 16;
constexpr int kBldOffVal = kBldOffIdx + kBldStage * 4;
constexpr int kBuildSmem = kBldOffVal + kBldStage * 4;
static_assert(kBldOffIdx % 16 == 0 && kBldOffVal % 16 == 0, "staging buffers must stay 16-byte aligned");
static_assert(kImgECap <= kHotMax * kTI * 4, "segment items are staged in the slab's space");
constexpr int kItemsPerWarp = kTI / (kBThreads / 32);  // builder: consecutive items per warp
static_assert(kItemsPerWarp * (kBThreads / 32) == kTI, "warps cover the tile's items exactly");
constexpr int32_t kCodeHot = -1;  // code of a hot (or unplaced) nonzero in the builder

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

// One block per tile of kTI items.  The tile's row offsets, and its
// nonzeros when they fit (kBldStage), are first copied on chip with
// asynchronous copies, so the two passes below read shared memory instead of
// waiting on dependent global loads.  Warp w handles items w, w + 32, ...,
// its lanes taking the row's nonzeros 32 at a time.  Hot values go to the
// tile's slab.  The cold nonzeros become the tile's image (dimension ->
// segment of (item, value)) when they fit; otherwise they go to the ELL block
// and the heavy list, and the tile joins the overflow list.
__global__ void __launch_bounds__(kBThreads, 1)
    k_build_tiles(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                  const float *__restrict__ values, int64_t row_begin, int64_t row_end,
                  const int32_t *__restrict__ hot, float *__restrict__ slab,
                  int2 *__restrict__ ell, int32_t *__restrict__ meta,
                  int32_t *__restrict__ heavy_k, float *__restrict__ heavy_v,
                  uint8_t *__restrict__ heavy_item, int32_t *__restrict__ counters,
                  int64_t heavy_cap, unsigned char *__restrict__ image, int32_t *status,
                  int32_t chunk_rows, int32_t chunk_tiles, int32_t n_chunks,
                  int4 *__restrict__ heavy_tbl) {
  extern __shared__ __align__(16) unsigned char bsm[];
  float *slab_s = reinterpret_cast<float *>(bsm + kBldOffSlab);  // [kHotMax][kTI]
  uint8_t *item_s = bsm + kBldOffSlab;  // segment items, once the slab has been written out
  int *ikeys = reinterpret_cast<int *>(bsm + kBldOffKeys);
  int *icnt = reinterpret_cast<int *>(bsm + kBldOffCnt);
  int *cold_n = reinterpret_cast<int *>(bsm + kBldOffCold);
  int64_t *ptr_s = reinterpret_cast<int64_t *>(bsm + kBldOffPtr);
  const int32_t *idx_s = reinterpret_cast<const int32_t *>(bsm + kBldOffIdx);
  const float *val_s = reinterpret_cast<const float *>(bsm + kBldOffVal);
  __shared__ int hkeys[kHotSlots];
  __shared__ int8_t hvals[kHotSlots];
  __shared__ int red[kBThreads / 32];
  __shared__ int heavy_base, img_fail;
  __shared__ int heavy_off[kTI];
  __shared__ uint32_t bits_s[(1 << kImgBitsLog2) / 32];
  __shared__ int cum_s[kBThreads / 32][kItemsPerWarp + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  // Block t builds tile tl of chunk kc of the build (chunks of chunk_rows
  // items from row_begin; only the last may be shorter).  Images, slabs,
  // meta and ELL blocks are indexed by t; the chunk's overflow list is ovf.
  const int t = blockIdx.x;
  const int kc = min(t / chunk_tiles, n_chunks - 1);
  const int tl = t - kc * chunk_tiles;
  const int64_t chunk_begin = row_begin + (int64_t)kc * chunk_rows;
  const int64_t chunk_end = min(chunk_begin + (int64_t)chunk_rows, row_end);
  const int64_t item0 = chunk_begin + (int64_t)tl * kTI;
  const int n_items = (int)min((int64_t)kTI, chunk_end - item0);
  int32_t *ovf = counters + 1 + (size_t)kc * (1 + chunk_tiles);  // [0] count, [1..] tile numbers
  const int H = hot[0];
  if (tid <= n_items) ptr_s[tid] = indptr[item0 + tid];
  for (int w = tid; w < (1 << kImgBitsLog2) / 32; w += kBThreads) bits_s[w] = 0u;
  for (int s = tid; s < kHotSlots; s += kBThreads) hkeys[s] = -1;
  for (int s = tid; s < kImgSlots; s += kBThreads) {
    ikeys[s] = -1;
    icnt[s] = 0;
  }
  for (int j = tid; j < H * kTI; j += kBThreads) slab_s[j] = 0.0f;
  if (tid == 0) img_fail = 0;
  __syncthreads();
  const int64_t p0 = ptr_s[0], p1 = ptr_s[n_items];
  const int64_t pa = p0 & ~(int64_t)3;  // staged element p sits at [p - pa]
  const bool staged = p1 - pa <= kBldStage;
  if (staged) {
    stage_words(bsm + kBldOffIdx, indices, p0, p1, kBThreads);
    stage_words(bsm + kBldOffVal, values, p0, p1, kBThreads);
  }
  cp_async_commit();
  if (tid < H) hot_insert(hkeys, hvals, hot[1 + tid], tid);
  cp_async_wait_all();
  __syncthreads();
  auto key_at = [&](int64_t p) -> int32_t { return staged ? idx_s[p - pa] : __ldg(indices + p); };
  auto val_at = [&](int64_t p) -> float { return staged ? val_s[p - pa] : __ldg(values + p); };

  // Pass 1: hot values into the slab; cold dims into the image hash.  The
  // atomic that counts a cold entry's dimension also gives the entry's rank
  // within that dimension's segment; on a staged tile the entry's staged key
  // is replaced by its code (slot | rank << 16, or kCodeHot), so the scatter
  // needs neither lookups nor atomics.  Warp w takes items w, w + 32, ...,
  // whose rows its lanes run through as one list, 32 entries at a time (so
  // the block works through the items roughly in ascending order, and each
  // segment lists its items roughly ascending, which spreads the scorer's
  // accumulator accesses over the banks).
  int32_t *code_s = reinterpret_cast<int32_t *>(bsm + kBldOffIdx);
  int *cum = cum_s[warp];  // cum[m]: entries of the warp's items before item w + 32 m
  {
    const int item = warp + 32 * lane;
    int len = (lane < kItemsPerWarp && item < n_items) ? (int)(ptr_s[item + 1] - ptr_s[item]) : 0;
#pragma unroll
    for (int o = 1; o < kItemsPerWarp; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, len, o);
      if (lane >= o) len += v;
    }
    if (lane < kItemsPerWarp) cum[lane + 1] = len;
    if (lane == 0) cum[0] = 0;
    __syncwarp();
  }
  const int warp_entries = cum[kItemsPerWarp];
  {
    int m = 0;
    for (int f = lane; f < warp_entries; f += 32) {
      while (cum[m + 1] <= f) ++m;  // ends below kItemsPerWarp, since f < cum[kItemsPerWarp]
      const int it = warp + 32 * m;
      const int64_t p = ptr_s[it] + (f - cum[m]);
      const int32_t k = key_at(p);
      const int h = hot_find(hkeys, hvals, k);
      int32_t code = kCodeHot;
      if (h >= 0) {
        slab_s[h * kTI + it] = val_at(p);
      } else {
        const int slot = img_insert(ikeys, bits_s, k);
        if (slot < 0) img_fail = 1;
        else code = slot | (atomicAdd(&icnt[slot], 1) << 16);
      }
      if (staged) code_s[p - pa] = code;
    }
  }
  __syncthreads();
  {
    float *dst = slab + (size_t)t * kHotMax * kTI;
    for (int j = tid; j < H * kTI; j += kBThreads) dst[j] = slab_s[j];
  }
  unsigned char *img = image + (size_t)t * kImgBytes;
  int32_t *hdr = reinterpret_cast<int32_t *>(img);

  // ---- image path (the scans' barriers also end the slab's reads above)
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
  const bool fits = !img_fail && E <= kImgECap && D <= kImgDCap;
  if (fits) {
    uint2 *gslot = reinterpret_cast<uint2 *>(img + kImgOffSlots);
    for (int j = 0; j < kPer; ++j) {
      const int s = tid * kPer + j;
      if (ikeys[s] >= 0) {
        const int c = icnt[s];
        gslot[s] = make_uint2((uint32_t)ikeys[s], (uint32_t)e_run | ((uint32_t)(e_run + c) << 16));
        icnt[s] = e_run;  // now the segment's start (the fill cursor on the unstaged path)
        e_run += c;
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
    float *gval = reinterpret_cast<float *>(img + kImgOffVal);
    if (staged) {
      int m = 0;
      for (int f = lane; f < warp_entries; f += 32) {
        while (cum[m + 1] <= f) ++m;
        const int it = warp + 32 * m;
        const int64_t p = ptr_s[it] + (f - cum[m]);
        const int32_t code = code_s[p - pa];
        if (code == kCodeHot) continue;
        const int pos = icnt[code & 0xffff] + (code >> 16);
        item_s[pos] = (uint8_t)it;
        gval[pos] = val_s[p - pa];
      }
    } else {
      for (int it = warp; it < n_items; it += kBThreads / 32) {
        const int64_t pb = ptr_s[it], pe = ptr_s[it + 1];
        for (int64_t p = pb + lane; p < pe; p += 32) {
          const int32_t k = __ldg(indices + p);
          if (hot_find(hkeys, hvals, k) >= 0) continue;
          const int pos = atomicAdd(&icnt[img_find(ikeys, k)], 1);
          item_s[pos] = (uint8_t)it;
          gval[pos] = __ldg(values + p);
        }
      }
    }
    __syncthreads();
    uint4 *gitem = reinterpret_cast<uint4 *>(img + kImgOffItem);
    const uint4 *sitem = reinterpret_cast<const uint4 *>(item_s);
    for (int j = tid; j < round16(E) / 16; j += kBThreads) gitem[j] = sitem[j];
  }

  // ---- ELL path for tiles whose cold part does not fit an image
  int32_t *m = meta + (size_t)t * kMetaInts;
  int heavy_total = 0, n_heavy_items = 0;
  bool heavy_ok = true;
  if (!fits) {
    // Cold nonzeros per item (keys read from the CSR itself: a staged tile's
    // keys have been replaced by codes).
    for (int it = warp; it < kTI; it += kBThreads / 32) {
      int cold = 0;
      if (it < n_items)
        for (int64_t p = ptr_s[it] + lane; p < ptr_s[it + 1]; p += 32)
          cold += hot_find(hkeys, hvals, __ldg(indices + p)) < 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cold += __shfl_xor_sync(0xffffffffu, cold, o);
      if (lane == 0) cold_n[it] = cold;
    }
    __syncthreads();
    const int my_cold = tid < kTI ? cold_n[tid] : 0;
    const int sum_cold = bblock_sum(my_cold, red);
    // Items far above the tile's mean go to the heavy list.
    const int mean = n_items > 0 ? sum_cold / n_items : 0;
    const int thr = min(kEllMaxW, 2 * mean + 32);
    const bool my_heavy = tid < n_items && my_cold > thr;
    const int off = bblock_exclusive_scan(my_heavy ? my_cold : 0, red, &heavy_total);
    if (tid < kTI) heavy_off[tid] = my_heavy ? off : -1;
    // The heavy items in item order, for the fallback scorer.
    const int hslot = bblock_exclusive_scan(my_heavy ? 1 : 0, red, &n_heavy_items);
    if (my_heavy) heavy_tbl[(size_t)t * kTI + hslot] = make_int4(tid, off, my_cold, 0);
    if (tid == 0) {
      heavy_base = heavy_total > 0 ? atomicAdd(&counters[0], heavy_total) : 0;
      hdr[2] = 0;
      const int c = atomicAdd(&ovf[0], 1);
      ovf[1 + c] = tl;
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
        const int64_t pb = ptr_s[it], pe = ptr_s[it + 1];
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
            const float v = val_at(pp);
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
  if (tid == 0) {
    if (fits) m[8] = 0;
    m[9] = (!fits && heavy_ok) ? heavy_total : 0;
    m[kMetaHeavyItems] = (!fits && heavy_ok) ? n_heavy_items : 0;
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
  const int4 *heavy_tbl;
  const float *inv_i;
  int32_t n_items;
  int32_t n_tiles;
  int64_t n_qtiles;
  const int32_t *counters;  // [1] tiles without an image, [2..] their ids
  float *out;
  int64_t ld_out;
  int32_t vec_ok;
  int32_t dim;
  ss_topk topk;     // k > 0: offer top-k candidates instead of storing the tile
  int32_t *status;
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
  // Heavy items: one warp per item.  Its lanes look up 32 of the item's
  // nonzeros (ascending dims) at a time; then the query lists of the hits
  // are applied one after another in lane order, all lanes sharing each
  // list (whose rows are distinct).  Only this warp writes the item's
  // column, and every entry's cold terms keep ascending dimension order, as
  // on the regular path, so the result does not depend on which items a
  // tile's layout makes heavy.
  const int hb = m[8], n_hv = m[kMetaHeavyItems];
  const int lane = tid & 31;
  for (int g = warp; g < n_hv; g += kThreads / 32) {
    const int4 hv = __ldg(a.heavy_tbl + (size_t)t * kTI + g);
    const int64_t e0 = (int64_t)hb + hv.y;
    float *acol = sm.acc + hv.x;
    for (int base = 0; base < hv.z; base += 32) {
      const int e = base + lane;
      int32_t k = -1;
      float v = 0.f;
      if (e < hv.z) {
        k = __ldg(a.heavy_k + e0 + e);
        v = __ldg(a.heavy_v + e0 + e);
      }
      const uint32_t hm = (k >= lo && k < hi) ? batch_find(sm, k) : 0u;
      unsigned pending = __ballot_sync(0xffffffffu, (hm & 0xffffu) != 0u);
      while (pending) {
        const int j = __ffs(pending) - 1;
        pending &= pending - 1u;
        const uint32_t hj = __shfl_sync(0xffffffffu, hm, j);
        const float vj = __shfl_sync(0xffffffffu, v, j);
        const uint32_t st = hj >> 16, cnt = hj & 0xffffu;
        for (uint32_t x = lane; x < cnt; x += 32) {
          const uint2 l = sm.lists[st + x];
          float *d = acol + l.x;
          *d = fmaf(__uint_as_float(l.y), vj, *d);
        }
        __syncwarp();
      }
    }
  }
}

__device__ __forceinline__ void store_tile(const Smem &sm, const HybridArgs &a, int64_t q0, int nq,
                                           int t) {
  const int tid = threadIdx.x;
  const int i0 = t * kTI;
  const int ni = min(kTI, a.n_items - i0);
  if (a.topk.k > 0) {  // one warp per row: lane l holds items 4l + [0, 4) and 128 + 4l + [0, 4)
    const int lane = tid & 31, warp = tid >> 5;
    const int ia = 4 * lane, ib = 128 + 4 * lane;
    float n[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      n[j] = ia + j < ni ? __ldg(a.inv_i + i0 + ia + j) : 0.f;
      n[4 + j] = ib + j < ni ? __ldg(a.inv_i + i0 + ib + j) : 0.f;
    }
    for (int r = warp; r < nq; r += kThreads / 32) {
      const float iq = __ldg(a.inv_q + q0 + r);
      const float4 va = *reinterpret_cast<const float4 *>(sm.acc + r * kTI + ia);
      const float4 vb = *reinterpret_cast<const float4 *>(sm.acc + r * kTI + ib);
      const float v[8] = {va.x * iq * n[0], va.y * iq * n[1], va.z * iq * n[2], va.w * iq * n[3],
                          vb.x * iq * n[4], vb.y * iq * n[5], vb.z * iq * n[6], vb.w * iq * n[7]};
      const int it[8] = {i0 + ia, i0 + ia + 1, i0 + ia + 2, i0 + ia + 3,
                         i0 + ib, i0 + ib + 1, i0 + ib + 2, i0 + ib + 3};
      const bool ok[8] = {ia < ni, ia + 1 < ni, ia + 2 < ni, ia + 3 < ni,
                          ib < ni, ib + 1 < ni, ib + 2 < ni, ib + 3 < ni};
      const float thr = __ldg(a.topk.best_val + (q0 + r) * a.topk.k + (a.topk.k - 1));
      topk_offer(a.topk, q0 + r, thr, v, it, ok, lane, a.status);
    }
    return;
  }
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
// One warp per group of kQGroup query rows.  Each row's hot values go into
// its column of the query tile's hot block ([tile][kHotMax][kTQ], zero where
// absent).  The group's cold nonzeros, as {dim, value bits}, are packed row
// after row (each row's in its original, ascending order) from the group's
// first CSR position, so a group's cold list is contiguous; each row's cold
// count is kept.  Rows past n_q in the last tile get a zero column.
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
  // One warp per group of kQGroup rows; the group's cold entries are packed
  // row after row from the group's first CSR position.
  const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
  for (int64_t j = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
       j < n_rows_padded / kQGroup; j += warps) {
    const int64_t q_first = j * kQGroup;
    const int64_t base = indptr[q_first < n_q ? q_first : n_q];
    int n = 0;
    for (int r = 0; r < kQGroup; ++r) {
      const int64_t q = q_first + r;
      float *col = qhot + (q / kTQ) * kHotMax * kTQ + (q % kTQ);
      for (int h = lane; h < kHotMax; h += 32) col[h * kTQ] = 0.f;
      __syncwarp();
      if (q >= n_q) continue;
      const int64_t b = indptr[q], e = indptr[q + 1];
      int n_row = 0;
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
        if (cold) qcold[base + n + __popc(m & lt_mask)] = make_int2(k, __float_as_int(v));
        n += __popc(m);
        n_row += __popc(m);
      }
      if (lane == 0) qcold_n[q] = n_row;
    }
  }
}

struct TileArgs {
  const int64_t *q_indptr;
  const int2 *qcold;
  const int32_t *qcold_n;
  int64_t n_q;
  int64_t q_nnz;  // qcold entries: indptr[n_q]
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
  ss_topk topk;  // k > 0: offer top-k candidates instead of storing the tile
};

constexpr int kFThreads = 512;                   // fast scorer: 16 warps
constexpr int kFWarps = kFThreads / 32;
constexpr int kGroup = 32 / kQGroup;             // lanes walking one row's segments
constexpr int kHitCap = 78;                      // hits of one row group held per round
constexpr int kPasses = 4;                       // lookup passes of 32 entries in flight
static_assert(kPasses == 4, "the lookup dispatch instantiates 1 to 4 passes");
static_assert(kHotMax % 4 == 0, "hot dims are padded to a multiple of 4 inside the slab");
constexpr int kMaxRounds = 1 << 20;              // far above any group's entry count
constexpr int kGroupsPerQTile = kTQ / kQGroup;
constexpr int kFOffAcc = 0;                                          // [warp][kQGroup][kTI] f32
constexpr int kFOffImg = kFOffAcc + kFWarps * kQGroup * kTI * 4;
constexpr int kFOffSlab = kFOffImg + kImgBytes;                      // [kHotMax][kTI] f32
constexpr int kFOffQh = kFOffSlab + kHotMax * kTI * 4;               // [warp][kHotMax][kQGroup] f32
constexpr int kFOffHits = kFOffQh + kFWarps * kHotMax * kQGroup * 4; // [warp][kHitCap] {segment, value}
constexpr int kFOffCtl = kFOffHits + kFWarps * kHitCap * 8;          // next row group of the tile
constexpr int kFastSmem = kFOffCtl + 16;
static_assert(kFastSmem <= 232448, "fast scoring block exceeds 227 KB of shared memory");
static_assert(kFOffImg % 16 == 0 && kFOffSlab % 16 == 0 && kFOffQh % 16 == 0 &&
                  kFOffHits % 16 == 0 && kFOffCtl % 16 == 0,
              "fast scorer shared sections must stay 16-byte aligned");
static_assert(kQGroup == 4 && kTI == 256 && kGroup == 8,
              "the fast scorer's lane mapping assumes 4 rows x 256 items per warp");

// Read-only global loads kept where they are written: the compiler may move
// plain __ldg loads past other work to their first use, which would defeat
// issuing them early so their latency hides behind that work.
__device__ __forceinline__ int32_t ld_early_s32(const int32_t *p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_early_f32(const float *p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
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
__device__ __forceinline__ float4 ld_early_f4(const float *p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Copies n bytes (a multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void cp_bytes(unsigned char *dst, const unsigned char *src, int n) {
  for (int j = threadIdx.x * 16; j < n; j += kFThreads * 16) cp_async16(dst + j, src + j);
}

// Lanes [0, x) of a warp (x clamped to [0, 32]).
__device__ __forceinline__ unsigned lanes_below(int x) {
  return x <= 0 ? 0u : x >= 32 ? 0xffffffffu : (1u << x) - 1u;
}

// The rest of a lookup whose home group of four slots held neither the key
// nor an empty slot: linear probing over the following groups.
__device__ __forceinline__ uint32_t image_find_rest(const uint2 *slots, int32_t k, uint32_t base) {
  const uint32_t ku = (uint32_t)k, empty = 0xffffffffu;
  for (int n = 1; n < kImgSlots / 4; ++n) {
    base = (base + 4) & (kImgSlots - 1);
    const uint4 a = *reinterpret_cast<const uint4 *>(slots + base);
    const uint4 b = *reinterpret_cast<const uint4 *>(slots + base + 2);
    if (a.x == ku) return a.y;
    if (a.z == ku) return a.w;
    if (b.x == ku) return b.y;
    if (b.z == ku) return b.w;
    if (a.x == empty || a.z == empty || b.x == empty || b.z == empty) return 0;
  }
  return 0;
}

// Looks up P <= kPasses dimensions per lane (k < 0: none) in the item tile's
// image and returns each one's segment [start, end) packed as start |
// end << 16 (0 if absent).  About half of a query row's cold dimensions are
// absent from a given tile; the membership bitmap turns most of those misses
// into one load.  The others read their home group of four slots (every key
// between the home slot and a key's own slot is occupied, so a key missing
// from a group that holds an empty slot is absent).  All passes' loads are
// issued before any result is used.
template <int P>
__device__ __forceinline__ void image_lookups(const uint2 *slots, const uint32_t *bits,
                                              const int2 (&x)[kPasses], uint32_t (&se)[kPasses]) {
  bool cand[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const uint32_t bb = hash_b(x[p].x, kImgBitsLog2);
    cand[p] = x[p].x >= 0 && ((bits[bb >> 5] >> (bb & 31)) & 1u);
  }
  uint4 ga[P], gb[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    ga[p] = make_uint4(0u, 0u, 0u, 0u);
    gb[p] = ga[p];
    if (cand[p]) {
      const uint32_t base = img_home(x[p].x);
      ga[p] = *reinterpret_cast<const uint4 *>(slots + base);
      gb[p] = *reinterpret_cast<const uint4 *>(slots + base + 2);
    }
  }
  const uint32_t empty = 0xffffffffu;
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const uint32_t ku = (uint32_t)x[p].x;
    const uint4 a = ga[p], b = gb[p];
    se[p] = 0u;
    if (cand[p]) {
      if (a.x == ku) se[p] = a.y;
      else if (a.z == ku) se[p] = a.w;
      else if (b.x == ku) se[p] = b.y;
      else if (b.z == ku) se[p] = b.w;
      else if (a.x != empty && a.z != empty && b.x != empty && b.z != empty)
        se[p] = image_find_rest(slots, x[p].x, img_home(x[p].x));
    }
  }
}

// Dense product over the hot dims for one warp's row group: lane l owns
// items 4l + [0, 4) and 128 + 4l + [0, 4) of all kQGroup rows.  The dims run
// four at a time (H rounded up to a multiple of 4; the slab and hot values
// hold zeros past H), their twelve operand loads issued before the packed
// multiply-adds.  Writes the group's accumulator rows (zeros when there are
// no hot dims).
__device__ __forceinline__ void hot_product_group(float *acc, const float *qh, const float *slab,
                                                  int H, int lane) {
  const int ia = 4 * lane, ib = 128 + 4 * lane;
  float2 c[kQGroup][4];
#pragma unroll
  for (int r = 0; r < kQGroup; ++r)
#pragma unroll
    for (int j = 0; j < 4; ++j) c[r][j] = make_float2(0.f, 0.f);
  const int Hp = (H + 3) & ~3;
  for (int h0 = 0; h0 < Hp; h0 += 4) {
    float4 q4[4], sa[4], sb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      q4[u] = *reinterpret_cast<const float4 *>(qh + (h0 + u) * kQGroup);
      sa[u] = *reinterpret_cast<const float4 *>(slab + (h0 + u) * kTI + ia);
      sb[u] = *reinterpret_cast<const float4 *>(slab + (h0 + u) * kTI + ib);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float qv[4] = {q4[u].x, q4[u].y, q4[u].z, q4[u].w};
      const float2 i0 = make_float2(sa[u].x, sa[u].y), i1 = make_float2(sa[u].z, sa[u].w);
      const float2 i2 = make_float2(sb[u].x, sb[u].y), i3 = make_float2(sb[u].z, sb[u].w);
#pragma unroll
      for (int r = 0; r < kQGroup; ++r) {
        const float2 qq = make_float2(qv[r], qv[r]);
        c[r][0] = __ffma2_rn(qq, i0, c[r][0]);
        c[r][1] = __ffma2_rn(qq, i1, c[r][1]);
        c[r][2] = __ffma2_rn(qq, i2, c[r][2]);
        c[r][3] = __ffma2_rn(qq, i3, c[r][3]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kQGroup; ++r) {
    *reinterpret_cast<float4 *>(acc + r * kTI + ia) =
        make_float4(c[r][0].x, c[r][0].y, c[r][1].x, c[r][1].y);
    *reinterpret_cast<float4 *>(acc + r * kTI + ib) =
        make_float4(c[r][2].x, c[r][2].y, c[r][3].x, c[r][3].y);
  }
}

// Adds q * value over one image segment into a row's accumulator: the lanes
// of a group take every kGroup-th entry, two entries per step, the second
// one predicated (the items of one segment are distinct, so the two
// read-modify-writes are independent, and one loop body serves every length
// without a separate tail for the group to diverge on).
__device__ __forceinline__ void walk_segment(float *arow, const uint8_t *seg_item,
                                             const float *seg_val, uint2 hh, int li) {
  const float qv = __uint_as_float(hh.y);
  const int end = (int)(hh.x >> 16);
  for (int j = (int)(hh.x & 0xffffu) + li; j < end; j += 2 * kGroup) {
    const bool two = j + kGroup < end;
    const int i0 = seg_item[j];
    const float v0 = seg_val[j];
    int i1 = 0;
    float v1 = 0.f;
    if (two) {
      i1 = seg_item[j + kGroup];
      v1 = seg_val[j + kGroup];
    }
    const float a0 = arow[i0];
    const float a1 = two ? arow[i1] : 0.f;
    arow[i0] = fmaf(qv, v0, a0);
    if (two) arow[i1] = fmaf(qv, v1, a1);
  }
}

// The persistent fast scorer for item tiles that have an image.  A block's
// range of (item tile, query tile) units is item-tile major: for each item
// tile in it, the block loads the tile's image, hot slab and item norms
// once, then its warps take groups of kQGroup query rows from a shared
// counter.  A warp scores its group against the tile on its own, with no
// block barrier: the hot product writes the group's accumulator rows; the
// group's cold nonzeros (contiguous, row after row) are looked up in the
// image 32 x kPasses at a time and the hits kept in order; one lane group
// per row walks that row's hit segments (a group only touches its own row,
// so no accumulator is shared, and each row's cold terms are added in
// ascending dimension order); then the normalised rows are stored.
// kTopk: offer top-k candidates (a.topk) instead of storing the tile; a
// separate instantiation, so the plain store path keeps its registers.
template <bool kTopk>
__global__ void __launch_bounds__(kFThreads, 1) k_score_tiles(const TileArgs a) {
  extern __shared__ __align__(16) unsigned char fsm[];
  unsigned char *img = fsm + kFOffImg;
  float *slab = reinterpret_cast<float *>(fsm + kFOffSlab);
  int *next_group = reinterpret_cast<int *>(fsm + kFOffCtl);
  const uint2 *slots = reinterpret_cast<const uint2 *>(img + kImgOffSlots);
  const uint32_t *bits = reinterpret_cast<const uint32_t *>(img + kImgOffBits);
  const uint8_t *seg_item = img + kImgOffItem;
  const float *seg_val = reinterpret_cast<const float *>(img + kImgOffVal);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float *acc = reinterpret_cast<float *>(fsm + kFOffAcc) + warp * kQGroup * kTI;
  float *qh = reinterpret_cast<float *>(fsm + kFOffQh) + warp * kHotMax * kQGroup;
  uint2 *hits = reinterpret_cast<uint2 *>(fsm + kFOffHits) + warp * kHitCap;
  const int grp = lane / kGroup, li = lane % kGroup;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int ia = 4 * lane, ib = 128 + 4 * lane;
  const int H = a.hot[0];
  const int64_t n_groups = (a.n_q + kQGroup - 1) / kQGroup;

  const int64_t u0 = (int64_t)blockIdx.x * a.n_units / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * a.n_units / gridDim.x;
  for (int64_t u = u0; u < u1;) {
    const int t = (int)(u / a.n_qtiles);
    const int64_t g_lo = u % a.n_qtiles;
    const int64_t u_end = u1 < (int64_t)(t + 1) * a.n_qtiles ? u1 : (int64_t)(t + 1) * a.n_qtiles;
    const int64_t g_hi = g_lo + (u_end - u);
    u = u_end;
    if (a.meta[(size_t)t * kMetaInts + kMetaFits] == 0) continue;  // same for the whole block
    __syncthreads();  // every warp is done with the previous tile
    {
      const unsigned char *src = a.image + (size_t)t * kImgBytes;
      const int32_t E = reinterpret_cast<const int32_t *>(src)[1];
      cp_bytes(img, src, kImgOffItem);  // header, slots, bitmap
      cp_bytes(img + kImgOffItem, src + kImgOffItem, round16(E));
      cp_bytes(img + kImgOffVal, src + kImgOffVal, round16(4 * E));
      cp_bytes(reinterpret_cast<unsigned char *>(slab),
               reinterpret_cast<const unsigned char *>(a.slab + (size_t)t * kHotMax * kTI),
               H * kTI * 4);
      cp_async_commit();
      for (int z = H * kTI + tid; z < ((H + 3) & ~3) * kTI; z += kFThreads) slab[z] = 0.f;  // pad rows
      if (tid == 0) *next_group = 0;
    }
    const int i0 = t * kTI;
    const int ni = a.n_items - i0 < kTI ? a.n_items - i0 : kTI;
    float na[4], nb[4];  // inverse norms of this lane's items (0 past the chunk)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      na[c] = ia + c < ni ? __ldg(a.inv_i + i0 + ia + c) : 0.f;
      nb[c] = ib + c < ni ? __ldg(a.inv_i + i0 + ib + c) : 0.f;
    }
    cp_async_wait_all();
    __syncthreads();

    const int64_t j_lo = g_lo * kGroupsPerQTile;
    const int64_t j_hi =
        g_hi * kGroupsPerQTile < n_groups ? g_hi * kGroupsPerQTile : n_groups;
    for (;;) {
      int jj = 0;
      if (lane == 0) jj = atomicAdd(next_group, 1);
      jj = __shfl_sync(0xffffffffu, jj, 0);
      const int64_t j = j_lo + jj;
      if (j >= j_hi) break;
      const int64_t q_first = j * kQGroup;
      const int nr = a.n_q - q_first < kQGroup ? (int)(a.n_q - q_first) : kQGroup;

      // Group metadata, hot values and the first cold entries, issued before
      // the hot product so their latency hides behind it.
      int cn = 0;
      float iq = 0.f, thr = 0.f;  // thr: the row's current k-th best (top-k epilogue)
      if (lane < nr) {
        cn = ld_early_s32(a.qcold_n + q_first + lane);
        iq = ld_early_f32(a.inv_q + q_first + lane);
        if (kTopk) thr = ld_early_f32(a.topk.best_val + (q_first + lane) * a.topk.k + (a.topk.k - 1));
      }
      const int64_t base = ld_early_s64(a.q_indptr + q_first);
      if (lane >= H && lane < ((H + 3) & ~3))  // pad rows of the hot values
        *reinterpret_cast<float4 *>(qh + lane * kQGroup) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane < H) {
        const float4 v = ld_early_f4(a.qhot + (size_t)(j / kGroupsPerQTile) * kHotMax * kTQ +
                                     lane * kTQ + (int)(j % kGroupsPerQTile) * kQGroup);
        *reinterpret_cast<float4 *>(qh + lane * kQGroup) = v;
      }
      int2 pf[kPasses];
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        pf[p] = make_int2(-1, 0);
        if (base + p * 32 + lane < a.q_nnz) pf[p] = ld_early_s64_as_int2(a.qcold + base + p * 32 + lane);
      }
      const int b1 = __shfl_sync(0xffffffffu, cn, 0);
      const int b2 = b1 + __shfl_sync(0xffffffffu, cn, 1);
      const int b3 = b2 + __shfl_sync(0xffffffffu, cn, 2);
      const int N = b3 + __shfl_sync(0xffffffffu, cn, 3);
      __syncwarp();

      // 1. hot dims
      hot_product_group(acc, qh, slab, H, lane);
      __syncwarp();

      // 2. cold dims, in rounds of at most kHitCap hits.  Every round starts
      // with room for 32 hits, so it consumes at least one pass of entries.
      int pos = 0;
      bool from_pf = true;
      for (int round = 0; pos < N; ++round) {
        if (round == kMaxRounds) {
          if (lane == 0) flag(a.status, DEV_STALL);
          break;
        }
        int nh = 0, h1 = 0, h2 = 0, h3 = 0;  // hits kept; of them, from rows before 1, 2, 3
        bool full = false;
        while (!full && pos < N) {
          int2 x[kPasses];
#pragma unroll
          for (int p = 0; p < kPasses; ++p) {
            const int e = pos + p * 32 + lane;
            if (from_pf) {
              x[p] = pf[p];
            } else {
              x[p] = make_int2(-1, 0);
              if (e < N) x[p] = __ldg(a.qcold + base + e);
            }
            if (e >= N) x[p].x = -1;
          }
          from_pf = false;
          // Only the passes that still hold entries are looked up.
          uint32_t se[kPasses] = {};
          const int live = (N - pos + 31) / 32;
          if (live >= kPasses) image_lookups<kPasses>(slots, bits, x, se);
          else if (live == 3) image_lookups<3>(slots, bits, x, se);
          else if (live == 2) image_lookups<2>(slots, bits, x, se);
          else image_lookups<1>(slots, bits, x, se);
          int next = pos + kPasses * 32 < N ? pos + kPasses * 32 : N;
#pragma unroll
          for (int p = 0; p < kPasses; ++p) {
            const int P = pos + p * 32;
            if (P >= N || full) continue;
            const bool hit = (se[p] >> 16) > (se[p] & 0xffffu);
            const unsigned mask = __ballot_sync(0xffffffffu, hit);
            const int room = kHitCap - nh;
            unsigned keep = mask;
            if (__popc(mask) > room) {
              // Keep the first `room` hits; the next round resumes at the
              // first hit not kept.
              unsigned rest = mask;
              for (int i = 0; i < room; ++i) rest &= rest - 1u;
              keep = mask & ~rest;
              next = P + __ffs(rest) - 1;
              full = true;
            }
            if ((keep >> lane) & 1u)
              hits[nh + __popc(keep & lt_mask)] = make_uint2(se[p], (uint32_t)x[p].y);  // value bits
            h1 += __popc(keep & lanes_below(b1 - P));
            h2 += __popc(keep & lanes_below(b2 - P));
            h3 += __popc(keep & lanes_below(b3 - P));
            nh += __popc(keep);
          }
          pos = next;
        }
        __syncwarp();
        // One lane group per row walks the row's hits, the next hit's record
        // loaded while the current segment is walked.
        const int hs = grp == 0 ? 0 : grp == 1 ? h1 : grp == 2 ? h2 : h3;
        const int he = grp == 0 ? h1 : grp == 1 ? h2 : grp == 2 ? h3 : nh;
        float *arow = acc + grp * kTI;
        uint2 hh = hits[hs < he ? hs : 0];
        for (int h = hs; h < he; ++h) {
          const uint2 nx = hits[h + 1 < he ? h + 1 : h];
          walk_segment(arow, seg_item, seg_val, hh, li);
          hh = nx;
        }
        __syncwarp();
      }

      // 3. normalise and store the group's rows (or offer them to the top-k)
      if constexpr (kTopk) {
        // Scores of row r of the group, normalised as the store path does.
        auto row_scores = [&](int r, float (&v)[8]) {
          const float iqr = __shfl_sync(0xffffffffu, iq, r);
          const float4 va = *reinterpret_cast<const float4 *>(acc + r * kTI + ia);
          const float4 vb = *reinterpret_cast<const float4 *>(acc + r * kTI + ib);
          v[0] = va.x * iqr * na[0];
          v[1] = va.y * iqr * na[1];
          v[2] = va.z * iqr * na[2];
          v[3] = va.w * iqr * na[3];
          v[4] = vb.x * iqr * nb[0];
          v[5] = vb.y * iqr * nb[1];
          v[6] = vb.z * iqr * nb[2];
          v[7] = vb.w * iqr * nb[3];
        };
        const int it[8] = {i0 + ia, i0 + ia + 1, i0 + ia + 2, i0 + ia + 3,
                           i0 + ib, i0 + ib + 1, i0 + ib + 2, i0 + ib + 3};
        const bool ok[8] = {ia < ni, ia + 1 < ni, ia + 2 < ni, ia + 3 < ni,
                            ib < ni, ib + 1 < ni, ib + 2 < ni, ib + 3 < ni};
        // Counts first, then lanes 0..3 reserve their rows' slots together,
        // then each row's offer is written.
        int mine = 0;
#pragma unroll
        for (int r = 0; r < kQGroup; ++r) {
          float v[8];
          row_scores(r, v);
          const int c = r < nr ? topk_count(__shfl_sync(0xffffffffu, thr, r), v, ok) : 0;
          if (lane == r) mine = c;
        }
        const int n_emit = mine < a.topk.k ? mine : a.topk.k;
        int base = 0;
        if (n_emit > 0) base = atomicAdd(a.topk.cand_n + q_first + lane, n_emit);
        if (n_emit > 0 && base + n_emit > a.topk.cand_cap) {  // cannot happen: at most k per tile
          flag(a.status, DEV_CAPACITY);
          mine = 0;
        }
#pragma unroll
        for (int r = 0; r < kQGroup; ++r) {
          const int c = __shfl_sync(0xffffffffu, mine, r);
          const int b = __shfl_sync(0xffffffffu, base, r);
          if (c == 0) continue;
          float v[8];
          row_scores(r, v);
          topk_emit(a.topk, q_first + r, __shfl_sync(0xffffffffu, thr, r), v, it, ok, b, c, lane);
        }
        __syncwarp();
        continue;
      }
#pragma unroll
      for (int r = 0; r < kQGroup; ++r) {
        const float iqr = __shfl_sync(0xffffffffu, iq, r);
        if (r >= nr) continue;
        float *dst = a.out + (q_first + r) * a.ld_out + i0;
        const float4 va = *reinterpret_cast<const float4 *>(acc + r * kTI + ia);
        const float4 vb = *reinterpret_cast<const float4 *>(acc + r * kTI + ib);
        const float oa[4] = {va.x * iqr * na[0], va.y * iqr * na[1], va.z * iqr * na[2],
                             va.w * iqr * na[3]};
        const float ob[4] = {vb.x * iqr * nb[0], vb.y * iqr * nb[1], vb.z * iqr * nb[2],
                             vb.w * iqr * nb[3]};
        if (a.vec_ok && ia + 4 <= ni) {
          __stcs(reinterpret_cast<float4 *>(dst + ia), make_float4(oa[0], oa[1], oa[2], oa[3]));
        } else {
          for (int c = 0; c < 4; ++c)
            if (ia + c < ni) dst[ia + c] = oa[c];
        }
        if (a.vec_ok && ib + 4 <= ni) {
          __stcs(reinterpret_cast<float4 *>(dst + ib), make_float4(ob[0], ob[1], ob[2], ob[3]));
        } else {
          for (int c = 0; c < 4; ++c)
            if (ib + c < ni) dst[ib + c] = ob[c];
        }
      }
      __syncwarp();
    }
  }
  cp_async_wait_all();
}

// The automatic choice between item tiles and posting lists: per item tile of
// a build, the cold entries (those outside the hot set) against the image's
// entry capacity kImgECap, the builder's own rule for a tile without an
// image.  probe[0] += tiles, probe[1] += tiles above the capacity.
__global__ void __launch_bounds__(256)
    k_auto_probe(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                 int64_t row_begin, int64_t row_end, const int32_t *__restrict__ hot,
                 int32_t *__restrict__ probe) {
  __shared__ int hkeys[kHotSlots];
  __shared__ int8_t hvals[kHotSlots];
  __shared__ int red[8];
  const int tid = threadIdx.x;
  const int64_t i0 = row_begin + (int64_t)blockIdx.x * kTI;
  const int64_t i1 = min(i0 + kTI, row_end);
  for (int j = tid; j < kHotSlots; j += 256) hkeys[j] = -1;
  __syncthreads();
  const int H = hot[0];
  if (tid < H) hot_insert(hkeys, hvals, hot[1 + tid], tid);
  __syncthreads();
  const int64_t p0 = indptr[i0], p1 = indptr[i1];
  int cold = 0;
  for (int64_t p = p0 + tid; p < p1; p += 256) cold += hot_find(hkeys, hvals, __ldg(indices + p)) < 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cold += __shfl_xor_sync(0xffffffffu, cold, o);
  if ((tid & 31) == 0) red[tid >> 5] = cold;
  __syncthreads();
  if (tid == 0) {
    int e = 0;
    for (int w = 0; w < 8; ++w) e += red[w];
    atomicAdd(probe, 1);
    if (e > kImgECap) atomicAdd(probe + 1, 1);
  }
}

}  // namespace

cudaError_t launch_auto_probe(ss_handle *h, const ss_csr &items, int64_t row_begin, int64_t row_end,
                              int32_t *probe, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(probe, 0, 2 * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (row_end - row_begin + kTI - 1) / kTI;
  if (tiles <= 0) return cudaSuccess;
  k_auto_probe<<<(unsigned)tiles, 256, 0, s>>>(items.indptr, items.indices, row_begin, row_end,
                                               h->hot, probe);
  return cudaGetLastError();
}



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
    cudaError_t e = ensure_dyn_smem(k_hot_select, smem);
    if (e != cudaSuccess) return e;
    k_hot_select<<<1, kSelThreads, smem, s>>>(items.indptr, items.indices, n, n_sample, h->hot);
    e = cudaGetLastError();
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
  const int64_t C = h->chunk_rows;
  const int T = h->chunk_tiles;
  const int n_chunks = (int)((row_end - row_begin + C - 1) / C);
  const int64_t last_len = row_end - (row_begin + (int64_t)(n_chunks - 1) * C);
  const int n_tiles = (n_chunks - 1) * T + (int)((last_len + kTI - 1) / kTI);
  h->n_views = 0;
  if (n_chunks < 1 || n_chunks > h->build_batch || n_tiles > h->max_tiles) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(h->counters, 0, sizeof(int32_t) * (1 + (size_t)n_chunks * (1 + T)), s);
  if (e != cudaSuccess) return e;
  if ((e = ensure_dyn_smem(k_build_tiles, kBuildSmem)) != cudaSuccess) return e;
  k_build_tiles<<<n_tiles, kBThreads, kBuildSmem, s>>>(
      items.indptr, items.indices, items.values, row_begin, row_end, h->hot, h->slab, h->ell,
      h->meta, h->heavy_k, h->heavy_v, h->heavy_item, h->counters, h->heavy_cap, h->image,
      h->d_status, (int32_t)C, T, n_chunks, h->heavy_tbl);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  for (int k = 0; k < n_chunks; ++k) {
    ss_index &ix = h->views[k];
    const size_t t0 = (size_t)k * T;
    ix = ss_index();
    ix.algo = ALGO_HYBRID;
    ix.row_begin = row_begin + (int64_t)k * C;
    ix.row_end = std::min<int64_t>(ix.row_begin + C, row_end);
    ix.n_items = (int32_t)(ix.row_end - ix.row_begin);
    ix.dim = h->dim;
    ix.n_tiles = (ix.n_items + kTI - 1) / kTI;
    ix.hot = h->hot;
    ix.slab = h->slab + t0 * kHotMax * kTI;
    ix.ell = h->ell + t0 * kEllMaxW * kTI;
    ix.meta = h->meta + t0 * kMetaInts;
    ix.heavy_k = h->heavy_k;
    ix.heavy_v = h->heavy_v;
    ix.heavy_item = h->heavy_item;
    ix.heavy_tbl = h->heavy_tbl + t0 * kTI;
    ix.image = h->image + t0 * kImgBytes;
    ix.counters = h->counters + (size_t)k * (1 + T);  // [1] the chunk's overflow count, [2..] its tiles
  }
  h->n_views = n_chunks;
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
      e = dev_alloc(&h->qhot, sizeof(float) * (size_t)need_hot);
      if (e != cudaSuccess) return e;
      h->qhot_cap = need_hot;
    }
    if (need_cold > h->qcold_cap) {
      cudaFree(h->qcold);
      h->qcold = nullptr;
      h->qcold_cap = 0;
      e = dev_alloc(&h->qcold, sizeof(int2) * (size_t)need_cold);
      if (e != cudaSuccess) return e;
      h->qcold_cap = need_cold;
    }
    if (need_n > h->qcold_n_cap) {
      cudaFree(h->qcold_n);
      h->qcold_n = nullptr;
      h->qcold_n_cap = 0;
      e = dev_alloc(&h->qcold_n, sizeof(int32_t) * (size_t)need_n);
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
                                int64_t ld_out, cudaStream_t s, int *queued, const ss_topk *topk) {
  *queued = 0;
  if (queries.n_rows == 0 || idx.n_items == 0) return cudaSuccess;
  cudaError_t e = ensure_dyn_smem(k_score_hybrid, kScoreSmem);
  if (e == cudaSuccess) e = ensure_dyn_smem(k_score_tiles<false>, kFastSmem);
  if (e == cudaSuccess) e = ensure_dyn_smem(k_score_tiles<true>, kFastSmem);
  if (e != cudaSuccess) return e;
  int prep = 0;
  e = prepare_queries(h, queries, s, &prep);
  if (e != cudaSuccess) return e;
  const int64_t n_qtiles = (queries.n_rows + kTQ - 1) / kTQ;
  const int vec_ok = ((reinterpret_cast<uintptr_t>(out) % 16) == 0) && (ld_out % 4 == 0);
  const int sms = h->sm_count > 0 ? h->sm_count : 148;

  TileArgs f;
  f.q_indptr = queries.indptr;
  f.qcold = h->qcold;
  f.qcold_n = h->qcold_n;
  f.n_q = queries.n_rows;
  f.q_nnz = queries.nnz;
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
  f.topk = topk ? *topk : ss_topk();
  const int grid_f = (int)std::min<int64_t>(f.n_units, sms);
  prof_mark(h, s);
  if (f.topk.k > 0) k_score_tiles<true><<<grid_f, kFThreads, kFastSmem, s>>>(f);
  else k_score_tiles<false><<<grid_f, kFThreads, kFastSmem, s>>>(f);
  prof_mark(h, s);
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
  a.heavy_tbl = idx.heavy_tbl;
  a.inv_i = inv_i;
  a.n_items = idx.n_items;
  a.n_tiles = idx.n_tiles;
  a.n_qtiles = n_qtiles;
  a.counters = idx.counters;
  a.out = out;
  a.ld_out = ld_out;
  a.vec_ok = vec_ok;
  a.dim = (int32_t)idx.dim;
  a.topk = topk ? *topk : ss_topk();
  a.status = h->d_status;
  k_score_hybrid<<<sms, kThreads, kScoreSmem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *queued = prep + 2;
  return cudaSuccess;
}

// ---------------------------------------------------------------- top-k merge
namespace {

__global__ void __launch_bounds__(256)
    k_topk_reset(int64_t n_q, int32_t k, float *best_val, int64_t *best_item, int32_t *cand_n) {
  const int64_t n = n_q * k;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    best_val[e] = -INFINITY;
    best_item[e] = -1;
  }
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n_q;
       q += (int64_t)gridDim.x * blockDim.x)
    cand_n[q] = 0;
}

// One warp per query row: the row's running best k and its candidates of
// the chunk (items item_base + chunk-relative number) go through k rounds
// of warp arg-best in the top-k order; then the candidates are cleared.
__global__ void __launch_bounds__(256)
    k_topk_merge(const ss_topk t, int64_t n_q, int64_t item_base, float *best_val,
                 int64_t *best_item) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t q = blockIdx.x * (int64_t)(blockDim.x / 32) + (threadIdx.x >> 5); q < n_q;
       q += warps) {
    const int m = t.cand_n[q];
    if (m == 0) continue;
    const int k = t.k, total = k + m;  // at most kTopkEntries (checked by the caller)
    float *bv = best_val + q * k;
    int64_t *bi = best_item + q * k;
    const float *cv = t.cand_val + q * t.cand_cap;
    const int32_t *ci = t.cand_item + q * t.cand_cap;
    float res_v[2] = {-INFINITY, -INFINITY};
    int64_t res_i[2] = {-1, -1};
    {
      uint32_t taken[kTopkEntries / 1024] = {};  // entries lane + 32 j
      for (int r = 0; r < k; ++r) {
        float lv = -INFINITY;
        int64_t li = INT64_MAX;
        int lj = -1;
        for (int j = 0; lane + 32 * j < total; ++j) {
          if ((taken[j >> 5] >> (j & 31)) & 1u) continue;
          const int e = lane + 32 * j;
          const float v = e < k ? bv[e] : cv[e - k];
          const int64_t it = e < k ? bi[e] : item_base + ci[e - k];
          if (topk_before(v, it, lv, li)) {
            lv = v;
            li = it;
            lj = j;
          }
        }
        float wv = lv;
        int64_t wi = li;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
          const int64_t oi = __shfl_xor_sync(0xffffffffu, wi, o);
          if (topk_before(ov, oi, wv, wi)) {
            wv = ov;
            wi = oi;
          }
        }
        if (lj >= 0 && lv == wv && li == wi) taken[lj >> 5] |= 1u << (lj & 31);
        if ((r & 31) == lane) {
          res_v[r >> 5] = wv;
          res_i[r >> 5] = wi < 0 || wi == INT64_MAX ? -1 : wi;
        }
      }
    }
    __syncwarp();
    for (int rr = 0; rr < 2; ++rr) {
      const int r = lane + 32 * rr;
      if (r < k) {
        bv[r] = res_v[rr];
        bi[r] = res_i[rr];
      }
    }
    if (lane == 0) t.cand_n[q] = 0;
  }
}

}  // namespace

cudaError_t launch_topk_reset(int64_t n_q, int32_t k, float *best_val, int64_t *best_item,
                              int32_t *cand_n, int sm_count, cudaStream_t s) {
  if (n_q == 0) return cudaSuccess;
  const int64_t need = (n_q * k + 255) / 256;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count * 8));
  k_topk_reset<<<grid, 256, 0, s>>>(n_q, k, best_val, best_item, cand_n);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const ss_topk &t, int64_t n_q, int64_t item_base, float *best_val,
                              int64_t *best_item, int sm_count, cudaStream_t s) {
  if (n_q == 0) return cudaSuccess;
  const int64_t need = (n_q + 7) / 8;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count * 16));
  k_topk_merge<<<grid, 256, 0, s>>>(t, n_q, item_base, best_val, best_item);
  return cudaGetLastError();
}
