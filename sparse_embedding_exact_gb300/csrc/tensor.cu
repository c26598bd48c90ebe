// Tensor-core scoring path: the hot dimensions as a dense product on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory),
// the cold dimensions as exact fixed-point records added in the epilogue.
//
// What is computed is the sparse dot product of the blog post "Engineering
// practice for bulk similarity calculation over sparse embeddings", section
// 3.1 (u.v over the shared support), of rows normalised first (section 4.4
// normalises right after the product; here the inputs are normalised, which
// is the same cosine and keeps every operand in [-1, 1]).
//
// In BM25/TF-IDF data the head of the dictionary (section 3.2) is held by a
// large share of the rows: on a Zipf(1.1) law over 1.2M words, the 160 most
// frequent dimensions carry 98.7% of the expected 6.8 shared dimensions of a
// pair.  Those dimensions are multiplied as a dense [128 queries x 256 items
// x H] product per tile pair.  The tensor cores take 16-bit operands, so
// each normalised value x (|x| <= 1) is split as x = hi + lo with hi =
// fp16(x) and lo = fp16(x - hi) (the split of Dekker / Ogita-Rump-Oishi
// used for extended-precision dot products), and the tile accumulates
// hi_q lo_v + lo_q hi_v (first, while the sum is small) then hi_q hi_v in
// FP32: the dropped lo_q lo_v and the splitting error are below 2^-22 |x|
// (2^-25 absolute for values in fp16's subnormal range).
//
// The remaining ("cold") dimensions are few per pair (0.09 expected on the
// 1.2M-word workload with 160 hot dimensions).  Once per query matrix the
// queries' cold nonzeros are sorted into lists by dimension (a counting
// sort, one set of lists per slice of query rows), and for each chunk a
// records kernel walks every item's cold nonzeros against the lists of
// their dimensions (a dimension no query holds cold has an empty list) and
// writes one record per product, bucketed by (32 query rows, 32 items):
// the position inside the bucket and the product rounded to a fixed-point
// integer of resolution 2^-28.  The scorer's epilogue adds a bucket's
// records into a 32 x 32 integer tile in shared memory (integer sums do not
// depend on order, so the result is the same bit for bit for any launch
// shape and chunking), adds that to the tensor result and stores the tile.
//
// Scorer (k_tc_score): persistent, one block per SM, 18 warps.  Warp 0
// loads operand tiles with bulk asynchronous copies (a query tile's operand
// stays while the block works through its item tiles, whose four K-half
// sub-parts stream through two buffers); warp 1 allocates
// tensor memory and one of its threads issues the MMAs into one of two
// accumulators; warps 2-17 run the epilogue, four per quarter of the 128
// accumulator lanes (each takes two of the eight 32-column blocks), on one
// tile pair while the MMAs of the next run, and store each 32 x 32 tile
// with one bulk tensor copy.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <cmath>

#include <string.h>

#include <algorithm>
#include <mutex>

#include "internal.cuh"
#include "topk.cuh"

namespace {

using namespace tcp;

constexpr int kHotSlotsBits = 9;
constexpr int kHotSlots = 1 << kHotSlotsBits;  // <= kHotMax keys: load <= 0.31
static_assert(kHotMax <= kHotSlots / 3, "the hot table stays sparse");
constexpr int kSelSort = 256;                  // the chosen dims, sorted (a power of two >= kHotMax)
static_assert(kSelSort >= kHotMax && (kSelSort & (kSelSort - 1)) == 0, "bitonic sort size");
constexpr int kSelSlotsBits = 16;
constexpr int kSelSlots = 1 << kSelSlotsBits;  // selection table (global memory)
constexpr int64_t kSampleEntries = 32768;      // nonzeros sampled to choose the hot set
constexpr int kSelThreads = 1024;
constexpr float kFixScale = 268435456.0f;      // 2^28: cold records' fixed point
constexpr float kFixInv = 1.0f / 268435456.0f;
constexpr float kMaxNormalised = 1.0f + 1.0f / 1024.0f;  // |x| of a normalised value
constexpr float kMaxSquareSum = 1.0f + 1.0f / 64.0f;     // sum of x^2 of a normalised row
constexpr int kStgInts = 32 * 32;              // one staging tile: 32 rows x 32 ints, 128-byte swizzle
constexpr int kBBufs = 2;                      // scorer: item sub-part buffers
constexpr int kEpiWarps = 16;                  // four per quarter of the accumulator lanes
constexpr int kWarpsPerQ = kEpiWarps / 4;      // epilogue warps per quarter
constexpr int kMine = 8 / kWarpsPerQ;          // 32-column blocks per warp and tile pair
constexpr int kSThreads = 64 + 32 * kEpiWarps; // producer, MMA, epilogue warps
constexpr int kStgTiles = kEpiWarps <= 8 ? 2 : 1;  // staging tiles per epilogue warp
constexpr int kStgBytes = kEpiWarps * kStgTiles * kStgInts * 4 + 1024;  // 1024-byte aligned
constexpr int kTailRecs = 128;                 // epilogue: a block's records past the register set staged in
                                               // shared memory (two slots per warp)
constexpr int kTailBytes = kEpiWarps * 2 * kTailRecs * 8;
static_assert(kEpiWarps % 4 == 0 && 8 % kWarpsPerQ == 0, "whole blocks per epilogue warp");
constexpr int kRThreads = 512;          // records: a block per 32-item column block, two per SM
constexpr int64_t kRecMaxQuarters = 16384;  // records: bucket counters in shared memory up to this many
constexpr double kRecSliceBytes = 48.0 * (1 << 20);  // records: expected bytes of one launch's buckets
constexpr int kPrepThreads = 256;
constexpr int kWalkUnroll = 8;          // list entries per lane loaded before use
constexpr int kRecPerLane = 4;          // epilogue: a block's first records per lane (128), fetched two blocks ahead
constexpr long long kWaitNs = 2000000000ll;    // bounded waits: 2 s

__device__ __forceinline__ void flag(int32_t *status, int32_t code) { atomicCAS(status, DEV_OK, code); }

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of `parity` to complete, for at most kWaitNs; false
// (and a DEV_STALL flag) when it runs out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t *status) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) {
      flag(status, DEV_STALL);
      return false;
    }
  }
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16),
// completing as transaction bytes on `bar`, with an L2 policy for the
// source lines.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
               : "memory");
}
// An L2 policy that keeps the lines it marks last: the operand tiles, read
// again by the blocks that score their other tile pairs.
__device__ __forceinline__ uint64_t evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Shared-memory matrix descriptor: K-major operand without swizzle, made of
// core matrices of 8 rows x 16 bytes (128 contiguous bytes); lbo = bytes
// between core matrices adjacent in K, sbo = bytes between adjacent groups
// of 8 rows.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (fp16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}
// Arrives on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// Element (r, c) of a 32 x 32 int staging tile with 16-byte chunk j of row r
// stored at chunk j ^ (r % 8): both the row-per-lane and the
// chunk-per-lane accesses of the epilogue are then free of bank conflicts.
__device__ __forceinline__ int stg_index(int r, int c) { return r * 32 + ((((c >> 2) ^ (r & 7)) << 2) | (c & 3)); }
// The fixed-point cold product of a normalised query value and a
// normalised list value (the records and the scorer's direct path agree on
// it bit for bit).
__device__ __forceinline__ int cold_fix(float qv, float vv) { return __float2int_rn((qv * vv) * kFixScale); }

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory writes of this thread made visible to the asynchronous
// (bulk copy) proxy.
__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk tensor store of a box (the tensor map's 32 x 32 floats, 128-byte
// swizzle) from shared memory to the tile at element (x, y), added to this
// thread's bulk group.  Parts of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int x, int y, uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;"
               ::"l"(tmap), "r"(src), "r"(x), "r"(y), "l"(policy)
               : "memory");
}
// An L2 policy that evicts the lines it marks first: the output, written
// once and never read back here, should not push the operands and records
// that the block still reads out of the cache.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Brings the 128-byte line holding p into this SM's L1 (no register).
__device__ __forceinline__ void prefetch_l1(const void *p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }
// Asynchronous 8-byte copy global -> shared memory by this thread (grouped
// by cp_async_commit, waited for by cp_async_wait1).
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Until all but the most recent of this thread's copy groups have landed.
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until all of this thread's bulk store groups have read their
// shared-memory source.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Until all but the most recent of this thread's bulk store groups have
// read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Until this thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Read-only loads issued exactly where they are written: the compiler may
// otherwise sink a plain load to its first use, which defeats a prefetch.
__device__ __forceinline__ int2 ld_keep_int2(const int2 *p) {
  int2 v;
  asm volatile("ld.global.nc.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ int ld_keep_int(const int32_t *p) {
  int v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------- hot table
// Dimension -> position in the ascending hot list, for <= kHotMax keys.
__device__ __forceinline__ uint32_t hot_hash(int32_t k) {
  return ((uint32_t)k * 0x9E3779B1u) >> (32 - kHotSlotsBits);
}
__device__ __forceinline__ int load_hot(const int32_t *hot, int *keys, uint8_t *vals) {
  for (int j = threadIdx.x; j < kHotSlots; j += blockDim.x) keys[j] = -1;
  __syncthreads();
  const int H = hot[0];
  for (int j = threadIdx.x; j < H; j += blockDim.x) {
    const int32_t k = hot[1 + j];
    uint32_t s = hot_hash(k);
    for (int n = 0; n < kHotSlots; ++n) {
      if (atomicCAS(&keys[s], -1, k) == -1) {
        vals[s] = (uint8_t)j;
        break;
      }
      s = (s + 1) & (kHotSlots - 1);
    }
  }
  __syncthreads();
  return H;
}
__device__ __forceinline__ int find_hot(const int *keys, const uint8_t *vals, int32_t k) {
  if (k < 0) return -1;  // empty slots hold -1; no hot dimension is negative
  uint32_t s = hot_hash(k);
  for (int n = 0; n < kHotSlots; ++n) {
    const int key = keys[s];
    if (key == k) return vals[s];
    if (key == -1) return -1;
    s = (s + 1) & (kHotSlots - 1);
  }
  return -1;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// ---------------------------------------------------------------- hot set
// Counts the dimensions of n_sample evenly spaced item rows in a global
// open-addressing table (keys then counts, kSelSlots each).
__global__ void __launch_bounds__(256)
    k_tc_sel_insert(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                    int64_t n_rows, int64_t n_sample, int32_t *__restrict__ tab) {
  int32_t *keys = tab, *cnts = tab + kSelSlots;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * 8;
  for (int64_t j = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); j < n_sample; j += warps) {
    const int64_t r = j * n_rows / n_sample;
    for (int64_t p = indptr[r] + lane; p < indptr[r + 1]; p += 32) {
      const int32_t k = indices[p];
      uint32_t s = ((uint32_t)k * 0x9E3779B1u) >> (32 - kSelSlotsBits);
      for (int n = 0; n < 256; ++n) {  // a full neighbourhood drops the sample
        const int prev = atomicCAS(&keys[s], -1, k);
        if (prev == -1 || prev == k) {
          atomicAdd(&cnts[s], 1);
          break;
        }
        s = (s + 1) & (kSelSlots - 1);
      }
    }
  }
}

// Ascending bitonic sort of n (a power of two) 64-bit keys in shared memory
// by the whole block.
__device__ void block_sort(unsigned long long *v, int n) {
  for (int k = 2; k <= n; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const unsigned long long x = v[i], y = v[ixj];
          if ((x > y) == up) {
            v[i] = y;
            v[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
}

// Visits the selection table's slots [64 t, 64 t + 64) as f(key, count),
// their loads issued 16 slots at a time (the table lives in global memory).
template <typename F>
__device__ __forceinline__ void for_my_slots(const int32_t *keys, const int32_t *cnts, int t, F f) {
  static_assert(kSelSlots == 64 * kSelThreads, "one run of 64 slots per thread");
#pragma unroll 1
  for (int h = 0; h < 4; ++h) {
    int4 k4[4], c4[4];
    const int base = 64 * t + 16 * h;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      k4[q] = *reinterpret_cast<const int4 *>(keys + base + 4 * q);
      c4[q] = *reinterpret_cast<const int4 *>(cnts + base + 4 * q);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f(k4[q].x, c4[q].x);
      f(k4[q].y, c4[q].y);
      f(k4[q].z, c4[q].z);
      f(k4[q].w, c4[q].w);
    }
  }
}

constexpr int kCountBins = 1024;  // sampled counts at or above the last bin share it
constexpr int kTieCap = 4096;     // dimensions tied at the threshold count that are ranked

// One block.  The hot set: the (at most kHotMax) most frequent sampled
// dimensions held by at least max(2, 0.2% of the sampled rows), ties to the
// lower dimension (counts of kCountBins - 1 or more count as equal); hot[0]
// = H, hot[1..H] ascending.  The threshold comes from a histogram of the
// counts; the dimensions tied at it are sorted, and when more than kTieCap
// are tied none of them is taken.  stats[0]: the sampled rows' expected
// number of shared dimensions outside the hot set per pair of rows, sum
// c (c - 1) / (n (n - 1)) over the other dimensions' counts c (an unbiased
// estimate of their sum of squared frequencies); stats[1] = H.
__global__ void __launch_bounds__(kSelThreads)
    k_tc_sel_pick(const int32_t *__restrict__ tab, int64_t n_sample, int32_t *__restrict__ hot,
                  float *__restrict__ stats) {
  const int32_t *keys = tab, *cnts = tab + kSelSlots;
  __shared__ int hist[kCountBins];
  __shared__ unsigned long long ties[kTieCap];
  __shared__ unsigned long long sel[kSelSort];
  __shared__ int n_above, n_ties, thr_sh, take_ties;
  __shared__ unsigned long long pairs_all, pairs_hot;
  const int tid = threadIdx.x;
  for (int j = tid; j < kCountBins; j += kSelThreads) hist[j] = 0;
  for (int j = tid; j < kSelSort; j += kSelThreads) sel[j] = ~0ull;
  for (int j = tid; j < kTieCap; j += kSelThreads) ties[j] = ~0ull;
  if (tid == 0) {
    n_above = n_ties = 0;
    pairs_all = pairs_hot = 0ull;
  }
  __syncthreads();
  const int floor_c = min(kCountBins - 1, max(2, (int)((n_sample * 2 + 999) / 1000)));
  unsigned long long my_pairs = 0;
  // Most sampled dimensions share a few small counts: the histogram adds
  // are combined per warp (one atomic per distinct bin of the warp).
  for_my_slots(keys, cnts, tid, [&](int key, int c) {
    const bool in = key >= 0 && c >= floor_c;
    if (key >= 0) my_pairs += (unsigned long long)c * (unsigned long long)(c - 1);
    const int bin = in ? min(c, kCountBins - 1) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    if (in && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) my_pairs += __shfl_xor_sync(0xffffffffu, my_pairs, o);
  if ((tid & 31) == 0) atomicAdd(&pairs_all, my_pairs);
  if (tid == 0) {
    thr_sh = -1;
    take_ties = 0;
  }
  __syncthreads();
  {
    // The threshold: the largest bin t where the dimensions in bins > t are
    // fewer than kHotMax and those in bins >= t reach it (-1 when all of
    // them fit).  Thread i takes bin kCountBins - 1 - i, so a scan over the
    // threads gives each bin the count of the bins at or above it.
    static_assert(kCountBins == kSelThreads, "one count bin per thread");
    __shared__ int wsum[kSelThreads / 32];
    const int lane = tid & 31, w = tid >> 5;
    const int c = kCountBins - 1 - tid;
    const int hc = hist[c];
    const int inc = warp_incl_scan(hc, lane);
    if (lane == 31) wsum[w] = inc;
    __syncthreads();
    int before = 0;
    for (int k = 0; k < w; ++k) before += wsum[k];
    const int at_or_above = before + inc, above = at_or_above - hc;
    if (c >= floor_c && at_or_above >= kHotMax && above < kHotMax) {
      thr_sh = c;  // one bin at most: the counts only grow as c falls
      take_ties = hc <= kTieCap;
    }
  }
  __syncthreads();
  const int thr = thr_sh;
  for_my_slots(keys, cnts, tid, [&](int kd, int c) {
    if (kd < 0 || c < floor_c) return;
    const int cc = min(c, kCountBins - 1);
    const unsigned long long key = ((unsigned long long)(uint32_t)kd << 32) | (uint32_t)c;
    if (thr < 0 || cc > thr) {
      sel[atomicAdd(&n_above, 1)] = key;  // fewer than kHotMax of them
    } else if (cc == thr && take_ties) {
      ties[atomicAdd(&n_ties, 1)] = key;
    }
  });
  __syncthreads();
  int nt = 1;
  while (nt < n_ties) nt <<= 1;
  block_sort(ties, nt);  // lower dimensions first
  const int above = n_above;
  const int need = min(kHotMax - above, n_ties);
  for (int j = tid; j < need; j += kSelThreads) sel[above + j] = ties[j];
  __syncthreads();
  block_sort(sel, kSelSort);
  const int H = above + max(need, 0);
  unsigned long long hp = 0;
  for (int j = tid; j < H; j += kSelThreads) {
    hot[1 + j] = (int32_t)(sel[j] >> 32);
    const unsigned long long c = sel[j] & 0xffffffffull;
    hp += c * (c - 1);
  }
  atomicAdd(&pairs_hot, hp);
  __syncthreads();
  if (tid == 0) {
    hot[0] = H;
    const double ns = (double)n_sample;
    stats[0] = ns > 1.0 ? (float)((double)(pairs_all - pairs_hot) / (ns * (ns - 1.0))) : 0.f;
    stats[1] = (float)H;
  }
}

// ---------------------------------------------------------------- build
// The build does not depend on the queries: one pass over the chunk's CSR
// rows (a warp per row, no atomics) writes each item's raw hot values into
// the dense slab (0 where absent), its sum of squares, and its cold entries
// {dim, raw value bits} packed in CSR order (dims ascending) at the row's
// own positions relative to the build's first nonzero, with {first, count}
// per item.  Each scoring call's records kernel walks these entries item by
// item, each into the queries' list of its dimension.
__global__ void __launch_bounds__(256)
    k_tc_build(const int64_t *__restrict__ indptr, const int32_t *__restrict__ indices,
               const float *__restrict__ values, int64_t row_begin, int64_t row_end, int64_t chunk_rows,
               int64_t dim, const int32_t *__restrict__ hot, float *__restrict__ slab,
               float *__restrict__ sq, int2 *__restrict__ icold, int2 *__restrict__ icold_rng,
               int32_t *status) {
  __shared__ int hkeys[kHotSlots];
  __shared__ uint8_t hvals[kHotSlots];
  load_hot(hot, hkeys, hvals);
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const int64_t p_base = indptr[row_begin];
  const int64_t warps = (int64_t)gridDim.x * 8;
  bool bad = false;
  for (int64_t r = row_begin + (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < row_end; r += warps) {
    const int64_t b = indptr[r], e = indptr[r + 1];
    const int64_t c = (r - row_begin) / chunk_rows;
    const int64_t item = r - row_begin - c * chunk_rows;
    float *srow = slab + (c * chunk_rows + item) * kHotMax;  // this item's hot values, zero if absent
    static_assert(kHotMax % 4 == 0, "an item's hot values are cleared as float4s");
    for (int h = 4 * lane; h < kHotMax; h += 128) *reinterpret_cast<float4 *>(srow + h) = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncwarp();
    float ss = 0.f;
    int nc = 0;
    for (int64_t j0 = b; j0 < e; j0 += 32) {
      const int64_t j = j0 + lane;
      bool cold = false;
      int32_t k = 0;
      float v = 0.f;
      if (j < e) {
        k = __ldg(indices + j);
        v = __ldg(values + j);
        ss = fmaf(v, v, ss);
        if (k >= 0 && (int64_t)k < dim) {
          const int h = find_hot(hkeys, hvals, k);
          if (h >= 0) srow[h] = v;
          else cold = true;
        } else {
          bad = true;
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, cold);
      if (cold) icold[(b - p_base) + nc + __popc(m & lt)] = make_int2(k, __float_as_int(v));
      nc += __popc(m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) {
      sq[c * chunk_rows + item] = ss;
      icold_rng[c * chunk_rows + item] = make_int2((int)(b - p_base), nc);
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag(status, DEV_OUT_OF_RANGE);
}

// The queries' lists, once per query matrix, inverse norms and hot set: a
// counting sort of the queries' cold entries by (slice of query rows,
// dimension), each slice holding its own set of d + 1 offsets.  A records
// launch walks one slice's lists, so that the buckets it fills at once
// stay few enough for their partly written lines to remain in L2.  The counts per
// dimension (k_tc_qcount), their exclusive scan (launch_count_scan: list d
// is entries [qptr[d], qptr[d + 1]) and is empty for a dimension no query
// row holds cold; the scan leaves each counter at its list's start), then
// the scatter (k_tc_qscatter), which takes each entry's place from its
// dimension's counter and writes {query row, normalised value bits}.  A list's order is unspecified:
// the records it makes are summed as integers.  Every scoring call walks
// the same lists from its chunk's items, so nothing is sorted per chunk.
__global__ void __launch_bounds__(256)
    k_tc_qcount(const int64_t *__restrict__ q_indptr, const int2 *__restrict__ qcold,
                const int32_t *__restrict__ qcold_n, int64_t n_q, int64_t slice_rows, int64_t stride,
                int32_t *__restrict__ count) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * 8;
  for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < n_q; r += warps) {
    const int64_t b = q_indptr[r];
    const int n = qcold_n[r];
    int32_t *cnt = count + (r / slice_rows) * stride;
    for (int j = lane; j < n; j += 32) atomicAdd(cnt + __ldg(qcold + b + j).x, 1);
  }
}

__global__ void __launch_bounds__(256)
    k_tc_qscatter(const int64_t *__restrict__ q_indptr, const int2 *__restrict__ qcold,
                  const int32_t *__restrict__ qcold_n, int64_t n_q, int64_t slice_rows, int64_t stride,
                  int32_t *__restrict__ cursor, int2 *__restrict__ qlist) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * 8;
  for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < n_q; r += warps) {
    const int64_t b = q_indptr[r];
    const int n = qcold_n[r];
    int32_t *cur = cursor + (r / slice_rows) * stride;
    for (int j = lane; j < n; j += 32) {
      const int2 e = __ldg(qcold + b + j);
      qlist[atomicAdd(cur + e.x, 1)] = make_int2((int)r, e.y);
    }
  }
}

// ---------------------------------------------------------------- operands
// An operand tile of R rows (R = kM queries or kN items) with Hp hot columns
// is stored as two parts, hi then lo, each in the no-swizzle K-major layout:
// 8-row groups of Hp / 8 core matrices (8 rows x 8 halves, 128 bytes), so a
// part is R * Hp halves and element (r, k) of a part sits at
// (r / 8) * 8 Hp + (k / 8) * 64 + (r % 8) * 8 + k % 8.
__device__ __forceinline__ int core_off(int r8, int k) { return (k >> 3) * 64 + r8 * 8 + (k & 7); }

struct PrepArgs {
  const int64_t *indptr;  // queries: the CSR
  const int32_t *idx;
  const float *val;
  const float *slab;      // items: [item][kHotMax] raw hot values of the chunk
  const float *sq;        // items: raw sum of squares per item
  int64_t n_rows;         // rows of the matrix (queries) or of the chunk (items)
  int64_t n_groups;       // 8-row groups to write (whole tiles)
  const float *inv;       // inverse norms of those rows
  const int32_t *hot;
  int32_t Hp;
  int32_t gpt;            // 8-row groups per tile (kM / 8 or kN / 8)
  uint16_t *op;           // operand tiles (hi part, lo part)
  int2 *qcold;            // queries: {dim, normalised value bits} at the row's CSR positions
  int32_t *qcold_n;       // queries: cold entries per row
  int64_t dim;            // queries: indices outside [0, dim) are left out and reported
  int32_t *status;
};

// The warp's group buffer holds the group's hi part ([0, 8 Hp) halves) then
// its lo part.
__device__ __forceinline__ void put_split(uint16_t *gs, int rr, int h, int Hp, float x) {
  const __half hi = __float2half_rn(x);
  const __half lo = __float2half_rn(x - __half2float(hi));
  gs[core_off(rr, h)] = __half_as_ushort(hi);
  gs[8 * Hp + core_off(rr, h)] = __half_as_ushort(lo);
}

// Writes a group buffer to group g of an operand (queries or items) whose
// tiles hold four sub-parts in the order the MMAs read them: lo part K columns
// [0, Hp/2), lo part [Hp/2, Hp), hi part [0, Hp/2), hi part [Hp/2, Hp); each
// sub-part is `gpt` groups of 8 rows x Hp/2 halves in the same no-swizzle
// K-major layout (in the group buffer a part's two halves are already
// contiguous: core matrices of K columns >= Hp/2 follow those below).
__device__ __forceinline__ void store_group_q(uint16_t *op, const uint16_t *gs, int64_t g, int gpt, int Hp,
                                              int lane) {
  const int64_t t = g / gpt, gl = g % gpt;
  const int P = 4 * Hp;  // halves of one group sub-part (8 rows x Hp / 2)
  uint16_t *tile = op + t * 4 * gpt * P + gl * P;
  const int src[4] = {2 * P, 3 * P, 0, P};  // lo K0, lo K1, hi K0, hi K1 in the group buffer
#pragma unroll
  for (int sp = 0; sp < 4; ++sp)
    for (int o = lane * 8; o < P; o += 256)
      *reinterpret_cast<uint4 *>(tile + (int64_t)sp * gpt * P + o) = *reinterpret_cast<const uint4 *>(gs + src[sp] + o);
}

// One warp per group of 8 query rows: the rows' normalised hot values split
// into fp16 hi (K columns [0, Hp)) and lo (columns [Hp, 2 Hp)), zero
// elsewhere, and the cold nonzeros in CSR order.  Checks that the inverse
// norms are the rows' own (every |x| <= 1 + 2^-10, sum x^2 <= 1 + 2^-6).
__global__ void __launch_bounds__(kPrepThreads) k_tc_prep_queries(const PrepArgs a) {
  __shared__ int hkeys[kHotSlots];
  __shared__ uint8_t hvals[kHotSlots];
  __shared__ __align__(16) uint16_t grp[kPrepThreads / 32][8 * 2 * kHotMax];
  load_hot(a.hot, hkeys, hvals);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int Hp = a.Hp, G = 16 * Hp;  // halves per group
  uint16_t *gs = grp[warp];
  bool bad = false, outside = false;
  for (int64_t g = (int64_t)blockIdx.x * (kPrepThreads / 32) + warp; g < a.n_groups;
       g += (int64_t)gridDim.x * (kPrepThreads / 32)) {
    for (int o = lane * 8; o < G; o += 256) *reinterpret_cast<uint4 *>(gs + o) = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    for (int rr = 0; rr < 8; ++rr) {
      const int64_t r = g * 8 + rr;
      if (r >= a.n_rows) break;
      const int64_t b = a.indptr[r], e = a.indptr[r + 1];
      const float iv = a.inv[r];
      float ss = 0.f;
      int nc = 0;
      for (int64_t p0 = b; p0 < e; p0 += 32) {
        const int64_t p = p0 + lane;
        const bool have = p < e;
        int32_t k = -1;
        float x = 0.f;
        int h = -1;
        if (have) {
          k = __ldg(a.idx + p);
          x = __ldg(a.val + p) * iv;
          ss = fmaf(x, x, ss);
          bad |= !(fabsf(x) <= kMaxNormalised);
          if (k < 0 || (int64_t)k >= a.dim) {
            outside = true;
            h = -2;  // neither hot nor a cold entry (and never looked up: -1 marks empty slots)
          } else {
            h = find_hot(hkeys, hvals, k);
            if (h >= 0) put_split(gs, rr, h, Hp, x);
          }
        }
        const bool cold = have && h == -1;
        const unsigned m = __ballot_sync(0xffffffffu, cold);
        if (cold) a.qcold[b + nc + __popc(m & lt)] = make_int2(k, __float_as_int(x));
        nc += __popc(m);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      bad |= !(ss <= kMaxSquareSum);
      if (lane == 0) a.qcold_n[r] = nc;
    }
    __syncwarp();
    store_group_q(a.op, gs, g, a.gpt, Hp, lane);
    __syncwarp();
  }
  if (__any_sync(0xffffffffu, outside) && lane == 0) flag(a.status, DEV_OUT_OF_RANGE);
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag(a.status, DEV_RANGE);
}

// The item operand of a chunk from its hot slab, written without a shared
// staging buffer: a warp takes a group of 8 items, and lane l the 16-byte
// chunks (item l % 8, K columns 8 kc .. + 7) for kc = l / 8, l / 8 + 4, ...:
// eight slab values, normalised and split, give one hi chunk and one lo
// chunk, each stored whole at its place in the K-half sub-part (a warp's
// 32 stores of a part are four 128-byte runs).  Every K column is written,
// zeros past the chunk; the inverse norms are checked against the items'
// sums of squares.  Runs as the trailing blocks of the records launch.
__device__ void prep_item_groups(const PrepArgs &a, int64_t g0, int64_t stride, int lane) {
  const int Hp = a.Hp, Kc = Hp / 8, halfKc = Kc / 2;  // 16-byte K chunks in all, in one K half
  const int r8 = lane & 7, kq = lane >> 3;
  const int P = 4 * Hp;  // halves of one group sub-part (8 rows x Hp / 2)
  bool bad = false;
  for (int64_t g = g0; g < a.n_groups; g += stride) {
    const int64_t r = g * 8 + r8;
    const bool in = r < a.n_rows;
    const float iv = in ? __ldg(a.inv + r) : 0.f;
    if (in && kq == 0) bad |= !(__ldg(a.sq + r) * iv * iv <= kMaxSquareSum);
    const int64_t t = g / a.gpt, gl = g % a.gpt;
    uint16_t *tile = a.op + t * 4 * a.gpt * P + gl * P;
    for (int kc = kq; kc < Kc; kc += 4) {
      float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
      if (in) {
        const float4 *src = reinterpret_cast<const float4 *>(a.slab + r * kHotMax + 8 * kc);
        v0 = __ldg(src);
        v1 = __ldg(src + 1);
      }
      const float x[8] = {v0.x * iv, v0.y * iv, v0.z * iv, v0.w * iv, v1.x * iv, v1.y * iv, v1.z * iv, v1.w * iv};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        bad |= !(fabsf(x[2 * e]) <= kMaxNormalised) || !(fabsf(x[2 * e + 1]) <= kMaxNormalised);
        const __half h0 = __float2half_rn(x[2 * e]), h1 = __float2half_rn(x[2 * e + 1]);
        const __half l0 = __float2half_rn(x[2 * e] - __half2float(h0));
        const __half l1 = __float2half_rn(x[2 * e + 1] - __half2float(h1));
        hi[e] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
        lo[e] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
      }
      const int khalf = kc >= halfKc ? 1 : 0, kk = kc - khalf * halfKc;
      const int off = kk * 64 + r8 * 8;  // the chunk inside its group sub-part
      // sub-parts: 0 lo K0, 1 lo K1, 2 hi K0, 3 hi K1
      *reinterpret_cast<uint4 *>(tile + (int64_t)(0 + khalf) * a.gpt * P + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4 *>(tile + (int64_t)(2 + khalf) * a.gpt * P + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag(a.status, DEV_RANGE);
}

// ---------------------------------------------------------------- records
// The cold products of one scoring call become records {position in the
// 32 x 32 swizzled staging tile of their bucket, fixed-point product}, a
// bucket being (32 query rows, 32 items) with room for bucket_cap records
// and a count (-1 when its records did not fit; the scorer then computes
// the bucket from the lists).
struct RecArgs {
  const int2 *icold;       // the chunk's items' cold entries {dim, raw value bits}
  const int2 *icold_rng;   // per item of the chunk: {first entry, count}
  int32_t n_items;
  const float *inv_i;      // the chunk's inverse norms
  const int32_t *qptr;     // the slice's lists: [dim + 1] offsets into qlist
  const int2 *qlist;       // {query row, normalised value bits}
  int64_t q0;              // the slice's first quarter (32-row group of queries)
  int64_t n_quarters;      // the slice's quarters
  int32_t n_cb;            // 32-item column blocks of the chunk
  int32_t bucket_cap;      // records a bucket holds
  int2 *rec;               // [quarter][column block][bucket_cap]
  int32_t *rec_n;          // [quarter][column block]
  int32_t *status;
  int64_t n_main;          // column blocks with a block of their own (whole waves of blocks)
  int64_t n_shared;        // blocks sharing the items of the column blocks after those
  int32_t pieces;          // main blocks: the parts each item's walk is cut into
  PrepArgs prep;           // the chunk's item operand (the blocks after all of these)
};

// Calls f(query row, product) for every cold product of item `it` with the
// queries.  One warp takes the item's cold entries 32 at a time and lays
// the queries' lists of their dimensions end to end; each lane then takes
// one list entry of every window of 32, finding its list from the bits
// that mark where lists start inside the window (a lane's list is the last
// one that starts at or before it).  The item's value is normalised once
// per entry; the product is the same fp32 product of the two normalised
// values, whichever side is walked.
template <typename F>
__device__ __forceinline__ void walk_item(const RecArgs &a, int it, int lane, int4 *slots, F f, int piece = 0,
                                          int pieces = 1) {
  const int2 rng = __ldg(a.icold_rng + it);
  const float ivi = __ldg(a.inv_i + it);
  const unsigned lt = (1u << lane) - 1u, lt_eq = (2u << lane) - 1u;
  for (int b0 = 0; b0 < rng.y; b0 += 32) {
    int s = 0, len = 0;
    float iv = 0.f;
    if (b0 + lane < rng.y) {
      const int2 e = __ldg(a.icold + rng.x + b0 + lane);
      iv = __int_as_float(e.y) * ivi;
      s = __ldg(a.qptr + e.x);
      len = __ldg(a.qptr + e.x + 1) - s;
    }
    // The non-empty lists move to the first lanes, in order.
    const unsigned nz = __ballot_sync(0xffffffffu, len > 0);
    if (len > 0) slots[__popc(nz & lt)] = make_int4(s, len, __float_as_int(iv), 0);
    __syncwarp();
    if (lane < __popc(nz)) {
      const int4 v = slots[lane];
      s = v.x;
      len = v.y;
      iv = __int_as_float(v.z);
    } else {
      s = 0;
      len = 0;
      iv = 0.f;
    }
    __syncwarp();
    const int incl = warp_incl_scan(len, lane);
    const int excl = incl - len;
    const int L = __shfl_sync(0xffffffffu, incl, 31);
    // Windows of 32 entries piece, piece + pieces, ... (all of them when
    // the walk is not shared), kWalkUnroll at a time.
    for (int base = piece; 32 * base < L; base += pieces * kWalkUnroll) {
      int pos[kWalkUnroll];
      float pv[kWalkUnroll];
      bool ok[kWalkUnroll];
#pragma unroll
      for (int u = 0; u < kWalkUnroll; ++u) {
        const int w0 = 32 * (base + pieces * u), fi = w0 + lane;
        const unsigned before = __ballot_sync(0xffffffffu, incl <= w0);  // lists ending at or before w0
        const bool starts = len > 0 && excl >= w0 && excl < w0 + 32;
        const unsigned m = __reduce_or_sync(0xffffffffu, starts ? (1u << ((excl - w0) & 31)) : 0u);
        const int first = __popc(before);  // the list holding entry w0 (if any entry is left)
        // If no list starts at w0 itself, entry w0 continues list `first`.
        const int j = first + __popc(m & lt_eq) - ((m & 1u) ? 1 : 0);
        const int jj = j < 31 ? j : 31;
        const int sj = __shfl_sync(0xffffffffu, s, jj);
        const int ej = __shfl_sync(0xffffffffu, excl, jj);
        pv[u] = __shfl_sync(0xffffffffu, iv, jj);
        ok[u] = fi < L;
        pos[u] = sj + (fi - ej);
      }
      int2 qe[kWalkUnroll];
#pragma unroll
      for (int u = 0; u < kWalkUnroll; ++u) {
        qe[u] = make_int2(0, 0);
        if (ok[u]) qe[u] = ld_keep_int2(a.qlist + pos[u]);
      }
#pragma unroll
      for (int u = 0; u < kWalkUnroll; ++u)
        if (ok[u]) f(qe[u].x, cold_fix(__int_as_float(qe[u].y), pv[u]));
    }
  }
}

// Every cold product of an item with the queries becomes a record in the
// bucket of its (32 rows, 32 items), at a slot taken from the bucket's
// counter (the order inside a bucket does not matter: the epilogue sums
// integers).  A column block gets a block of its own (its 32 items taken a
// warp at a time, a counter per quarter in shared memory) when the column
// blocks fill whole waves of blocks, or one wave that gives every SM a
// block; otherwise the items of the column blocks past the whole waves are
// shared by all warps of one more wave of blocks (several warps per item
// when there are few, counters in global memory).  Blocks after those
// write the item operand.
__global__ void __launch_bounds__(kRThreads, 2) k_tc_records(const RecArgs a) {
  const int64_t bid = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ncb = a.n_cb, cap = a.bucket_cap;
  if (bid >= a.n_main + a.n_shared) {  // a trailing block: the item operand, a warp per group
    const int64_t warps = (int64_t)(gridDim.x - a.n_main - a.n_shared) * (kRThreads / 32);
    prep_item_groups(a.prep, (bid - a.n_main - a.n_shared) * (kRThreads / 32) + warp, warps, lane);
    return;
  }
  __shared__ int4 slots_all[kRThreads / 32][32];
  int4 *slots = slots_all[warp];
  if (bid >= a.n_main) {
    // The items past the main column blocks, shared by every warp of these
    // blocks: item e gets `pieces` warps, warp k of them walking the windows
    // k, k + pieces, ... of its lists (when the items outnumber the warps,
    // each warp takes every warps-th item).  Their buckets are counted in
    // global memory (zeroed before the launch): a count above the bucket's
    // room marks it as not fitting.
    const int64_t item0 = a.n_main * 32, items = a.n_items - item0;
    const int64_t warps = a.n_shared * (kRThreads / 32);
    const int64_t per_item = warps / (items > 0 ? items : 1);
    const int pieces = (int)(per_item > 1 ? per_item : 1);
    for (int64_t w = (bid - a.n_main) * (kRThreads / 32) + warp; w < items * pieces; w += warps) {
      const int it = (int)(item0 + w % items);
      const int piece = (int)(w / items);
      const int cb = it >> 5, il = it & 31;
      walk_item(
          a, it, lane, slots,
          [&](int q, int p) {
            const int64_t Q = q >> 5;
            const int slot = atomicAdd(a.rec_n + Q * ncb + cb, 1);
            if (slot < cap) a.rec[(Q * ncb + cb) * cap + slot] = make_int2(stg_index(q & 31, il), p);
          },
          piece, pieces);
    }
    return;
  }
  extern __shared__ int rcnt[];  // [n_quarters] from q0
  const int tid = threadIdx.x;
  const int64_t cb = bid;
  const int nqt = (int)a.n_quarters;
  __shared__ int next_part;
  if (tid == 0) next_part = 0;
  for (int c = tid; c < nqt; c += kRThreads) rcnt[c] = 0;
  __syncthreads();
  // The block's 32 items, each cut into `pieces` parts (part k walks the
  // windows k, k + pieces, ... of the item's lists): a warp takes the next
  // part as it finishes one, so items of unequal length even out.
  const int parts = 32 * a.pieces;
  for (;;) {
    int u = 0;
    if (lane == 0) u = atomicAdd(&next_part, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= parts) break;
    const int il = u & 31, piece = u >> 5;
    const int it = (int)(cb * 32 + il);
    if (it < a.n_items)
      walk_item(
          a, it, lane, slots,
          [&](int q, int p) {
            const int Q = q >> 5;
            const int slot = atomicAdd(&rcnt[Q - a.q0], 1);
            if (slot < cap) a.rec[((int64_t)Q * ncb + cb) * cap + slot] = make_int2(stg_index(q & 31, il), p);
          },
          piece, a.pieces);
  }
  __syncthreads();
  for (int c = tid; c < nqt; c += kRThreads) a.rec_n[(a.q0 + c) * ncb + cb] = rcnt[c] <= cap ? rcnt[c] : -1;
}

// ---------------------------------------------------------------- scorer
struct ScoreArgs {
  CUtensorMap out_map;     // the output tile for bulk tensor stores (when use_tma)
  int32_t use_tma;         // device-memory output with 16-byte rows: stores by the tensor map
  const uint16_t *A;       // query operand tiles
  const uint16_t *B;       // item operand tiles
  const int2 *rec;         // the call's records (k_tc_records)
  const int32_t *rec_n;    // their counts per bucket (-1: did not fit)
  int32_t bucket_cap;
  // For buckets that did not fit: the chunk's items' cold entries and the
  // queries' lists.
  const int2 *icold;
  const int2 *icold_rng;
  const int32_t *qptr;     // slice s's offsets at qptr + s * qptr_stride
  int64_t qptr_stride;
  int64_t slice_rows;
  const int2 *qlist;
  const float *inv_i;
  int64_t n_quarters;
  int32_t n_cb;
  float *out;
  int64_t ld_out;
  int64_t n_q;
  int32_t n_items;
  int64_t n_qtiles;
  int64_t n_tiles;         // item tiles
  int64_t n_units;         // query tiles x item tiles
  int32_t Hp;
  int32_t vec_ok;          // 16-byte aligned output rows: vector stores
  int32_t use_tail;        // records past the register set staged in shared memory
  int32_t *status;
};

// Bytes of the scorer's dynamic shared memory for Hp hot columns: the query
// tile (hi, lo: 512 Hp), kBBufs buffers of one item sub-part (256 Hp each),
// the staging tiles of the epilogue, its staged records (kTailBytes, when
// they fit: at Hp = 128, not at Hp = 160).
size_t score_smem_bytes(int Hp, bool tail) {
  return (size_t)(512 + 256 * kBBufs) * Hp + kStgBytes + (tail ? kTailBytes : 0);
}
constexpr size_t kMaxDynSmem = 232448;  // shared memory a block may take
// Whether the staged records fit beside the operands at Hp hot columns.
bool score_tail_fits(int Hp) { return score_smem_bytes(Hp, true) <= kMaxDynSmem; }

// Ties registers just loaded from tensor memory to the wait that completes
// the load, so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_regs_ready(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                 "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                 "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

__global__ void __launch_bounds__(kSThreads, 1)
    k_tc_score(const __grid_constant__ ScoreArgs a) {
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ __align__(8) uint64_t bars[7 + 2 * kBBufs];
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hp = a.Hp;
  // The query tile (four sub-parts of 128 rows x Hp / 2 halves: lo K0,
  // lo K1, hi K0, hi K1) stays while the block works through its item
  // tiles; each item tile's four sub-parts (256 items x Hp / 2 halves, the
  // same order) stream through kBBufs buffers.
  const uint32_t bytesAsub = 128u * (uint32_t)Hp, bytesA = 4u * bytesAsub;
  const uint32_t bytesBsub = 256u * (uint32_t)Hp;
  unsigned char *sA = sm;
  unsigned char *sB = sm + bytesA;
  int *stg_all = reinterpret_cast<int *>(
      (reinterpret_cast<uintptr_t>(sB + kBBufs * bytesBsub) + 1023) & ~static_cast<uintptr_t>(1023));
  // bars[0]: query tile landed; bars[1]: query tile read by the MMAs;
  // bars[2..3]: accumulator b written (MMA commit); bars[4..5]: accumulator
  // b read out (one arrival per epilogue warp); bars[6]: the MMA thread's
  // last commit; then per item buffer: landed, read by the MMAs.
  const uint32_t a_full = smem_u32(&bars[0]), a_free = smem_u32(&bars[1]);
  const uint32_t acc_full0 = smem_u32(&bars[2]), acc_full1 = smem_u32(&bars[3]);
  const uint32_t acc_free0 = smem_u32(&bars[4]), acc_free1 = smem_u32(&bars[5]);
  const uint32_t drain = smem_u32(&bars[6]);
  auto b_full = [&](int buf) { return smem_u32(&bars[7 + buf]); };
  auto b_free = [&](int buf) { return smem_u32(&bars[7 + kBBufs + buf]); };
  if (tid == 0) {
    for (int i = 0; i < 7 + 2 * kBBufs; ++i) mbar_init(smem_u32(&bars[i]), 1);
    mbar_init(acc_free0, kEpiWarps);
    mbar_init(acc_free1, kEpiWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Units are (query tile g, item tile t) pairs, u = g * n_tiles + t; each
  // block takes a contiguous range, so its query tile rarely changes.
  const int64_t u0 = (int64_t)blockIdx.x * a.n_units / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * a.n_units / gridDim.x;
  const int64_t nj = u1 - u0;

  if (warp == 0) {
    // ---- producer: the query tile when it changes (once the MMAs have
    // released the previous one), then per unit the item tile's four
    // sub-parts, copy n into buffer n % kBBufs once the MMAs have released
    // that buffer's previous copy.
    if (lane == 0) {
      const uint64_t keep = evict_last_policy();
      int64_t prev_g = -1;
      int na = 0;        // query tile copies issued
      int64_t nbc = 0;   // item sub-part copies issued
      bool ok = true;
      for (int64_t j = 0; j < nj && ok; ++j) {
        const int64_t u = u0 + j, g = u / a.n_tiles, t = u % a.n_tiles;
        if (g != prev_g) {
          if (na > 0 && !(ok = mbar_wait(a_free, (uint32_t)((na - 1) & 1), a.status))) break;
          mbar_expect_tx(a_full, bytesA);
          bulk_g2s_hint(smem_u32(sA), a.A + (size_t)g * (bytesA / 2), bytesA, a_full, keep);
          ++na;
          prev_g = g;
        }
        const uint16_t *Bt = a.B + (size_t)t * (2 * (size_t)bytesBsub);  // 4 sub-parts of bytesBsub bytes
        for (int sp = 0; sp < 4; ++sp) {
          const int buf = (int)(nbc % kBBufs);
          const int64_t k = nbc / kBBufs;  // copies into this buffer before this one
          if (k > 0 && !(ok = mbar_wait(b_free(buf), (uint32_t)((k - 1) & 1), a.status))) break;
          mbar_expect_tx(b_full(buf), bytesBsub);
          bulk_g2s_hint(smem_u32(sB) + (uint32_t)buf * bytesBsub, Bt + (size_t)sp * (bytesBsub / 2), bytesBsub,
                        b_full(buf), keep);
          ++nbc;
        }
      }
      // Every copy issued lands before the block exits, also when a wait
      // above gave up: copy k into a buffer is issued only after the MMAs
      // released copy k - 1 (which had landed), so at most the last copy of
      // each buffer is in flight, and a bulk copy completes by itself.
      for (int buf = 0; buf < kBBufs; ++buf) {
        const int64_t n_buf = (nbc + kBBufs - 1 - buf) / kBBufs;  // copies issued into this buffer
        if (n_buf > 0) mbar_wait(b_full(buf), (uint32_t)((n_buf - 1) & 1), a.status);
      }
      if (na > 0) mbar_wait(a_full, (uint32_t)((na - 1) & 1), a.status);
    }
  } else if (warp == 1) {
    // ---- MMA issue, per unit: the cross terms hi_q x lo_v and lo_q x hi_v
    // first (while the sum is small), then hi_q x hi_v.
    if (lane == 0) {
      const uint32_t idesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
      const int Kp = Hp / 2;
      const uint32_t sbo = 16u * (uint32_t)Kp, lbo = 128u;
      const uint32_t aa = smem_u32(sA);
      const uint32_t a_lo0 = aa, a_lo1 = aa + bytesAsub, a_hi0 = aa + 2 * bytesAsub, a_hi1 = aa + 3 * bytesAsub;
      // The Kp-column product of a query sub-part with an item sub-part.
      auto mma_sub = [&](uint32_t d, uint32_t a_addr, uint32_t b_addr, bool first) {
        for (int kk = 0; kk < Kp; kk += 16)
          mma_f16(d, smem_desc(a_addr + (uint32_t)(kk / 8) * 128u, lbo, sbo),
                  smem_desc(b_addr + (uint32_t)(kk / 8) * 128u, lbo, sbo), idesc, (first && kk == 0) ? 0u : 1u);
      };
      int64_t prev_g = -1;
      int na = 0;
      int64_t nbc = 0;
      bool ok = true;
      uint32_t bb[4];
      int bufs[4];
      // Waits for item sub-part s of the current unit (copy nbc + s).
      auto wait_sub = [&](int s) -> bool {
        const int64_t n = nbc + s;
        const int buf = (int)(n % kBBufs);
        bufs[s] = buf;
        bb[s] = smem_u32(sB) + (uint32_t)buf * bytesBsub;
        return mbar_wait(b_full(buf), (uint32_t)((n / kBBufs) & 1), a.status);
      };
      for (int64_t j = 0; j < nj && ok; ++j) {
        const int64_t g = (u0 + j) / a.n_tiles;
        if (g != prev_g) {
          if (prev_g >= 0) mma_commit(a_free);  // the previous query tile is no longer read
          ok = mbar_wait(a_full, (uint32_t)(na & 1), a.status);
          ++na;
          prev_g = g;
          if (!ok) break;
        }
        const int b = (int)(j & 1);
        if (j >= 2 && !(ok = mbar_wait(b ? acc_free1 : acc_free0, (uint32_t)(((j - 2) >> 1) & 1), a.status))) break;
        const uint32_t d = tmem + (uint32_t)(b * kN);
        if (!(ok = wait_sub(0))) break;
        tc_fence_after();
        mma_sub(d, a_hi0, bb[0], true);   // hi_q x lo_v, K half 0
        mma_commit(b_free(bufs[0]));
        if (!(ok = wait_sub(1))) break;
        tc_fence_after();
        mma_sub(d, a_hi1, bb[1], false);  // hi_q x lo_v, K half 1
        mma_commit(b_free(bufs[1]));
        if (!(ok = wait_sub(2))) break;
        tc_fence_after();
        mma_sub(d, a_lo0, bb[2], false);  // lo_q x hi_v, K half 0
        if (!(ok = wait_sub(3))) break;
        tc_fence_after();
        mma_sub(d, a_lo1, bb[3], false);  // lo_q x hi_v, K half 1
        mma_sub(d, a_hi0, bb[2], false);  // hi_q x hi_v, K half 0
        mma_commit(b_free(bufs[2]));
        mma_sub(d, a_hi1, bb[3], false);  // hi_q x hi_v, K half 1
        mma_commit(b_free(bufs[3]));
        mma_commit(b ? acc_full1 : acc_full0);
        nbc += 4;
      }
      // Every MMA this thread issued has completed before the tensor memory
      // is freed, also when a wait above gave up: a commit arrives once all
      // of the thread's earlier MMAs are done, and an MMA completes by itself.
      mma_commit(drain);
      mbar_wait(drain, 0u, a.status);
    }
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. the
    // unit's query rows 32 (w % 4) .. + 31; the kWarpsPerQ warps of a
    // quarter share its eight 32-column blocks (warp `sub` takes blocks
    // sub, sub + kWarpsPerQ, ...).  A block's records are fetched one block
    // ahead (across units); its accumulator columns are loaded while they
    // land.
    const int qd = warp & 3;
    const int sub = (warp - 2) >> 2;
    int *stg_mine = stg_all + (warp - 2) * kStgTiles * kStgInts;  // this warp's staging tiles (swizzled)
    // This warp's two slots of staged records (a block's records
    // 32 kRecPerLane .. + kTailRecs - 1), slot i % 2 for its block i of a unit.
    int2 *tail_mine = reinterpret_cast<int2 *>(stg_all + kEpiWarps * kStgTiles * kStgInts) +
                      (warp - 2) * 2 * kTailRecs;
    int n_blocks = 0;                                              // blocks done (tile n_blocks % kStgTiles next)
    const bool vec = a.vec_ok != 0;
    const bool tma = a.use_tma != 0;
    const bool tail_on = a.use_tail != 0;
    const uint64_t out_policy = evict_first_policy();
    const int sw = lane & 7;
    const int cap = a.bucket_cap;
    // Lanes 0..7: the record counts of the unit's 8 column blocks (0 past
    // the chunk or the queries).
    const int n_tiles = (int)a.n_tiles, n_quarters = (int)a.n_quarters, n_cb = a.n_cb;
    // Units are numbered (g, t): query tile g, item tile t; next(g, t)
    // steps to the following unit without a division.
    auto next_unit = [&](int &g, int &t) {
      if (++t == n_tiles) {
        t = 0;
        ++g;
      }
    };
    auto load_cnt = [&](int g, int t) -> int {
      const int Q = g * 4 + qd;
      const int cb = t * 8 + lane;
      const int v = (Q < n_quarters && lane < 8 && cb < n_cb) ? ld_keep_int(a.rec_n + (int64_t)Q * n_cb + cb) : 0;
      return v > cap ? -1 : v;  // a shared count above the room: the bucket did not fit
    };
    // The bucket of the unit's column block 0 (block c's follows at c * cap).
    auto bucket0 = [&](int g, int t) -> const int2 * {
      const int Q = g * 4 + qd;
      return a.rec + ((int64_t)Q * n_cb + t * 8) * cap;
    };
    // Block c's first 32 kRecPerLane records into dst; the next kTailRecs
    // into shared-memory slot `slot` by asynchronous copies (each lane
    // copies the records it will add), one copy group per call.
    auto fetch = [&](int counts, const int2 *bucket, int c, int2(&dst)[kRecPerLane], int slot) {
      const int n = __shfl_sync(0xffffffffu, counts, c);
      const int2 *bc = bucket + (int64_t)c * cap;
#pragma unroll
      for (int m = 0; m < kRecPerLane; ++m) {
        const int p = 32 * m + lane;
        dst[m] = make_int2(0, 0);  // no record
        if (p < n) dst[m] = ld_keep_int2(bc + p);
      }
      if (tail_on) {
        const uint32_t ts = smem_u32(tail_mine + slot * kTailRecs);
#pragma unroll
        for (int m = 0; m < kTailRecs / 32; ++m) {
          const int q = 32 * m + lane;
          if (32 * kRecPerLane + q < n) cp_async8(ts + 8u * (uint32_t)q, bc + 32 * kRecPerLane + q);
        }
      } else {  // the lines of the rest into L1 instead (16 records a lane)
        const int p = 32 * kRecPerLane + 16 * lane;
        if (p < n) prefetch_l1(bc + p);
      }
      cp_async_commit();
    };
    // The warp's blocks in order: block kMine j + i is column block
    // sub + kWarpsPerQ i of unit j.  Its records sit in register set i % 2;
    // those of the block two later are loaded into the same set once its
    // records are added, so that each load has about two blocks of work to
    // land in.  Record counts are read two units ahead.
    static_assert(kMine >= 2 && kMine % 2 == 0, "two register sets of records");
    const int nv = (int)nj;  // units fit 32 bits (checked at launch)
    int g = (int)(u0 / n_tiles), t = (int)(u0 - (int64_t)g * n_tiles);  // the current unit
    int g1 = g, t1 = t;
    next_unit(g1, t1);  // the next one
    int g2 = g1, t2 = t1;
    next_unit(g2, t2);  // the one after
    int cnt = nv > 0 ? load_cnt(g, t) : 0, cnt_n = nv > 1 ? load_cnt(g1, t1) : 0, cnt_nn = 0;
    int2 R[2][kRecPerLane];
    if (nv > 0) {
      fetch(cnt, bucket0(g, t), sub, R[0], 0);
      fetch(cnt, bucket0(g, t), sub + kWarpsPerQ, R[1], 1);
    }
    for (int j = 0; j < nv; ++j) {
      const int b = j & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(b ? acc_full1 : acc_full0, (uint32_t)((j >> 1) & 1), a.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      if (j + 2 < nv) cnt_nn = load_cnt(g2, t2);
      const int qrow0 = (g * 4 + qd) * 32;
      const int item0 = t * kN;
      const uint32_t tbase = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(b * kN);
#pragma unroll
      for (int i = 0; i < kMine; ++i) {
        const int c = sub + kWarpsPerQ * i;
        int2(&Rc)[kRecPerLane] = R[i & 1];
        int *stg = stg_mine + (kStgTiles > 1 ? (n_blocks % kStgTiles) * kStgInts : 0);
        int *row = stg + lane * 32;
        ++n_blocks;
        uint32_t rc[32];
        tmem_ld32(tbase + (uint32_t)(c * kColBlock), rc);  // lands while the records are added
        const int n = __shfl_sync(0xffffffffu, cnt, c);
        // The records of the block two later, into the set just used.
        auto prefetch = [&]() {
          if (i + 2 < kMine) fetch(cnt, bucket0(g, t), c + 2 * kWarpsPerQ, Rc, i & 1);
          else if (j + 1 < nv) fetch(cnt_n, bucket0(g1, t1), sub + kWarpsPerQ * (i + 2 - kMine), Rc, i & 1);
          else cp_async_commit();  // an empty group keeps one group per block
        };
        if (tma) {  // the bulk store that last read this staging tile is done reading it
          if (lane == 0) {
            if (kStgTiles > 1) bulk_wait_read1();
            else bulk_wait_read0();
          }
          __syncwarp();
        }
        if (n != 0) {
          // The records, summed as integers in the tile (lane = row, chunk
          // k of the row at chunk k ^ (row % 8)), then added to the
          // accumulator with one rounding.
#pragma unroll
          for (int k = 0; k < 8; ++k) *reinterpret_cast<int4 *>(row + 4 * (k ^ sw)) = make_int4(0, 0, 0, 0);
          __syncwarp();
#pragma unroll
          for (int m = 0; m < kRecPerLane; ++m)
            if (Rc[m].y != 0) atomicAdd(stg + Rc[m].x, Rc[m].y);
          if (n > 32 * kRecPerLane) {
            // The staged records (this block's group is complete once at
            // most the next block's group is pending), then any past them.
            int p0 = 32 * kRecPerLane;
            if (tail_on) {
              cp_async_wait1();
              const int2 *ts = tail_mine + (i & 1) * kTailRecs;
              for (int q = lane; q < kTailRecs && 32 * kRecPerLane + q < n; q += 32) {
                const int2 rr = ts[q];
                atomicAdd(stg + rr.x, rr.y);
              }
              p0 += kTailRecs;
            }
            const int2 *bc = bucket0(g, t) + (int64_t)c * cap;
            for (int p = p0 + lane; p < n; p += 32) {  // rare
              const int2 rr = ld_keep_int2(bc + p);
              atomicAdd(stg + rr.x, rr.y);
            }
          }
          prefetch();
          if (n < 0) {
            // The bucket did not fit: each lane walks its item's cold
            // entries through the queries' lists and keeps the rows of this
            // block (rare; exact, the same sums).
            const int it = item0 + c * kColBlock + lane;
            if (it < a.n_items) {
              const int2 rng = __ldg(a.icold_rng + it);
              const float ivi = __ldg(a.inv_i + it);
              const int32_t *qp = a.qptr + (int64_t)qrow0 / a.slice_rows * a.qptr_stride;  // the rows' slice
              for (int e = 0; e < rng.y; ++e) {
                const int2 ie = __ldg(a.icold + rng.x + e);
                const float iv = __int_as_float(ie.y) * ivi;
                const int p1 = __ldg(qp + ie.x + 1);
                for (int p = __ldg(qp + ie.x); p < p1; ++p) {
                  const int2 qe = __ldg(a.qlist + p);
                  const int d = qe.x - (int)qrow0;
                  if ((unsigned)d < 32u) atomicAdd(stg + stg_index(d, lane), cold_fix(__int_as_float(qe.y), iv));
                }
              }
            }
          }
          __syncwarp();
          tmem_wait_ld();
          tmem_regs_ready(rc);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            int *chunk = row + 4 * (k ^ sw);
            const int4 ci = *reinterpret_cast<const int4 *>(chunk);
            float4 o;
            o.x = fmaf((float)ci.x, kFixInv, __uint_as_float(rc[4 * k + 0]));
            o.y = fmaf((float)ci.y, kFixInv, __uint_as_float(rc[4 * k + 1]));
            o.z = fmaf((float)ci.z, kFixInv, __uint_as_float(rc[4 * k + 2]));
            o.w = fmaf((float)ci.w, kFixInv, __uint_as_float(rc[4 * k + 3]));
            *reinterpret_cast<float4 *>(chunk) = o;
          }
        } else {
          prefetch();
          tmem_wait_ld();
          tmem_regs_ready(rc);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4 *>(row + 4 * (k ^ sw)) =
                make_float4(__uint_as_float(rc[4 * k + 0]), __uint_as_float(rc[4 * k + 1]),
                            __uint_as_float(rc[4 * k + 2]), __uint_as_float(rc[4 * k + 3]));
        }
        __syncwarp();
        if (tma) {
          // One bulk tensor store of the tile (its layout is the map's
          // 128-byte swizzle); rows past the queries and columns past the
          // chunk are left out by the map's bounds.
          fence_async_shared();
          __syncwarp();
          if (lane == 0) {
            if (qrow0 < a.n_q && item0 + c * kColBlock < a.n_items)
              tma_store_2d(&a.out_map, smem_u32(stg), item0 + c * kColBlock, (int)qrow0, out_policy);
            bulk_commit();
          }
        } else if (vec && qrow0 + 32 <= a.n_q && item0 + (c + 1) * kColBlock <= a.n_items) {
          // Row-contiguous stores: lane l writes items 4 (l % 8) .. + 3 of
          // rows 4 s + l / 8 (chunk l % 8 of the row, found through the swizzle).
          float *my_row = a.out + ((int64_t)qrow0 + (lane >> 3)) * a.ld_out + item0 + c * kColBlock + 4 * (lane & 7);
#pragma unroll
          for (int sidx = 0; sidx < 8; ++sidx) {
            const int rl = 4 * sidx + (lane >> 3);
            const float4 v = *reinterpret_cast<const float4 *>(stg + rl * 32 + 4 * ((lane & 7) ^ (rl & 7)));
            __stcs(reinterpret_cast<float4 *>(my_row + (int64_t)(4 * sidx) * a.ld_out), v);
          }
        } else {
          const int it = item0 + c * kColBlock + 4 * (lane & 7);
#pragma unroll
          for (int sidx = 0; sidx < 8; ++sidx) {
            const int rl = 4 * sidx + (lane >> 3);
            const float4 v = *reinterpret_cast<const float4 *>(stg + rl * 32 + 4 * ((lane & 7) ^ (rl & 7)));
            const int64_t q = (int64_t)qrow0 + rl;
            if (q < a.n_q && it < a.n_items) {
              float *dst = a.out + q * a.ld_out + it;
              if (vec && it + 4 <= a.n_items) {
                __stcs(reinterpret_cast<float4 *>(dst), v);
              } else {
                const float vv[4] = {v.x, v.y, v.z, v.w};
                for (int e2 = 0; e2 < 4 && it + e2 < a.n_items; ++e2) dst[e2] = vv[e2];
              }
            }
          }
        }
        __syncwarp();
      }
      cnt = cnt_n;
      cnt_n = cnt_nn;
      g = g1;
      t = t1;
      g1 = g2;
      t1 = t2;
      next_unit(g2, t2);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b ? acc_free1 : acc_free0);
    }
    // The bulk stores this warp issued complete before the block exits
    // (also after a wait above gave up: a bulk store completes by itself),
    // and so do its staged-record copies.
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (tma && lane == 0) bulk_wait_all();
    __syncwarp();
  }
  // Tensor-memory reads of every warp are ordered before the release.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// Top-k on the tensor path: offers one row's scores of one 256-item slice
// of a dense score matrix (the chunk's scores, written by the scorer).
__global__ void __launch_bounds__(256)
    k_tc_topk_offer(const float *__restrict__ scores, int64_t n_q, int32_t n_items, ss_topk t,
                    int32_t *status) {
  using namespace topk_dev;
  const int lane = threadIdx.x & 31;
  const int n_sl = (n_items + kN - 1) / kN;
  const int64_t n_jobs = n_q * n_sl;
  for (int64_t jb = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); jb < n_jobs;
       jb += (int64_t)gridDim.x * 8) {
    const int64_t q = jb / n_sl;
    const int sl = (int)(jb % n_sl);
    const float thr = t.best_val[q * t.k + (t.k - 1)];
    float v[8];
    int item[8];
    bool ok[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int it = sl * kN + (j < 4 ? 4 * lane + j : 128 + 4 * lane + (j - 4));
      ok[j] = it < n_items;
      item[j] = it;
      v[j] = ok[j] ? scores[q * n_items + it] : -INFINITY;
    }
    topk_offer(t, q, thr, v, item, ok, lane, status);
  }
}

template <typename T>
cudaError_t grow(T **p, int64_t *cap, int64_t need, cudaStream_t s) {
  if (need <= *cap) return cudaSuccess;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  cudaFree(*p);
  *p = nullptr;
  *cap = 0;
  const int64_t n = std::max<int64_t>(need, *cap + *cap / 2);
  e = dev_alloc(p, sizeof(T) * (size_t)n);
  if (e != cudaSuccess) return e;
  *cap = n;
  return cudaSuccess;
}

// Hot columns rounded up to a multiple of 32: each K half of the query
// operand then holds whole MMA steps of 16.
int padded_hot(int H) { return std::max(32, (H + 31) / 32 * 32); }

}  // namespace

cudaError_t launch_tc_hot_select(ss_handle *h, const ss_csr &items, cudaStream_t s, int *queued) {
  *queued = 0;
  if (h->tc_hot_src[0] == items.indptr && h->tc_hot_src[1] == items.indices &&
      h->tc_hot_src[2] == items.values && h->tc_hot_rows == items.n_rows && h->tc_hot_nnz == items.nnz)
    return cudaSuccess;
  cudaError_t e = cudaSuccess;
  if (!h->tc_hot) {
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
    if ((e = dev_alloc(&h->tc_hot, sizeof(int32_t) * (1 + kHotMax))) != cudaSuccess) return e;
    if ((e = dev_alloc(&h->tc_sel, sizeof(int32_t) * 2 * kSelSlots)) != cudaSuccess) return e;
    if ((e = dev_alloc(&h->tc_stats, sizeof(float) * 2)) != cudaSuccess) return e;
  }
  const int64_t n = items.n_rows;
  int64_t n_sample = 0;
  if (n > 0 && items.nnz > 0) {
    n_sample = (int64_t)((double)kSampleEntries * (double)n / (double)items.nnz);
    n_sample = std::max<int64_t>(16, std::min<int64_t>(n, n_sample));
  }
  float stats[2] = {0.f, 0.f};
  if (n_sample == 0) {
    if ((e = cudaMemsetAsync(h->tc_hot, 0, sizeof(int32_t), s)) != cudaSuccess) return e;
  } else {
    if ((e = cudaMemsetAsync(h->tc_sel, 0xFF, sizeof(int32_t) * kSelSlots, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(h->tc_sel + kSelSlots, 0, sizeof(int32_t) * kSelSlots, s)) != cudaSuccess)
      return e;
    const int sms = h->sm_count > 0 ? h->sm_count : 148;
    k_tc_sel_insert<<<sms * 2, 256, 0, s>>>(items.indptr, items.indices, n, n_sample, h->tc_sel);
    k_tc_sel_pick<<<1, kSelThreads, 0, s>>>(h->tc_sel, n_sample, h->tc_hot, h->tc_stats);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    *queued = 2;
    if ((e = cudaMemcpyAsync(stats, h->tc_stats, sizeof(stats), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
      return e;
  }
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  h->tc_est_cold = stats[0];
  h->tc_H = (int32_t)stats[1];
  h->tc_hot_src[0] = items.indptr;
  h->tc_hot_src[1] = items.indices;
  h->tc_hot_src[2] = items.values;
  h->tc_hot_rows = items.n_rows;
  h->tc_hot_nnz = items.nnz;
  ++h->tc_hot_generation;
  return cudaSuccess;
}

cudaError_t launch_build_tc(ss_handle *h, const ss_csr &items, int64_t row_begin, int64_t row_end,
                            cudaStream_t s, int *queued) {
  *queued = 0;
  const int64_t C = h->chunk_rows;
  const int n_chunks = (int)((row_end - row_begin + C - 1) / C);
  h->n_views = 0;
  if (n_chunks < 1 || n_chunks > h->build_batch) return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  if (!h->tc_slab) {  // the three exist together or not at all (reset_after_oom)
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
    const size_t rows = (size_t)h->build_batch * C;
    if ((e = dev_alloc(&h->tc_slab, sizeof(float) * rows * kHotMax)) != cudaSuccess) return e;
    if ((e = dev_alloc(&h->tc_sq, sizeof(float) * rows)) != cudaSuccess) return e;
    if ((e = dev_alloc(&h->tc_icold_rng, sizeof(int2) * rows)) != cudaSuccess) return e;
  }
  const int grid = (h->sm_count > 0 ? h->sm_count : 148) * 8;
  // The build's cold entries go to the entry array sized for the matrix
  // (post_hat, post_cap >= items.nnz), at the rows' own positions.
  k_tc_build<<<grid, 256, 0, s>>>(items.indptr, items.indices, items.values, row_begin, row_end, C, h->dim,
                                  h->tc_hot, h->tc_slab, h->tc_sq, h->post_hat, h->tc_icold_rng, h->d_status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  *queued = 1;
  for (int k = 0; k < n_chunks; ++k) {
    ss_index &ix = h->views[k];
    ix = ss_index();
    ix.algo = ALGO_TENSOR;
    ix.row_begin = row_begin + (int64_t)k * C;
    ix.row_end = std::min<int64_t>(ix.row_begin + C, row_end);
    ix.n_items = (int32_t)(ix.row_end - ix.row_begin);
    ix.dim = h->dim;
    ix.capacity = h->post_cap;
    ix.hot = h->tc_hot;
    ix.slab = h->tc_slab + (size_t)k * C * kHotMax;
    ix.slab_ld = kHotMax;
    ix.sq = h->tc_sq + (size_t)k * C;
    ix.icold = h->post_hat;
    ix.icold_rng = h->tc_icold_rng + (size_t)k * C;
  }
  h->n_views = n_chunks;
  return cudaSuccess;
}

// The driver's tensor-map encoder, looked up once (null when unavailable).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
  });
  return fn;
}

// A tensor map of the output tile (n_q rows x n_items floats, row stride
// ld floats) in boxes of 32 x 32 with the 128-byte swizzle of the scorer's
// staging tiles.  Only for device memory (not page-locked host memory
// mapped into the device); false when the map cannot be made, and the
// scorer then stores with plain instructions.
static bool encode_out_map(CUtensorMap *map, float *out, int64_t n_q, int64_t n_items, int64_t ld) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode || n_q <= 0 || n_items <= 0 || (reinterpret_cast<uintptr_t>(out) & 15) != 0 || (ld & 3) != 0)
    return false;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, out) != cudaSuccess || attr.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    return false;
  }
  const cuuint64_t dims[2] = {(cuuint64_t)n_items, (cuuint64_t)n_q};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t elem[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, out, dims, strides, box, elem,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_score_tc(ss_handle *h, const ss_csr &q, const float *inv_q, const ss_index &idx,
                            const float *inv_i, float *out, int64_t ld_out, cudaStream_t s,
                            int *queued, const ss_topk *topk) {
  *queued = 0;
  if (q.n_rows == 0 || idx.n_items == 0) return cudaSuccess;
  const int sms = h->sm_count > 0 ? h->sm_count : 148;
  const int Hp = padded_hot(h->tc_H);
  const int64_t n_q = q.n_rows;
  const int64_t n_qtiles = (n_q + kM - 1) / kM;
  const int32_t n_items = idx.n_items;
  const int64_t n_tiles = (n_items + kN - 1) / kN;
  const int64_t dim = idx.dim;
  cudaError_t e = cudaSuccess;
  int nq = 0;

  // Query operand, cold entries and the queries' lists, once per query
  // matrix, inverse norms and hot set.
  if (!(h->tcq_src[0] == q.indptr && h->tcq_src[1] == q.indices && h->tcq_src[2] == q.values &&
        h->tcq_src[3] == inv_q && h->tcq_rows == q.n_rows && h->tcq_nnz == q.nnz &&
        h->tcq_generation == h->tc_hot_generation)) {
    h->tcq_rows = -1;  // not prepared until the end of this block
    // Slices of whole query tiles whose records in one chunk (the sample's
    // estimate) take about kRecSliceBytes: one records launch each.
    const double quarter_bytes =
        8.0 * std::max(1e-3, h->tc_est_cold) * 1024.0 * (double)((h->chunk_rows + kColBlock - 1) / kColBlock);
    const int64_t tiles_per_slice = std::max<int64_t>(1, (int64_t)((double)kRecSliceBytes / quarter_bytes) / (kM / 32));
    const int64_t slice_rows = std::min<int64_t>(n_qtiles, tiles_per_slice) * kM;
    const int64_t n_slices = (n_q + slice_rows - 1) / slice_rows;
    const int64_t n_cnt = n_slices * (dim + 1);
    if ((e = grow(&h->tc_A, &h->tc_A_cap, n_qtiles * kM * 2 * Hp, s)) != cudaSuccess) return e;
    if ((e = grow(&h->tc_qcold, &h->tc_qcold_cap, std::max<int64_t>(1, q.nnz), s)) != cudaSuccess) return e;
    if ((e = grow(&h->tc_qcold_n, &h->tc_qcold_n_cap, n_q, s)) != cudaSuccess) return e;
    if ((e = grow(&h->tc_qcnt, &h->tc_qcnt_cap, n_cnt, s)) != cudaSuccess) return e;
    if ((e = grow(&h->tc_qptr, &h->tc_qptr_cap, n_cnt, s)) != cudaSuccess) return e;
    if ((e = grow(&h->tc_qpart, &h->tc_qpart_cap, scan_tile_count(n_cnt) + 1, s)) != cudaSuccess) return e;
    if ((e = grow(&h->tc_qlist, &h->tc_qlist_cap, std::max<int64_t>(1, q.nnz), s)) != cudaSuccess) return e;
    PrepArgs pa;
    pa.indptr = q.indptr;
    pa.idx = q.indices;
    pa.val = q.values;
    pa.slab = nullptr;
    pa.sq = nullptr;
    pa.n_rows = n_q;
    pa.n_groups = n_qtiles * (kM / 8);
    pa.inv = inv_q;
    pa.hot = idx.hot;
    pa.Hp = Hp;
    pa.gpt = kM / 8;
    pa.op = h->tc_A;
    pa.qcold = h->tc_qcold;
    pa.qcold_n = h->tc_qcold_n;
    pa.dim = dim;
    pa.status = h->d_status;
    const int64_t blocks = std::min<int64_t>((pa.n_groups + 7) / 8, (int64_t)sms * 8);
    k_tc_prep_queries<<<(unsigned)blocks, kPrepThreads, 0, s>>>(pa);
    if ((e = cudaMemsetAsync(h->tc_qcnt, 0, sizeof(int32_t) * (size_t)n_cnt, s)) != cudaSuccess) return e;
    const int64_t row_blocks = std::min<int64_t>((n_q + 7) / 8, (int64_t)sms * 8);
    k_tc_qcount<<<(unsigned)row_blocks, 256, 0, s>>>(q.indptr, h->tc_qcold, h->tc_qcold_n, n_q, slice_rows, dim + 1,
                                                     h->tc_qcnt);
    if ((e = launch_count_scan(h->tc_qcnt, n_cnt, h->tc_qpart, h->tc_qptr, s)) != cudaSuccess) return e;
    k_tc_qscatter<<<(unsigned)row_blocks, 256, 0, s>>>(q.indptr, h->tc_qcold, h->tc_qcold_n, n_q, slice_rows,
                                                       dim + 1, h->tc_qcnt, h->tc_qlist);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    nq += 6;
    h->tcq_src[0] = q.indptr;
    h->tcq_src[1] = q.indices;
    h->tcq_src[2] = q.values;
    h->tcq_src[3] = inv_q;
    h->tcq_rows = q.n_rows;
    h->tcq_nnz = q.nnz;
    h->tcq_generation = h->tc_hot_generation;
    h->tcq_slice_rows = slice_rows;
    h->tcq_slices = n_slices;
  }
  const int64_t slice_rows = h->tcq_slice_rows, n_slices = h->tcq_slices;

  // Item operand of this chunk (written by the records launch's trailing
  // blocks).
  if ((e = grow(&h->tc_B, &h->tc_B_cap, n_tiles * kN * 2 * Hp, s)) != cudaSuccess) return e;
  PrepArgs pa;
  {
    pa.indptr = nullptr;
    pa.idx = nullptr;
    pa.val = nullptr;
    pa.slab = idx.slab;
    pa.sq = idx.sq;
    pa.n_rows = n_items;
    pa.n_groups = n_tiles * (kN / 8);
    pa.inv = inv_i;
    pa.hot = idx.hot;
    pa.Hp = Hp;
    pa.gpt = kN / 8;
    pa.op = h->tc_B;
    pa.qcold = nullptr;
    pa.qcold_n = nullptr;
    pa.dim = dim;
    pa.status = h->d_status;
  }

  // Cold records: a bucket per (32 query rows, 32 items) holding three
  // times the sample's estimate of its records plus 64 (at least 64, at
  // most 1024); the scorer computes the blocks of fuller buckets from the
  // lists.
  const int64_t n_quarters = (n_q + 31) / 32;
  const int32_t n_cb = (n_items + kColBlock - 1) / kColBlock;
  const double est = std::max(0.0, h->tc_est_cold);
  const int32_t cap = (int32_t)std::min<double>(
      1024.0, std::max<double>(64.0, std::ceil((3.0 * est * 1024.0 + 64.0) / 32.0) * 32.0));
  if ((e = grow(&h->tc_rec_n, &h->tc_rec_n_cap, n_quarters * n_cb, s)) != cudaSuccess) return e;
  if ((e = grow(&h->tc_rec, &h->tc_rec_cap, n_quarters * n_cb * (int64_t)cap, s)) != cudaSuccess) return e;
  // One records launch per slice of query rows; the first also writes the
  // item operand (its trailing blocks).
  for (int64_t sl = 0; sl < n_slices; ++sl) {
    const int64_t q_lo = sl * slice_rows, q_hi = std::min<int64_t>(n_q, q_lo + slice_rows);
    const int64_t q0 = q_lo / 32, nqs = (q_hi + 31) / 32 - q0;  // the slice's quarters
    RecArgs ra;
    ra.icold = idx.icold;
    ra.icold_rng = idx.icold_rng;
    ra.n_items = n_items;
    ra.inv_i = inv_i;
    ra.qptr = h->tc_qptr + sl * (dim + 1);
    ra.qlist = h->tc_qlist;
    ra.q0 = q0;
    ra.n_quarters = nqs;
    ra.n_cb = n_cb;
    ra.bucket_cap = cap;
    ra.rec = h->tc_rec;
    ra.rec_n = h->tc_rec_n;
    ra.status = h->d_status;
    ra.prep = pa;
    // A main block counts its buckets in shared memory (one counter per
    // quarter); past kRecMaxQuarters every item goes the shared way.
    const bool own = nqs <= kRecMaxQuarters;
    const size_t smem = own ? sizeof(int) * (size_t)nqs : 0;
    if ((e = ensure_dyn_smem(k_tc_records, smem)) != cudaSuccess) return e;
    // Whole waves of column blocks, then one wave sharing the rest.
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_tc_records, kRThreads, smem) != cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    const int64_t wave = (int64_t)sms * per_sm;
    // A chunk of at most one wave of column blocks that still gives every
    // SM one runs as main blocks only; a smaller one is shared out.
    ra.n_main = !own ? 0 : (n_cb <= wave && 2 * n_cb >= wave) ? n_cb : n_cb / wave * wave;
    ra.n_shared = ra.n_main < n_cb ? wave : 0;
    // An item's walk is cut into parts of about 32 windows of 32 records
    // (the sample's estimate of its records in the slice: est x rows), at
    // most 8.
    ra.pieces = (int32_t)std::max<double>(1.0, std::min<double>(8.0, std::floor(est * (double)(q_hi - q_lo) / 1024.0)));
    // The shared column blocks' counters: [n_main, n_cb) of the slice's quarters.
    if (ra.n_shared > 0 &&
        (e = cudaMemset2DAsync(h->tc_rec_n + q0 * n_cb + ra.n_main, sizeof(int32_t) * (size_t)n_cb, 0,
                               sizeof(int32_t) * (size_t)(n_cb - ra.n_main), (size_t)nqs, s)) != cudaSuccess)
      return e;
    // The operand's blocks (a warp per group of 8 items) come last.
    const int64_t prep_blocks = sl == 0 ? (pa.n_groups + kRThreads / 32 - 1) / (kRThreads / 32) : 0;
    k_tc_records<<<(unsigned)(ra.n_main + ra.n_shared + prep_blocks), kRThreads, smem, s>>>(ra);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++nq;
  }

  // Scores (full chunk, or the dense scratch the top-k offers read).
  float *dst = out;
  int64_t ld_dst = ld_out;
  if (topk && topk->k > 0) {
    if ((e = grow(&h->hot_scratch, &h->hot_scratch_cap, n_q * (int64_t)n_items, s)) != cudaSuccess) return e;
    dst = h->hot_scratch;
    ld_dst = n_items;
  }
  {
    if ((e = ensure_dyn_smem(k_tc_score, std::max(score_smem_bytes(kHotMax, false), score_smem_bytes(128, true)))) !=
        cudaSuccess)
      return e;
    ScoreArgs sa;
    sa.A = h->tc_A;
    sa.B = h->tc_B;
    sa.rec = h->tc_rec;
    sa.rec_n = h->tc_rec_n;
    sa.bucket_cap = cap;
    sa.icold = idx.icold;
    sa.icold_rng = idx.icold_rng;
    sa.qptr = h->tc_qptr;
    sa.qptr_stride = dim + 1;
    sa.slice_rows = slice_rows;
    sa.qlist = h->tc_qlist;
    sa.inv_i = inv_i;
    sa.n_quarters = n_quarters;
    sa.n_cb = n_cb;
    sa.out = dst;
    sa.ld_out = ld_dst;
    sa.n_q = n_q;
    sa.n_items = n_items;
    sa.n_qtiles = n_qtiles;
    sa.n_tiles = n_tiles;
    sa.n_units = n_tiles * n_qtiles;
    sa.Hp = Hp;
    sa.vec_ok = ((reinterpret_cast<uintptr_t>(dst) % 16) == 0) && (ld_dst % 4 == 0);
    sa.use_tma = sa.vec_ok && encode_out_map(&sa.out_map, dst, n_q, n_items, ld_dst) ? 1 : 0;
    sa.use_tail = score_tail_fits(Hp) ? 1 : 0;
    sa.status = h->d_status;
    if (sa.n_units > INT32_MAX || n_q > INT32_MAX - 256) return cudaErrorInvalidValue;  // 32-bit unit and row numbers
    const int64_t grid = std::min<int64_t>(sms, sa.n_units);
    prof_mark(h, s);
    k_tc_score<<<(unsigned)grid, kSThreads, score_smem_bytes(Hp, sa.use_tail != 0), s>>>(sa);
    prof_mark(h, s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++nq;
  }
  if (topk && topk->k > 0) {
    const int64_t jobs = n_q * n_tiles;
    const int64_t blocks = std::min<int64_t>((jobs + 7) / 8, (int64_t)sms * 16);
    k_tc_topk_offer<<<(unsigned)blocks, 256, 0, s>>>(dst, n_q, n_items, *topk, h->d_status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++nq;
  }
  *queued = nq;
  return cudaSuccess;
}
