// Posting-list scorer: for each query row, walk the chunk's posting lists of
// the row's dimensions and add every product into a per-item accumulator.
//
// Blog post "Engineering practice for bulk similarity calculation over sparse
// embeddings": section 3.1 (u.v summed over the dimensions both supports
// hold; the posting list of dimension k names the items whose support holds
// k) and section 4.4 (normalise by the two norms).  This path suits item
// matrices whose rows are long or evenly spread over the dimensions (every
// item tile of the hybrid path would overflow its shared-memory image).
//
// Exact, order-free accumulation.  The products are formed from normalised
// values, p = (q_k * inv_q) * (v_ik * inv_i), so every |p| <= 1 and the sum
// over k of |p| is at most 1 (Cauchy-Schwarz).  Each p is rounded once to a
// fixed-point number of resolution 2^-38, held as two int32 parts:
//   x  = p * 2^21                     (|x| <= 2^21 + a rounding or two)
//   hi = round(x)                     (exact: magic-number rounding)
//   lo = round((x - hi) * 2^17)       (x - hi is exact, |lo| <= 2^16)
//   p ~ (hi * 2^17 + lo) * 2^-38      (error <= 2^-39)
// and the two parts are added with 32-bit shared-memory atomics.  Integer
// sums do not depend on their order, so any lane or warp may add any
// product: the result is the same bits on every run, for every chunking and
// every launch shape.  The lo sums are folded into hi before n * 2^16 could
// reach 2^31 (every kFoldDims query dimensions).  The store converts the
// int64 total to float once.  Error per score: float rounding of the three
// products (<= ~4 * 2^-24 in all, against the sum of |p| <= 1), plus 2^-39
// per shared dimension, plus the final rounding.
//
// Block shape: kCons consumer warps and one producer warp.  The producer takes
// query rows from a global counter, and for each segment of up to kSeg of a
// row's dimensions looks up each dimension's list (start, length) in the
// chunk's column pointers, drops empty lists, and writes the segment's lists
// with their inclusive length prefix into one of two shared buffers.  The
// consumers split the segment's entries evenly (each warp a contiguous
// range, 32 entries per round, a 32-wide window search to find each entry's
// list) and add the products; at the end of a row they convert, store (or
// offer top-k candidates) and zero the accumulator.  Named barriers hand the
// buffers back and forth, so the producer's global-memory latency overlaps
// the consumers' walk.
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "internal.cuh"
#include "topk.cuh"

namespace {

using namespace topk_dev;

constexpr int kCons = 12;                    // consumer warps
constexpr int kPThreads = (kCons + 1) * 32;  // + one producer warp
constexpr int kSeg = 128;                    // query dimensions per segment
constexpr int kBlocksPerSm = 3;              // 3 x (64 KB accumulator + lists) fit in shared memory
constexpr int kPerLane = kSeg / 32;
constexpr int kWindowMax = 8192;             // items per accumulator window
constexpr int kRoundsPerStep = 2;            // 32-entry rounds whose loads are issued together
constexpr int kFoldDims = 16384;             // lo sums stay below 2^31
constexpr float kXScale = 2097152.0f;        // 2^21
constexpr float kLoScale = 131072.0f;        // 2^17
constexpr float kMagic = 12582912.0f;        // 1.5 * 2^23: adding it rounds |x| <= 2^22 to an integer
constexpr int32_t kMagicBits = 0x4B400000;
constexpr float kXMax = 4194304.0f;          // 2^22: clamp (far above any valid |x|)
constexpr float kXValid = 2099200.0f;        // 2^21 * (1 + 2^-11): larger means unnormalised input
constexpr float kOutScale = 0x1p-38f;

// Named barriers (0 is __syncthreads, unused in the loop).
constexpr int kBarFull = 1;   // + buffer: the producer filled it
constexpr int kBarEmpty = 3;  // + buffer: the consumers are done with it
constexpr int kBarCons = 5;   // the consumer warps

// Job header flags.
constexpr int kJobFirst = 1;  // first segment of a (row, window)
constexpr int kJobLast = 2;   // last segment: store after it
constexpr int kJobDone = 4;   // no more rows
constexpr int kJobFold = 8;   // fold lo into hi before this segment

struct Job {
  int64_t row;
  int32_t window;  // first item of the accumulator window
  int32_t n_lists;
  int32_t n_entries;
  int32_t flags;
};

struct PostArgs {
  const int64_t *q_indptr;
  const int32_t *q_idx;
  const float *q_val;
  int64_t n_q;
  const float *inv_q;
  const int32_t *col_ptr;  // [dim + 1] of this chunk (absolute positions)
  const int2 *post_hat;    // {item in chunk, normalised value bits} at those positions
  int32_t capacity;        // entries the lists may address (longer lists are cut here)
  int32_t dim;
  int32_t n_items;
  int32_t window;          // accumulator width (multiple of 256, <= kWindowMax)
  float *out;
  int64_t ld_out;
  int32_t vec_ok;
  ss_topk topk;
  int32_t *row_next;       // [0] next row, [1] blocks finished (the last one resets both)
  int32_t *status;
};

__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

// Inclusive warp scan.
__device__ __forceinline__ int warp_incl(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Producer: one segment of row q's dimensions [s0, s1) for the window
// starting at w0, loaded into registers (list start, length, scaled value).
struct SegRegs {
  int32_t start[kPerLane];
  int32_t len[kPerLane];
  float qv[kPerLane];
};

__device__ __forceinline__ void load_segment(const PostArgs &a, int64_t s0, int64_t s1, float iq,
                                             int lane, SegRegs &r) {
  int32_t k[kPerLane];
  float v[kPerLane];
#pragma unroll
  for (int m = 0; m < kPerLane; ++m) {
    const int64_t j = s0 + lane + 32 * m;
    k[m] = -1;
    v[m] = 0.f;
    if (j < s1) {
      k[m] = __ldg(a.q_idx + j);
      v[m] = __ldg(a.q_val + j);
    }
  }
#pragma unroll
  for (int m = 0; m < kPerLane; ++m) {
    r.start[m] = 0;
    r.len[m] = 0;
    r.qv[m] = (v[m] * iq) * kXScale;  // normalise first: iq * 2^21 alone may overflow
    if ((uint32_t)k[m] < (uint32_t)a.dim) {
      r.start[m] = __ldg(a.col_ptr + k[m]);
      r.len[m] = max(0, min(__ldg(a.col_ptr + k[m] + 1), a.capacity) - r.start[m]);
    }
  }
}

// Compacts the segment's non-empty lists into lists[]: {inclusive entry
// prefix, start - exclusive prefix, value bits, 0}.  Returns the counts.
__device__ __forceinline__ int2 write_segment(const SegRegs &r, int4 *lists, int lane) {
  int n_lists = 0, n_entries = 0;
  const unsigned below = (1u << lane) - 1u;
#pragma unroll
  for (int m = 0; m < kPerLane; ++m) {
    const bool has = r.len[m] > 0;
    const unsigned mask = __ballot_sync(0xffffffffu, has);
    const int incl = warp_incl(r.len[m], lane) + n_entries;
    if (has) {
      const int pos = n_lists + __popc(mask & below);
      lists[pos] = make_int4(incl, r.start[m] - (incl - r.len[m]), __float_as_int(r.qv[m]), 0);
    }
    n_lists += __popc(mask);
    n_entries = __shfl_sync(0xffffffffu, incl, 31);
  }
  return make_int2(n_lists, n_entries);
}

__device__ __forceinline__ void producer(const PostArgs &a, int4 *lists, Job *jobs) {
  const int lane = threadIdx.x & 31;
  const int n_windows = (a.n_items + a.window - 1) / a.window;
  int n_job = 0;
  for (;;) {
    int64_t q = 0;
    if (lane == 0) q = atomicAdd(a.row_next, 1);
    q = __shfl_sync(0xffffffffu, q, 0);
    const bool done = q >= a.n_q;
    int64_t jb = 0, je = 0;
    float iq = 0.f;
    if (!done) {
      jb = __ldg(a.q_indptr + q);
      je = __ldg(a.q_indptr + q + 1);
      iq = __ldg(a.inv_q + q);
    }
    for (int w = 0; w < (done ? 1 : n_windows); ++w) {
      int64_t s0 = jb;
      int since_fold = 0;
      do {  // at least one job per (row, window), even for an empty row
        const int64_t s1 = s0 + kSeg < je ? s0 + kSeg : je;
        SegRegs r;
        if (!done) {
          load_segment(a, s0, s1, iq, lane, r);
        } else {
#pragma unroll
          for (int m = 0; m < kPerLane; ++m) r.len[m] = 0;
        }
        const int b = n_job & 1;
        if (n_job >= 2) bar_sync(kBarEmpty + b, kPThreads);  // job n_job - 2 released buffer b
        const int2 cnt = write_segment(r, lists + b * kSeg, lane);
        if (lane == 0) {
          Job &j = jobs[b];
          j.row = q;
          j.window = w * a.window;
          j.n_lists = cnt.x;
          j.n_entries = cnt.y;
          int f = 0;
          if (s0 == jb) f |= kJobFirst;
          if (s1 >= je) f |= kJobLast;
          if (done) f |= kJobDone;
          if (since_fold >= kFoldDims) f |= kJobFold;
          j.flags = f;
        }
        if (since_fold >= kFoldDims) since_fold = 0;
        since_fold += kSeg;
        __syncwarp();
        bar_arrive(kBarFull + b, kPThreads);
        ++n_job;
        s0 = s1;
      } while (!done && s0 < je);
    }
    if (done) break;
  }
  // The consumers released every job but the last (the done job, which they
  // do not release) and possibly the one before it: match those arrivals.
  if (n_job >= 2) bar_sync(kBarEmpty + (n_job & 1), kPThreads);
  if (lane == 0) {
    __threadfence();
    if (atomicAdd(a.row_next + 1, 1) == (int)gridDim.x - 1) {
      a.row_next[0] = 0;
      a.row_next[1] = 0;
      __threadfence();
    }
  }
}

// Adds one entry's product to the accumulator.
__device__ __forceinline__ void add_product(int32_t *acc_hi, int32_t *acc_lo, int it, float x,
                                            bool &bad) {
  bad |= fabsf(x) > kXValid;
  x = fminf(fmaxf(x, -kXMax), kXMax);
  const float y = x + kMagic;
  const int32_t hi = __float_as_int(y) - kMagicBits;
  const float rem = x - (y - kMagic);
  const int32_t lo = __float_as_int(fmaf(rem, kLoScale, kMagic)) - kMagicBits;
  atomicAdd(acc_hi + it, hi);
  atomicAdd(acc_lo + it, lo);
}

// One consumer warp's share [e0, e1) of a segment's entries.
__device__ __forceinline__ void walk(const PostArgs &a, const int4 *lists, int n_lists, int e0,
                                     int e1, int w0, int32_t *acc_hi, int32_t *acc_lo, int lane,
                                     bool &bad) {
  if (e0 >= e1) return;
  // First list whose inclusive prefix exceeds e0.
  int lo = 0, hi = n_lists - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (lists[mid].x > e0) hi = mid;
    else lo = mid + 1;
  }
  int jc = lo;
  const unsigned W = (unsigned)a.window;
  for (int base = e0; base < e1; base += 32 * kRoundsPerStep) {
    int2 ent[kRoundsPerStep];
    float qv[kRoundsPerStep];
    bool live[kRoundsPerStep];
#pragma unroll
    for (int u = 0; u < kRoundsPerStep; ++u) {
      const int rb = base + 32 * u;
      const int cand = jc + lane;
      const int4 c = cand < n_lists ? lists[cand] : make_int4(INT_MAX, 0, 0, 0);
      const int e = rb + lane;
      // Entry e lies in list jc + pos, pos = candidates whose prefix <= e.
      int pos = 0;
#pragma unroll
      for (int step = 16; step > 0; step >>= 1) {
        const int pv = __shfl_sync(0xffffffffu, c.x, pos + step - 1);
        if (pv <= e) pos += step;
      }
      const int bj = __shfl_sync(0xffffffffu, c.y, pos);
      qv[u] = __int_as_float(__shfl_sync(0xffffffffu, c.z, pos));
      live[u] = e < e1;
      ent[u] = live[u] ? __ldg(a.post_hat + (bj + e)) : make_int2(0, 0);
      jc += __popc(__ballot_sync(0xffffffffu, c.x <= rb + 32));
    }
#pragma unroll
    for (int u = 0; u < kRoundsPerStep; ++u) {
      const unsigned it = (unsigned)(ent[u].x - w0);
      if (live[u] && it < W) add_product(acc_hi, acc_lo, (int)it, qv[u] * __int_as_float(ent[u].y), bad);
    }
  }
}

// Converts the window's accumulators of row q to scores, stores them (or
// offers them to the row's top-k), and zeroes the accumulators.
__device__ __forceinline__ void store_window(const PostArgs &a, int64_t q, int w0, int32_t *acc_hi,
                                             int32_t *acc_lo, int ctid) {
  const int width = min(a.window, a.n_items - w0);
  if (a.topk.k > 0) {
    const int lane = ctid & 31, warp = ctid >> 5;
    const float thr = __ldg(a.topk.best_val + q * a.topk.k + (a.topk.k - 1));
    for (int s = warp * 256; s < a.window; s += kCons * 256) {
      const int ia = s + 4 * lane, ib = s + 128 + 4 * lane;
      const int4 ha = *reinterpret_cast<const int4 *>(acc_hi + ia);
      const int4 la = *reinterpret_cast<const int4 *>(acc_lo + ia);
      const int4 hb = *reinterpret_cast<const int4 *>(acc_hi + ib);
      const int4 lb = *reinterpret_cast<const int4 *>(acc_lo + ib);
      const int4 z = make_int4(0, 0, 0, 0);
      *reinterpret_cast<int4 *>(acc_hi + ia) = z;
      *reinterpret_cast<int4 *>(acc_lo + ia) = z;
      *reinterpret_cast<int4 *>(acc_hi + ib) = z;
      *reinterpret_cast<int4 *>(acc_lo + ib) = z;
      if (s >= width) continue;  // warp-uniform
      const int hv[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
      const int lv[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
      float v[8];
      int it[8];
      bool ok[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = __ll2float_rn((long long)hv[j] * 131072LL + lv[j]) * kOutScale;
        const int c = (j < 4 ? ia : ib) + (j & 3);
        it[j] = w0 + c;
        ok[j] = c < width;
      }
      topk_offer(a.topk, q, thr, v, it, ok, lane, a.status);
    }
    return;
  }
  float *orow = a.out + q * a.ld_out + w0;
  for (int c = ctid * 4; c < a.window; c += kCons * 32 * 4) {
    const int4 h4 = *reinterpret_cast<const int4 *>(acc_hi + c);
    const int4 l4 = *reinterpret_cast<const int4 *>(acc_lo + c);
    *reinterpret_cast<int4 *>(acc_hi + c) = make_int4(0, 0, 0, 0);
    *reinterpret_cast<int4 *>(acc_lo + c) = make_int4(0, 0, 0, 0);
    if (c >= width) continue;
    const float o[4] = {__ll2float_rn((long long)h4.x * 131072LL + l4.x) * kOutScale,
                        __ll2float_rn((long long)h4.y * 131072LL + l4.y) * kOutScale,
                        __ll2float_rn((long long)h4.z * 131072LL + l4.z) * kOutScale,
                        __ll2float_rn((long long)h4.w * 131072LL + l4.w) * kOutScale};
    if (a.vec_ok && c + 4 <= width) {
      __stcs(reinterpret_cast<float4 *>(orow + c), make_float4(o[0], o[1], o[2], o[3]));
    } else {
      for (int j = 0; j < 4 && c + j < width; ++j) orow[c + j] = o[j];
    }
  }
}

__global__ void __launch_bounds__(kPThreads, kBlocksPerSm) k_score_lists(const PostArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  int32_t *acc_hi = reinterpret_cast<int32_t *>(smem);
  int32_t *acc_lo = acc_hi + a.window;
  int4 *lists = reinterpret_cast<int4 *>(acc_lo + a.window);  // [2][kSeg]
  Job *jobs = reinterpret_cast<Job *>(lists + 2 * kSeg);       // [2]

  for (int c = threadIdx.x * 4; c < 2 * a.window; c += kPThreads * 4)
    *reinterpret_cast<int4 *>(acc_hi + c) = make_int4(0, 0, 0, 0);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kCons) {
    producer(a, lists, jobs);
    return;
  }
  bool bad = false;
  for (int n_job = 0;; ++n_job) {
    const int b = n_job & 1;
    bar_sync(kBarFull + b, kPThreads);
    const Job j = jobs[b];
    if (j.flags & kJobDone) break;
    if (j.flags & kJobFold) {
      // Every warp has added the earlier segments once all reach here.
      bar_sync(kBarCons, kCons * 32);
      for (int c = threadIdx.x; c < a.window; c += kCons * 32) {
        const int32_t carry = acc_lo[c] >> 17;
        acc_hi[c] += carry;
        acc_lo[c] -= carry * (1 << 17);
      }
      bar_sync(kBarCons, kCons * 32);
    }
    const int e0 = (int)((int64_t)j.n_entries * warp / kCons);
    const int e1 = (int)((int64_t)j.n_entries * (warp + 1) / kCons);
    walk(a, lists + b * kSeg, j.n_lists, e0, e1, j.window, acc_hi, acc_lo, lane, bad);
    __syncwarp();
    bar_arrive(kBarEmpty + b, kPThreads);
    if (j.flags & kJobLast) {
      bar_sync(kBarCons, kCons * 32);
      store_window(a, j.row, j.window, acc_hi, acc_lo, threadIdx.x);
      bar_sync(kBarCons, kCons * 32);
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(a.status, DEV_RANGE);
}

// Normalised copy of a chunk's posting entries: {item, value * inv_i[item]}.
__global__ void __launch_bounds__(256)
    k_post_normalize(const int32_t *__restrict__ col_ptr, int32_t dim, int32_t capacity,
                     const uint16_t *__restrict__ post_item, const float *__restrict__ post_val,
                     const float *__restrict__ inv_i, int2 *__restrict__ post_hat) {
  const int32_t p0 = __ldg(col_ptr), p1 = min(__ldg(col_ptr + dim), capacity);
  for (int64_t p = p0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < p1;
       p += (int64_t)gridDim.x * blockDim.x) {
    const int it = post_item[p];
    post_hat[p] = make_int2(it, __float_as_int(post_val[p] * __ldg(inv_i + it)));
  }
}

}  // namespace

int32_t posting_window(int32_t n_items) {
  const int32_t w = (std::max<int32_t>(n_items, 1) + 255) / 256 * 256;
  return std::min<int32_t>(w, kWindowMax);
}

size_t posting_smem_bytes(int32_t window) {
  return sizeof(int32_t) * 2 * (size_t)window + sizeof(int4) * 2 * kSeg + sizeof(Job) * 2;
}

cudaError_t launch_score_lists(ss_handle *h, const ss_csr &queries, const float *inv_q,
                               const ss_index &idx, const float *inv_i, float *out, int64_t ld_out,
                               cudaStream_t s, int *queued, const ss_topk *topk) {
  *queued = 0;
  if (queries.n_rows == 0 || idx.n_items == 0) return cudaSuccess;
  if (queries.n_rows >= INT32_MAX - 65536) return cudaErrorInvalidValue;
  const int sms = h->sm_count > 0 ? h->sm_count : 148;
  const int32_t capacity = (int32_t)std::min<int64_t>(idx.capacity, INT32_MAX);
  k_post_normalize<<<sms * 4, 256, 0, s>>>(idx.col_ptr, (int32_t)idx.dim, capacity, idx.post_item,
                                            idx.post_val, inv_i, h->post_hat);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  PostArgs a;
  a.q_indptr = queries.indptr;
  a.q_idx = queries.indices;
  a.q_val = queries.values;
  a.n_q = queries.n_rows;
  a.inv_q = inv_q;
  a.col_ptr = idx.col_ptr;
  a.post_hat = h->post_hat;
  a.capacity = capacity;
  a.dim = (int32_t)idx.dim;
  a.n_items = idx.n_items;
  a.window = posting_window(idx.n_items);
  a.out = out;
  a.ld_out = ld_out;
  a.vec_ok = ((reinterpret_cast<uintptr_t>(out) % 16) == 0) && (ld_out % 4 == 0);
  a.topk = topk ? *topk : ss_topk();
  a.row_next = h->row_next;
  a.status = h->d_status;
  const size_t smem = posting_smem_bytes(a.window);
  static size_t configured = 0;
  if (configured < smem) {
    e = cudaFuncSetAttribute(k_score_lists, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_score_lists, kPThreads, smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(queries.n_rows, (int64_t)sms * std::max(per_sm, 1)));
  k_score_lists<<<(unsigned)grid, kPThreads, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *queued = 2;
  return cudaSuccess;
}
