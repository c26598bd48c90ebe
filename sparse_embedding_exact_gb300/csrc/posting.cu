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
// reach 2^31 (every kFoldDims query dimensions).  The store rounds the exact
// total to float once.  Error per score: float rounding of the three
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

#include "hotset.cuh"
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
  const int32_t *hot;      // the item matrix's hot set: hot[0] = H
  const float *base;       // split lists (H >= kSplitMinHot): the dense hot scores to add to
  int64_t ld_base;
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

// Producer.  Jobs follow one another: every segment of kSeg dimensions of a
// row, for every accumulator window, rows in the order the row counter hands
// them out.  Each job takes two dependent loads (the query entries, then the
// column pointers of their dimensions), so the producer runs a two-stage
// pipeline: while the column pointers of job n are in flight it already
// loads the query entries of job n + 1; rows are claimed two ahead and their
// row pointers read one row ahead.  All positions fit in 32 bits (nnz < 2^31).
struct RowQ {
  int32_t q, jb, je;
  float iq;
};

__device__ __forceinline__ RowQ load_row(const PostArgs &a, int32_t q) {
  RowQ r{q, 0, 0, 0.f};
  if (q < a.n_q) {
    r.jb = (int32_t)__ldg(a.q_indptr + q);
    r.je = (int32_t)__ldg(a.q_indptr + q + 1);
    r.iq = __ldg(a.inv_q + q);
  }
  return r;
}

struct JobD {
  int32_t q, s0, s1, w, flags;
  float iq;
};

// Stage 1: the job's query entries (dimension, value).
__device__ __forceinline__ void load_entries(const PostArgs &a, const JobD &d, int lane,
                                             int32_t (&k)[kPerLane], float (&v)[kPerLane]) {
#pragma unroll
  for (int m = 0; m < kPerLane; ++m) {
    const int32_t j = d.s0 + lane + 32 * m;
    k[m] = -1;
    v[m] = 0.f;
    if (j < d.s1) {
      k[m] = __ldg(a.q_idx + j);
      v[m] = __ldg(a.q_val + j);
    }
  }
}

// Stage 2: each dimension's list (start, length) and the scaled query value.
struct SegRegs {
  int32_t start[kPerLane];
  int32_t len[kPerLane];
  float qv[kPerLane];
};

__device__ __forceinline__ void lookup_lists(const PostArgs &a, float iq, const int32_t (&k)[kPerLane],
                                             const float (&v)[kPerLane], SegRegs &r) {
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
// prefix, start - exclusive prefix, value bits, exclusive prefix}.  Returns
// the counts.
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
      lists[pos] = make_int4(incl, r.start[m] - (incl - r.len[m]), __float_as_int(r.qv[m]), incl - r.len[m]);
    }
    n_lists += __popc(mask);
    n_entries = __shfl_sync(0xffffffffu, incl, 31);
  }
  return make_int2(n_lists, n_entries);
}

__device__ __forceinline__ int32_t claim_row(const PostArgs &a, int lane) {
  int32_t q = 0;
  if (lane == 0) q = atomicAdd(a.row_next, 1);
  return __shfl_sync(0xffffffffu, q, 0);
}

__device__ __forceinline__ void producer(const PostArgs &a, int4 *lists, Job *jobs) {
  const int lane = threadIdx.x & 31;
  const int n_windows = (a.n_items + a.window - 1) / a.window;
  // Rows: cur (being cut into jobs), nxt (row pointers loaded), q_after (claimed).
  const int32_t q0 = claim_row(a, lane);
  const int32_t q1 = claim_row(a, lane);
  int32_t q_after = claim_row(a, lane);
  RowQ cur = load_row(a, q0);
  RowQ nxt = load_row(a, q1);
  int w = 0, since_fold = 0;
  int32_t s0 = cur.jb;
  // The job at the cursor; advancing moves the cursor to the next job.
  auto make_job = [&]() {
    JobD d;
    d.q = cur.q;
    d.iq = cur.iq;
    d.w = w;
    d.s0 = s0;
    d.s1 = min(s0 + kSeg, cur.je);
    int f = 0;
    if (cur.q >= a.n_q) f |= kJobDone;
    if (s0 == cur.jb) f |= kJobFirst;
    if (d.s1 >= cur.je) f |= kJobLast;
    if (since_fold >= kFoldDims) f |= kJobFold;
    d.flags = f;
    return d;
  };
  auto advance = [&](const JobD &d) {
    since_fold = (d.flags & kJobFold) ? kSeg : since_fold + kSeg;
    if (d.s1 < cur.je) {
      s0 = d.s1;
    } else if (w + 1 < n_windows) {
      ++w;
      s0 = cur.jb;
      since_fold = 0;
    } else {
      cur = nxt;
      nxt = load_row(a, q_after);  // its claim returned long ago
      q_after = claim_row(a, lane);
      w = 0;
      s0 = cur.jb;
      since_fold = 0;
    }
  };
  JobD d = make_job();
  int32_t k[kPerLane];
  float v[kPerLane];
  if (!(d.flags & kJobDone)) load_entries(a, d, lane, k, v);
  int n_job = 0;
  for (;;) {
    const bool done = (d.flags & kJobDone) != 0;
    SegRegs r;
    if (!done) {
      lookup_lists(a, d.iq, k, v, r);
    } else {
#pragma unroll
      for (int m = 0; m < kPerLane; ++m) r.len[m] = 0;
    }
    JobD dn = d;
    if (!done) {  // stage 1 of the next job overlaps stage 2 of this one
      advance(d);
      dn = make_job();
      if (!(dn.flags & kJobDone)) load_entries(a, dn, lane, k, v);
    }
    const int b = n_job & 1;
    if (n_job >= 2) bar_sync(kBarEmpty + b, kPThreads);  // job n_job - 2 released buffer b
    const int2 cnt = write_segment(r, lists + b * kSeg, lane);
    if (lane == 0) {
      Job &j = jobs[b];
      j.row = d.q;
      j.window = d.w * a.window;
      j.n_lists = cnt.x;
      j.n_entries = cnt.y;
      j.flags = d.flags;
    }
    __syncwarp();
    bar_arrive(kBarFull + b, kPThreads);
    ++n_job;
    if (done) break;
    d = dn;
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

// Adds one entry's product to the accumulator.  A |x| above the bound of
// normalised products is reported (the sum is then not exact); it is not
// clamped, the magic-number split stays defined for any float.
__device__ __forceinline__ void add_product(int32_t *acc_hi, int32_t *acc_lo, int it, float x,
                                            bool &bad) {
  bad |= fabsf(x) > kXValid;
  const float y = x + kMagic;
  const int32_t hi = __float_as_int(y) - kMagicBits;
  const float rem = x - (y - kMagic);
  const int32_t lo = __float_as_int(fmaf(rem, kLoScale, kMagic)) - kMagicBits;
  atomicAdd(acc_hi + it, hi);
  atomicAdd(acc_lo + it, lo);
}

// Number of the segment's lists whose inclusive prefix is <= e (the list
// holding entry e): 32 samples, then the 32 lists after the last sample that
// passed.  lists[].x increases strictly, and n_lists <= kSeg <= 32 * 32.
__device__ __forceinline__ int first_list(const int4 *lists, int n_lists, int e, int lane) {
  const int stride = (n_lists + 31) >> 5;
  const int js = lane * stride;
  const int c1 = __popc(__ballot_sync(0xffffffffu, js < n_lists && lists[js].x <= e));
  if (c1 == 0) return 0;
  const int j0 = (c1 - 1) * stride + 1;
  const int j = j0 + lane;
  return j0 + __popc(__ballot_sync(0xffffffffu, lane < stride - 1 && j < n_lists && lists[j].x <= e));
}

// One consumer warp's share [e0, e1) of a segment's entries, 32 per round.
// Lane t of a round takes entry rb + t.  Candidate lane l holds list jc + l;
// the lists that start inside the round set one bit each at their start
// offset, and lane t's list is jc + (bits set in 1..t).
template <bool kWindowed>
__device__ __forceinline__ void walk(const PostArgs &a, const int4 *lists, int n_lists, int e0,
                                     int e1, int w0, int32_t *acc_hi, int32_t *acc_lo, int lane,
                                     bool &bad) {
  if (e0 >= e1) return;
  int jc = first_list(lists, n_lists, e0, lane);
  const unsigned upto = (lane == 31 ? 0xffffffffu : ((2u << lane) - 1u)) & ~1u;  // bits 1..lane
  const unsigned W = (unsigned)a.window;
  for (int base = e0; base < e1; base += 32 * kRoundsPerStep) {
    int2 ent[kRoundsPerStep];
    float qv[kRoundsPerStep];
    bool live[kRoundsPerStep];
#pragma unroll
    for (int u = 0; u < kRoundsPerStep; ++u) {
      const int rb = base + 32 * u;
      live[u] = false;
      ent[u] = make_int2(0, 0);
      qv[u] = 0.f;
      if (rb < e1) {  // warp-uniform
        const int cand = jc + lane;
        const int4 c = cand < n_lists ? lists[cand] : make_int4(INT_MAX, 0, 0, INT_MAX);
        const int off = c.w - rb;
        const unsigned starts = __reduce_or_sync(0xffffffffu, (off > 0 && off < 32) ? (1u << off) : 0u);
        const int pos = __popc(starts & upto);
        const int bj = __shfl_sync(0xffffffffu, c.y, pos);
        qv[u] = __int_as_float(__shfl_sync(0xffffffffu, c.z, pos));
        const int e = rb + lane;
        live[u] = e < e1;
        if (live[u]) ent[u] = __ldg(a.post_hat + (bj + e));
        jc += __popc(__ballot_sync(0xffffffffu, c.x <= rb + 32));
      }
    }
#pragma unroll
    for (int u = 0; u < kRoundsPerStep; ++u) {
      if (kWindowed) {
        const unsigned it = (unsigned)(ent[u].x - w0);
        if (live[u] && it < W) add_product(acc_hi, acc_lo, (int)it, qv[u] * __int_as_float(ent[u].y), bad);
      } else if (live[u]) {
        add_product(acc_hi, acc_lo, ent[u].x, qv[u] * __int_as_float(ent[u].y), bad);
      }
    }
  }
}

// The score of one accumulator pair, rounded once: the carry of lo moves
// into hi (lo in [0, 2^17), |hi| < 2^24 for any realistic count of shared
// dimensions), so both convert to float exactly, hi * 2^-21 is exact, and
// the fused multiply-add rounds the exact total (hi * 2^17 + lo) * 2^-38.
__device__ __forceinline__ float acc_value(int32_t hi, int32_t lo) {
  const int32_t carry = lo >> 17;  // arithmetic shift: floor(lo / 2^17)
  hi += carry;
  lo -= carry * (1 << 17);
  return fmaf((float)lo, kOutScale, (float)hi * 0x1p-21f);
}

// Converts the window's accumulators of row q to scores, stores them (or
// offers them to the row's top-k), and zeroes the accumulators.
__device__ __forceinline__ void store_window(const PostArgs &a, int64_t q, int w0, int32_t *acc_hi,
                                             int32_t *acc_lo, int ctid, const float *base_row) {
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
        const int c = (j < 4 ? ia : ib) + (j & 3);
        v[j] = acc_value(hv[j], lv[j]);
        if (base_row && c < width) v[j] += base_row[c];
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
    float o[4] = {acc_value(h4.x, l4.x), acc_value(h4.y, l4.y), acc_value(h4.z, l4.z),
                  acc_value(h4.w, l4.w)};
    if (base_row) {
      if (a.vec_ok && c + 4 <= width) {
        const float4 b4 = *reinterpret_cast<const float4 *>(base_row + c);
        o[0] += b4.x;
        o[1] += b4.y;
        o[2] += b4.z;
        o[3] += b4.w;
      } else {
        for (int j = 0; j < 4 && c + j < width; ++j) o[j] += base_row[c + j];
      }
    }
    if (a.vec_ok && c + 4 <= width) {
      __stcs(reinterpret_cast<float4 *>(orow + c), make_float4(o[0], o[1], o[2], o[3]));
    } else {
      for (int j = 0; j < 4 && c + j < width; ++j) orow[c + j] = o[j];
    }
  }
}

template <bool kWindowed>
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
  const bool add_base = a.base != nullptr && __ldg(a.hot) >= kSplitMinHot;
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
    const int e0 = (int)((uint32_t)j.n_entries * (uint32_t)warp / kCons);  // n_entries < 2^27
    const int e1 = (int)((uint32_t)j.n_entries * (uint32_t)(warp + 1) / kCons);
    walk<kWindowed>(a, lists + b * kSeg, j.n_lists, e0, e1, j.window, acc_hi, acc_lo, lane, bad);
    __syncwarp();
    bar_arrive(kBarEmpty + b, kPThreads);
    if (j.flags & kJobLast) {
      bar_sync(kBarCons, kCons * 32);
      store_window(a, j.row, j.window, acc_hi, acc_lo, threadIdx.x,
                   add_base ? a.base + j.row * a.ld_base + j.window : nullptr);
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


// ---------------------------------------------------------------- split lists
// With kSplitMinHot or more hot dimensions, the hot part of every score is a
// small dense product, computed first and written normalised:
//   dst[q][i] = (sum over h of qhot[q][h] * slab[h][i]) * inv_q[q] * inv_i[i]
// (float32, h ascending); the list walk of the cold dimensions then adds its
// exact fixed-point sum to it.  kDQ x kDI tiles, K = H <= kHotMax, an 8 x 8
// register tile per thread.
constexpr int kDQ = 128, kDI = 128, kDThreads = 256;

// Query hot values, per tile of kDQ rows transposed: qhot[tile][h][row]
// (0 where the row lacks dimension h; rows past n_q are 0).  One warp per row.
__global__ void __launch_bounds__(256)
    k_prep_hot_dense(const int64_t *__restrict__ indptr, const int32_t *__restrict__ idx,
                     const float *__restrict__ val, int64_t n_q, int64_t n_rows_padded,
                     const int32_t *__restrict__ hot, float *__restrict__ qhot) {
  __shared__ int hkeys[hotset::kHotSlots];
  __shared__ int8_t hvals[hotset::kHotSlots];
  hotset::load_hot_set(hot, hkeys, hvals);
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < n_rows_padded; r += warps) {
    float *t = qhot + (r / kDQ) * hyb::kHotMax * kDQ + (r % kDQ);
    t[lane * kDQ] = 0.f;  // kHotMax == 32: one slot per lane
    __syncwarp();
    if (r >= n_q) continue;
    for (int64_t p = indptr[r] + lane; p < indptr[r + 1]; p += 32) {
      const int hh = hotset::hot_find(hkeys, hvals, __ldg(idx + p));
      if (hh >= 0) t[hh * kDQ] = __ldg(val + p);
    }
  }
}

__global__ void __launch_bounds__(kDThreads)
    k_hot_dense(const float *__restrict__ qhot, int64_t n_q, const float *__restrict__ inv_q,
                const int32_t *__restrict__ hot, const float *__restrict__ slab, int32_t slab_ld,
                int32_t n_items, const float *__restrict__ inv_i, float *__restrict__ dst,
                int64_t ld_dst, int vec_ok) {
  const int H = __ldg(hot);
  if (H < kSplitMinHot) return;
  __shared__ __align__(16) float qs[hyb::kHotMax][kDQ];
  __shared__ __align__(16) float is[hyb::kHotMax][kDI];
  const int64_t q0 = (int64_t)blockIdx.x * kDQ;
  const int i0 = blockIdx.y * kDI;
  const int tid = threadIdx.x;
  const float *qt = qhot + (int64_t)blockIdx.x * hyb::kHotMax * kDQ;
  for (int j = tid; j < H * kDQ / 4; j += kDThreads)
    reinterpret_cast<float4 *>(&qs[0][0])[j] = __ldg(reinterpret_cast<const float4 *>(qt) + j);
  for (int j = tid; j < H * kDI; j += kDThreads) {
    const int hh = j / kDI, c = j % kDI;
    is[hh][c] = i0 + c < n_items ? __ldg(slab + (size_t)hh * slab_ld + i0 + c) : 0.f;
  }
  __syncthreads();
  const int tx = tid & 15, ty = tid >> 4;
  float acc[8][8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
  for (int hh = 0; hh < H; ++hh) {
    const float4 a0 = *reinterpret_cast<const float4 *>(&qs[hh][ty * 8]);
    const float4 a1 = *reinterpret_cast<const float4 *>(&qs[hh][ty * 8 + 4]);
    const float4 b0 = *reinterpret_cast<const float4 *>(&is[hh][tx * 4]);
    const float4 b1 = *reinterpret_cast<const float4 *>(&is[hh][64 + tx * 4]);
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
  }
  int col[8];
  float ni[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    col[c] = (c < 4 ? tx * 4 + c : 64 + tx * 4 + (c - 4));
    ni[c] = i0 + col[c] < n_items ? __ldg(inv_i + i0 + col[c]) : 0.f;
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int64_t q = q0 + ty * 8 + r;
    if (q >= n_q) break;
    const float iq = __ldg(inv_q + q);
    float *row = dst + q * ld_dst + i0;
    float o[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = acc[r][c] * iq * ni[c];
    if (vec_ok && i0 + kDI <= n_items) {
      *reinterpret_cast<float4 *>(row + tx * 4) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4 *>(row + 64 + tx * 4) = make_float4(o[4], o[5], o[6], o[7]);
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (i0 + col[c] < n_items) row[col[c]] = o[c];
    }
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

// Dense query hot values for the current hot set, redone when the query
// matrix or the hot set changes.
static cudaError_t prepare_hot_dense(ss_handle *h, const ss_csr &q, cudaStream_t s, int *queued) {
  *queued = 0;
  if (h->qd_src[0] == q.indptr && h->qd_src[1] == q.indices && h->qd_src[2] == q.values &&
      h->qd_rows == q.n_rows && h->qd_nnz == q.nnz && h->qd_generation == h->hot_generation)
    return cudaSuccess;
  const int64_t rows_padded = (q.n_rows + kDQ - 1) / kDQ * kDQ;
  const int64_t need = std::max<int64_t>(1, rows_padded * hyb::kHotMax);
  cudaError_t e;
  if (need > h->qhot_dense_cap) {
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
    cudaFree(h->qhot_dense);
    h->qhot_dense = nullptr;
    h->qhot_dense_cap = 0;
    if ((e = dev_alloc(&h->qhot_dense, sizeof(float) * (size_t)need)) != cudaSuccess) return e;
    h->qhot_dense_cap = need;
  }
  const int64_t blocks = (rows_padded + 7) / 8;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)h->sm_count * 8));
  k_prep_hot_dense<<<grid, 256, 0, s>>>(q.indptr, q.indices, q.values, q.n_rows, rows_padded, h->hot,
                                        h->qhot_dense);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  h->qd_src[0] = q.indptr;
  h->qd_src[1] = q.indices;
  h->qd_src[2] = q.values;
  h->qd_rows = q.n_rows;
  h->qd_nnz = q.nnz;
  h->qd_generation = h->hot_generation;
  *queued = 1;
  return cudaSuccess;
}

cudaError_t launch_score_lists(ss_handle *h, const ss_csr &queries, const float *inv_q,
                               const ss_index &idx, const float *inv_i, float *out, int64_t ld_out,
                               cudaStream_t s, int *queued, const ss_topk *topk) {
  *queued = 0;
  if (queries.n_rows == 0 || idx.n_items == 0) return cudaSuccess;
  if (queries.n_rows >= INT32_MAX - 65536) return cudaErrorInvalidValue;
  const int sms = h->sm_count > 0 ? h->sm_count : 148;
  cudaError_t e = cudaSuccess;
  int queued_prep = 0;
  if (idx.hot) {
    // Split lists: the query hot values (once per query matrix and hot set),
    // then the dense hot scores of the chunk, which the walk adds to.
    e = prepare_hot_dense(h, queries, s, &queued_prep);
    if (e != cudaSuccess) return e;
  }
  const int32_t capacity = (int32_t)std::min<int64_t>(idx.capacity, INT32_MAX);
  k_post_normalize<<<sms * 4, 256, 0, s>>>(idx.col_ptr, (int32_t)idx.dim, capacity, idx.post_item,
                                            idx.post_val, inv_i, h->post_hat);
  e = cudaGetLastError();
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
  a.hot = idx.hot;
  a.base = nullptr;
  a.ld_base = 0;
  a.status = h->d_status;
  const size_t smem = posting_smem_bytes(a.window);
  int queued_dense = 0;
  if (idx.hot) {
    // The dense hot scores go straight to the output (full scores) or to a
    // scratch matrix the top-k offers read; both kernels skip the split on
    // the device when the hot set is smaller than kSplitMinHot.
    float *dst = out;
    int64_t ld_dst = ld_out;
    if (a.topk.k > 0) {
      const int64_t need = queries.n_rows * (int64_t)idx.n_items;
      if (need > h->hot_scratch_cap) {
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
        cudaFree(h->hot_scratch);
        h->hot_scratch = nullptr;
        h->hot_scratch_cap = 0;
        if ((e = dev_alloc(&h->hot_scratch, sizeof(float) * (size_t)need)) != cudaSuccess) return e;
        h->hot_scratch_cap = need;
      }
      dst = h->hot_scratch;
      ld_dst = idx.n_items;
    }
    const int dvec = ((reinterpret_cast<uintptr_t>(dst) % 16) == 0) && (ld_dst % 4 == 0);
    dim3 dgrid((unsigned)((queries.n_rows + kDQ - 1) / kDQ), (unsigned)((idx.n_items + kDI - 1) / kDI));
    k_hot_dense<<<dgrid, kDThreads, 0, s>>>(h->qhot_dense, queries.n_rows, inv_q, idx.hot, idx.slab,
                                            idx.slab_ld, idx.n_items, inv_i, dst, ld_dst, dvec);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    a.base = dst;
    a.ld_base = ld_dst;
    queued_dense = 1;
  }
  // One window covers the chunk unless it is wider than kWindowMax items.
  const bool windowed = a.n_items > a.window;
  auto kernel = windowed ? k_score_lists<true> : k_score_lists<false>;
  if ((e = ensure_dyn_smem(kernel, smem)) != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kPThreads, smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(queries.n_rows, (int64_t)sms * std::max(per_sm, 1)));
  prof_mark(h, s);
  kernel<<<(unsigned)grid, kPThreads, smem, s>>>(a);
  prof_mark(h, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *queued = 2 + queued_prep + queued_dense;
  return cudaSuccess;
}
