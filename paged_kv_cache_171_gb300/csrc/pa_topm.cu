// pa_topm.cu -- budgeted global top-M KV retention.
//
// "推理系统与性能工程" 19.4.3 (KV-cache compression, budgeted eviction): given
// a score per (layer l, head h, token t) and a global budget of M kept K/V
// rows, position C of every (layer, head) is kept unconditionally and the
// other (l, h, t) compete for the remaining M - L*H rows in ONE global order,
// key = (-score, l, h, t) ascending.  The key is a total order, so the kept
// set is unique.
//
// On the GPU the order is split in two parts.  The score part is a 32-bit
// key f(score) whose ascending order is descending score (-0.0 as 0.0, NaN
// after every number); the (l, h, t) part is the element's index in the
// [L][H][N] array, so index order already is the tie order.  A radix select
// over f (digits of 11, 11 and 10 bits, most significant first) finds the key
// S* of the K-th candidate and its rank r among the candidates whose key
// equals S*.  The kept candidates are then exactly: f < S*, plus the first r
// with f = S* in index order.
//
// One pass streams the scores when a sample can name the first digit.  A
// histogram of the top 11 bits over every 32nd chunk of the array, and a
// one-CTA pick, name the bucket b1 that holds the K-th key -- if the K-th
// sample lies more than six standard deviations of its sampling error from
// both edges of its bucket.  The split pass then settles every element
// outside b1 (kept if its bucket is below b1, dropped if above), writes the
// keep mask, appends the (index, key) of b1's elements to a candidate list,
// and counts the kept elements below b1 exactly; b1 is confirmed when the
// K-th key falls among b1's candidates by those counts.  Otherwise (the
// sample unsure, or wrong) the exact first digit runs: a histogram over every
// element, its pick, and the split pass again.  Arrays under 512 chunks take
// the exact first digit directly.  The remaining digits, the tie rank and the
// final keeps then run over the candidates alone: the r-th tie is located by
// counting ties per chunk of the array, then (one launch) scanning the counts
// to find its chunk and ranking that one chunk's ties; with its index idx*, a
// candidate is kept when (f, index) <= (S*, idx*).
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 16;                     // consecutive elements per thread
constexpr int kChunk = kThreads * kPerThread;      // elements per chunk (final passes)

constexpr int kBins1 = 2048, kBins2 = 2048, kBins3 = 1024;  // digits of 11, 11, 10 bits
constexpr int kShift1 = 21, kShift2 = 10;
constexpr int kSampleStep = 32;  // the first-digit sample: every 32nd chunk

// Division by the row length N (tokens per (layer, head)) for dividends below
// 2^31 by a multiply and a shift -- division by an invariant integer
// (Granlund and Montgomery, 1994): with s = ceil(log2 N) and
// M = ceil(2^(31+s) / N) < 2^32, floor(x / N) = floor(x M / 2^(31+s)) for every
// x < 2^31, since x (M - 2^(31+s)/N) / 2^(31+s) < 2^-s <= 1/N.
struct RowDiv {
  int N;
  uint32_t M, sh;
  __device__ __forceinline__ int div(int x) const {
    return static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(x)) * M) >> sh);
  }
};

RowDiv make_rowdiv(int N) {
  uint32_t s = 0;
  while ((static_cast<int64_t>(1) << s) < N) ++s;
  const uint64_t p = static_cast<uint64_t>(1) << (31 + s);
  return RowDiv{N, static_cast<uint32_t>((p + static_cast<uint64_t>(N) - 1) / static_cast<uint64_t>(N)),
                31 + s};
}

// The state of the select, in the workspace after the histograms (128-byte
// aligned).  The split pass's counters sit in a cache line of their own: every
// split CTA reads b1 from the first line, and an atomic on that line would
// evict the copies the SMs' L1 caches hold.
struct TopmState {
  uint32_t prefix;     // key bits decided so far (S* at the end)
  uint32_t mask;       // which bits are decided
  uint32_t k_rem;      // 1-based rank still to find inside the current bucket
  uint32_t tie_chunk;  // chunk holding the k_rem-th candidate with key S*
  uint32_t tie_rank;   // its 1-based rank among that chunk's ties
  uint32_t idx_star;   // its index: the last kept candidate
  uint32_t pad0[2];
  uint32_t sure;       // 1: b1 named by the sample (the split pass ran on it)
  uint32_t redo;       // 1: b1 not confirmed; the exact first digit runs
  uint32_t k_total;    // K, the candidates to keep
  uint32_t pad1[21];
  uint32_t n_cand;     // elements of bucket b1 appended to the candidate list
  uint32_t kept_below; // kept candidates of buckets below b1 (the split pass)
  uint32_t pad2[30];
};
static_assert(sizeof(TopmState) == 256 && offsetof(TopmState, n_cand) == 128,
              "two cache lines, the counters in the second");
static_assert(offsetof(TopmState, kept_below) == offsetof(TopmState, n_cand) + 4,
              "n_cand and kept_below are the low and high words of one 64-bit counter");
static_assert((kBins1 + kBins2 + kBins3) * 4 % 128 == 0, "the state starts a cache line");
static_assert(offsetof(TopmState, n_cand) % 8 == 0 &&
                  offsetof(TopmState, kept_below) == offsetof(TopmState, n_cand) + 4,
              "n_cand and kept_below are the low and high words of one 64-bit counter");

// Ascending f <=> descending score; -0.0 as 0.0; NaN after every number.
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0xFFFFFFFFu;
  uint32_t u = __float_as_uint(s == 0.f ? 0.f : s);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending order of s
  return ~u;                                        // descending
}

// A score s that is a number has key f(s) <= K exactly when s >= key_floor(K):
// the number whose key is K (f is strictly decreasing on the numbers once -0.0
// is read as 0.0, which float comparison does too); +NaN when K is below the
// key of +inf (no number qualifies: every comparison with NaN is false); -inf
// when K is at least the key of -inf (every number qualifies).  A NaN score
// compares false with every bound; its key is the largest.
__device__ __forceinline__ float key_floor(uint32_t K) {
  if (K < 0x007FFFFFu) return __uint_as_float(0x7FC00000u);
  if (K >= 0xFF800000u) return __uint_as_float(0xFF800000u);
  const uint32_t u = ~K;
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Zeroes the three histograms, the per-chunk tie counts and the kept-row
// counts, sets the state.
__global__ void __launch_bounds__(kThreads)
    topm_init_kernel(uint32_t *__restrict__ hist, int n_hist, uint32_t *__restrict__ tiecnt,
                     int n_chunks, int32_t *__restrict__ per_head, int n_rows,
                     TopmState *__restrict__ st, uint32_t k) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  const int stride = gridDim.x * kThreads;
  for (int i = blockIdx.x * kThreads + threadIdx.x; i < n_hist; i += stride) hist[i] = 0;
  for (int i = blockIdx.x * kThreads + threadIdx.x; i < n_chunks; i += stride) tiecnt[i] = 0;
  if (per_head)
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < n_rows; i += stride) per_head[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    TopmState z = {};
    z.k_rem = z.k_total = k;
    *st = z;
  }
}

// The kPerThread consecutive scores from `base` (16-byte aligned when the
// run is whole; the array holds fewer than 2^31 elements).
__device__ __forceinline__ void load_run(const float *__restrict__ scores, int n, int base,
                                         float (&sc)[kPerThread]) {
  if (base + kPerThread <= n) {
#pragma unroll
    for (int e = 0; e < kPerThread; e += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(scores + base + e));
      sc[e] = v.x;
      sc[e + 1] = v.y;
      sc[e + 2] = v.z;
      sc[e + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) sc[e] = base + e < n ? __ldg(scores + base + e) : 0.f;
  }
}

// Inclusive prefix sum of v over the CTA's NT threads (NT a multiple of 32,
// at most 1024; once per kernel): a shuffle scan inside each warp, then one
// over the warp totals -- two barriers.
template <int NT>
__device__ __forceinline__ uint32_t block_scan_incl(uint32_t v) {
  __shared__ uint32_t wsum[NT / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) wsum[wid] = v;
  __syncthreads();
  if (wid == 0) {
    uint32_t w = lane < NT / 32 ? wsum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < NT / 32) wsum[lane] = w;
  }
  __syncthreads();
  return v + (wid > 0 ? wsum[wid - 1] : 0u);
}

// First digit: histogram of the top 11 key bits over the candidate elements
// of every `step`-th chunk (32: the sample; 1: every element).  Each quarter
// of the CTA's warps counts into its own copy in shared memory (fewer
// collisions on the few crowded bins), summed at the end.  gated: the exact
// pass after the split, run only when the split pass's counts do not confirm
// the sampled b1 (every CTA decides alike from fields no kernel of this step
// writes; CTA 0 records it, and the remaining rank when confirmed).
__global__ void __launch_bounds__(kThreads)
    topm_hist1_kernel(const float *__restrict__ scores, int n, RowDiv rd, int current,
                      uint32_t *__restrict__ hist, int step, TopmState *__restrict__ st,
                      int gated) {
  const int N = rd.N;
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  if (gated) {
    const uint32_t K = st->k_total, below = st->kept_below, nc = st->n_cand;
    const bool ok = st->sure && below < K && K <= below + nc;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      st->redo = ok ? 0u : 1u;
      st->k_rem = ok ? K - below : K;
    }
    if (ok) return;
  }
  constexpr int kCopies = 4;
  __shared__ uint32_t h[kCopies][kBins1];
  for (int i = threadIdx.x; i < kCopies * kBins1; i += kThreads) h[i / kBins1][i % kBins1] = 0;
  __syncthreads();
  uint32_t *mine = h[(threadIdx.x >> 5) & (kCopies - 1)];
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kChunk * step;
  float nx[kPerThread];  // the next chunk's run, loaded while this one is counted
  int64_t cbase = static_cast<int64_t>(blockIdx.x) * kChunk * step;
  if (cbase < n) load_run(scores, n, static_cast<int>(cbase) + threadIdx.x * kPerThread, nx);
  for (; cbase < n; cbase += stride) {
    const int base = static_cast<int>(cbase) + threadIdx.x * kPerThread;
    float sc[kPerThread];
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) sc[e] = nx[e];
    if (cbase + stride < n)
      load_run(scores, n, static_cast<int>(cbase + stride) + threadIdx.x * kPerThread, nx);
    const int t0 = base - rd.div(base) * N;
    uint32_t skip;  // elements that are a current position or past the array
    if (base + kPerThread <= n && N >= kPerThread) {
      skip = 0;
      if (current >= t0 && current - t0 < kPerThread) skip |= 1u << (current - t0);
      const unsigned e1 = static_cast<unsigned>(N - t0) + static_cast<unsigned>(current);
      if (e1 < static_cast<unsigned>(kPerThread)) skip |= 1u << e1;
    } else {
      skip = 0;
      int t = t0;
#pragma unroll
      for (int e = 0; e < kPerThread; ++e) {
        if (base + e >= n || t == current) skip |= 1u << e;
        if (++t == N) t = 0;
      }
    }
#pragma unroll
    for (int e = 0; e < kPerThread; ++e)
      if (!(skip >> e & 1u)) atomicAdd(&mine[score_key(sc[e]) >> kShift1], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBins1; i += kThreads) {
    uint32_t v = 0;
#pragma unroll
    for (int c = 0; c < kCopies; ++c) v += h[c][i];
    if (v) atomicAdd(&hist[i], v);
  }
}

// One CTA of 1024 threads: the bin of `hist` (BINS bins, digit at `shift`)
// holding the k_rem-th key of the current bucket; clears the histogram.
// gated (the exact first digit): only when the sampled b1 was not confirmed,
// after clearing what the split pass on it counted.
template <int BINS>
__global__ void __launch_bounds__(1024)
    topm_pick_kernel(uint32_t *__restrict__ hist, TopmState *__restrict__ st, int shift,
                     int gated, int32_t *__restrict__ per_head, int n_rows) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  if (gated) {
    if (!st->redo) return;
    if (per_head)
      for (int i = threadIdx.x; i < n_rows; i += 1024) per_head[i] = 0;
    if (threadIdx.x == 0) {
      st->n_cand = 0u;
      st->kept_below = 0u;
      st->prefix = 0u;
      st->mask = 0u;
    }
    __syncthreads();
  }
  constexpr int kPer = BINS / 1024;
  const int t = threadIdx.x;
  uint32_t v[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    v[i] = hist[kPer * t + i];
    sum += v[i];
  }
  const uint32_t incl = block_scan_incl<1024>(sum);
  const uint32_t k = st->k_rem;
  uint32_t before = incl - sum;
  if (before < k && k <= incl) {  // exactly one thread
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (before < k && k <= before + v[i]) {
        st->k_rem = k - before;
        st->prefix |= static_cast<uint32_t>(kPer * t + i) << shift;
        st->mask |= static_cast<uint32_t>(BINS - 1) << shift;
      }
      before += v[i];
    }
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) hist[kPer * t + i] = 0;
}

// One CTA of 1024 threads: b1 from the sample histogram (kBins1 bins) when
// the K-th key's place among the sampled candidates, K_s = K n_s / n_c, lies
// more than 6 sigma + 4 (sigma^2 = K_s (1 - K_s / n_s), the binomial
// sampling error) inside its bucket; clears the histogram.  Single precision
// and one thread for the bounds: a bin qualifies when its cumulative counts
// satisfy before < K_s - margin and after >= K_s + margin, which at most one
// bin does (the conversions to float keep the counts' order).
__global__ void __launch_bounds__(1024)
    topm_pick_sample_kernel(uint32_t *__restrict__ hist, TopmState *__restrict__ st,
                            float n_cands) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  constexpr int kPer = kBins1 / 1024;
  const int t = threadIdx.x;
  uint32_t v[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    v[i] = hist[kPer * t + i];
    sum += v[i];
  }
  const uint32_t incl = block_scan_incl<1024>(sum);
  __shared__ float s_lo, s_hi;
  if (t == 1023) {
    const float ns = static_cast<float>(incl);
    const float ks = static_cast<float>(st->k_total) * ns / n_cands;
    const float margin = 6.f * sqrtf(fmaxf(ks * (1.f - ks / fmaxf(ns, 1.f)), 0.f)) + 4.f;
    s_lo = incl >= 4096u ? ks - margin : -1.f;  // too small a sample: no bin
    s_hi = ks + margin;
  }
  __syncthreads();
  const float lo = s_lo, hi = s_hi;
  uint32_t before = incl - sum;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t after = before + v[i];
    if (static_cast<float>(before) < lo && static_cast<float>(after) >= hi) {
      st->prefix = static_cast<uint32_t>(kPer * t + i) << kShift1;
      st->mask = static_cast<uint32_t>(kBins1 - 1) << kShift1;
      st->sure = 1u;
    }
    before = after;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) hist[kPer * t + i] = 0;
}

// Second pass over the scores.  Every element outside bucket b1 is settled:
// kept (current position, or a bucket below b1) or dropped; b1's elements
// are written 0 here and appended to the candidate list.  Kept rows per
// (layer, head) are summed in shared memory, then added once per CTA; so are
// the kept elements of buckets below b1 (current positions excepted), in the
// high word of the same 64-bit atomic that reserves the CTA's candidate slots.
// LONG (rows of at least kChunk tokens): a chunk meets at most two rows, so
// each warp sums its kept counts of the two by shuffles and the CTA adds them
// from the warp totals -- no shared counters to clear or contend on.
template <bool LONG>
__device__ __forceinline__ void split_chunk(const float *__restrict__ scores, int n, RowDiv rd,
                                            int current, uint32_t b1, int cbase,
                                            TopmState *__restrict__ st,
                                            uint8_t *__restrict__ keep,
                                            int32_t *__restrict__ per_head,
                                            uint32_t *__restrict__ cand,
                                            uint32_t *__restrict__ ckey) {
  __shared__ int cnt[LONG ? 1 : kChunk + 2];  // rows of this chunk, relative to its first
  __shared__ uint32_t wsum[kThreads / 32 + 1], wbel[kThreads / 32], wrow[2][kThreads / 32];
  const int N = rd.N;
  const int row0 = rd.div(cbase);
  const int cend = min(n, cbase + kChunk);
  const int n_rows = rd.div(cend - 1) - row0 + 1;
  if (!LONG && per_head) {
    for (int i = threadIdx.x; i < n_rows; i += kThreads) cnt[i] = 0;
    __syncthreads();
  }
  const int base = cbase + threadIdx.x * kPerThread;
  float sc[kPerThread];
  load_run(scores, n, base, sc);
  const int rb = rd.div(base);
  const int t0 = base - rb * N, r0 = rb - row0;
  // Bucket b1 holds keys [b1 << 21, (b1 + 1) << 21): a score is below it when
  // s >= lo_s, in it or below when s >= hi_s, by float comparisons instead of
  // keys.  NaN scores (the largest key) are in b1 only when b1 is the last
  // bucket, where every number is below it.
  const float lo_s = b1 == 0u ? __uint_as_float(0x7FC00000u) : key_floor((b1 << kShift1) - 1u);
  const float hi_s = key_floor(((b1 + 1u) << kShift1) - 1u);
  const bool last = b1 == static_cast<uint32_t>(kBins1 - 1);
  // bit e (e < 16): element base + e is kept / a candidate; bits 16..: the
  // kept candidates (not current positions) below b1
  uint32_t kbits = 0, cbits = 0;
  if (base + kPerThread <= n && N >= kPerThread) {
    // Whole run, at most one row boundary (at element N - t0 when t0 + 16 > N):
    // decisions as bit masks, no per-element branches.
    uint32_t cur = 0;  // the current positions among the 16
    if (current >= t0 && current - t0 < kPerThread) cur |= 1u << (current - t0);
    const unsigned e1 = static_cast<unsigned>(N - t0) + static_cast<unsigned>(current);
    if (e1 < static_cast<unsigned>(kPerThread)) cur |= 1u << e1;  // in the next row
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      kbits |= static_cast<uint32_t>(sc[e] >= lo_s) << e;
      cbits |= static_cast<uint32_t>(sc[e] >= hi_s) << e;
    }
    cbits = (last ? (1u << kPerThread) - 1u : cbits) & ~kbits;
    cbits = (cbits & ~cur) | static_cast<uint32_t>(__popc(kbits & ~cur)) << kPerThread;
    kbits |= cur;
    uint4 w;  // bit e of kbits -> byte e
    w.x = ((kbits & 15u) * 0x00204081u) & 0x01010101u;
    w.y = (((kbits >> 4) & 15u) * 0x00204081u) & 0x01010101u;
    w.z = (((kbits >> 8) & 15u) * 0x00204081u) & 0x01010101u;
    w.w = (((kbits >> 12) & 15u) * 0x00204081u) & 0x01010101u;
    *reinterpret_cast<uint4 *>(keep + base) = w;
    if (!LONG && per_head) {
      const int split = N - t0 < kPerThread ? N - t0 : kPerThread;  // elements in row r0
      const uint32_t lo = kbits & ((1u << split) - 1u), hi = kbits >> split;
      if (lo) atomicAdd(&cnt[r0], __popc(lo));
      if (hi) atomicAdd(&cnt[r0 + 1], __popc(hi));
    }
  } else {
    // The array's ragged end, or rows shorter than a run: element by element.
    int t = t0, row = r0;
    int run_row = -1, run = 0;  // kept count of the current (layer, head) run
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      if (base + e >= n) break;
      const bool below = sc[e] >= lo_s, in = !below && (last || sc[e] >= hi_s);
      const bool k = t == current || below;
      if (t != current && in) cbits |= 1u << e;
      if (t != current && below) cbits += 1u << kPerThread;
      kbits |= static_cast<uint32_t>(k) << e;
      keep[base + e] = k ? 1u : 0u;
      if (!LONG && per_head && k) {
        if (row != run_row) {
          if (run) atomicAdd(&cnt[run_row], run);
          run_row = row;
          run = 0;
        }
        ++run;
      }
      if (++t == N) {
        t = 0;
        ++row;
      }
    }
    if (!LONG && per_head && run) atomicAdd(&cnt[run_row], run);
  }
  if (LONG && per_head) {  // kept counts of rows row0 and row0 + 1, per warp
    const int64_t in0 = static_cast<int64_t>(row0 + 1) * N - base;  // this run's in row0
    const uint32_t m0 =
        in0 >= kPerThread ? 0xFFFFu : (in0 <= 0 ? 0u : (1u << static_cast<int>(in0)) - 1u);
    const uint32_t c0 = __reduce_add_sync(0xffffffffu, __popc(kbits & m0));
    const uint32_t c1 = __reduce_add_sync(0xffffffffu, __popc(kbits & ~m0));
    if ((threadIdx.x & 31) == 0) {
      wrow[0][threadIdx.x >> 5] = c0;
      wrow[1][threadIdx.x >> 5] = c1;
    }
  }
  // append the candidates in index order and add the kept-below count: one
  // 64-bit atomic per CTA (candidates in the low word, which cannot carry)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t wbelow = __reduce_add_sync(0xffffffffu, cbits >> kPerThread);
  cbits &= (1u << kPerThread) - 1u;
  const uint32_t mine = __popc(cbits);
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) {
    wsum[warp] = incl;
    wbel[warp] = wbelow;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t tot = 0, bel = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const uint32_t v = wsum[w];
      wsum[w] = tot;
      tot += v;
      bel += wbel[w];
    }
    const unsigned long long add = static_cast<unsigned long long>(bel) << 32 | tot;
    wsum[kThreads / 32] =
        add ? static_cast<uint32_t>(atomicAdd(
                  reinterpret_cast<unsigned long long *>(&st->n_cand), add))
            : 0u;
  }
  __syncthreads();
  uint32_t pos = wsum[kThreads / 32] + wsum[warp] + incl - mine;
  for (uint32_t bits = cbits; bits; bits &= bits - 1) {  // scores re-read: L1 hits
    const int i = base + __ffs(bits) - 1;
    cand[pos] = static_cast<uint32_t>(i);
    ckey[pos++] = score_key(__ldg(scores + i));
  }
  if (LONG) {
    if (per_head && threadIdx.x < 64) {  // warp 0: row0, warp 1: row0 + 1
      const int r = threadIdx.x >> 5, lane = threadIdx.x & 31;
      const uint32_t c =
          __reduce_add_sync(0xffffffffu, lane < kThreads / 32 ? wrow[r][lane] : 0u);
      if (lane == 0 && c) atomicAdd(per_head + row0 + r, static_cast<int>(c));
    }
  } else if (per_head) {
    for (int i = threadIdx.x; i < n_rows; i += kThreads)
      if (cnt[i]) atomicAdd(per_head + row0 + i, cnt[i]);
  }
}

// The split pass, one CTA per chunk.  gate 0: always; 1: on the sampled b1,
// if the sample named one.
template <bool LONG>
__global__ void __launch_bounds__(kThreads, 8)
    topm_split_kernel(const float *__restrict__ scores, int n, RowDiv rd, int current,
                      TopmState *__restrict__ st, uint8_t *__restrict__ keep,
                      int32_t *__restrict__ per_head, uint32_t *__restrict__ cand,
                      uint32_t *__restrict__ ckey, int gate) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  if (gate == 1 && !st->sure) return;
  split_chunk<LONG>(scores, n, rd, current, st->prefix >> kShift1, blockIdx.x * kChunk, st, keep,
              per_head, cand, ckey);
}

// The split pass on the exact b1, only if the sampled one was not confirmed:
// a grid-stride loop over the chunks, so that the usual case (nothing to do)
// costs a small grid.
template <bool LONG>
__global__ void __launch_bounds__(kThreads, 8)
    topm_split_redo_kernel(const float *__restrict__ scores, int n, RowDiv rd, int current,
                           TopmState *__restrict__ st, uint8_t *__restrict__ keep,
                           int32_t *__restrict__ per_head, uint32_t *__restrict__ cand,
                           uint32_t *__restrict__ ckey) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  if (!st->redo) return;
  const uint32_t b1 = st->prefix >> kShift1;
  for (int64_t cbase = static_cast<int64_t>(blockIdx.x) * kChunk; cbase < n;
       cbase += static_cast<int64_t>(gridDim.x) * kChunk) {
    split_chunk<LONG>(scores, n, rd, current, b1, static_cast<int>(cbase), st, keep, per_head, cand,
                ckey);
    __syncthreads();  // the shared counts are reused by the next chunk
  }
}

// Candidate passes.  Each warp takes 32 x kCandPer consecutive entries of the
// candidate list (index and key) per step; every lane runs every step, lanes
// past the end carry no candidate.
// Counts go through warp-aggregated atomics: the lanes that share a target
// (a bin, a chunk, a row) elect one to add their number, which keeps heavily
// tied scores from serializing on one address.
constexpr int kCandPer = 8;

__device__ __forceinline__ void warp_add(uint32_t *addr_base, int slot, bool on, uint32_t n = 1) {
  const unsigned act = __ballot_sync(0xffffffffu, on);
  if (!on) return;
  const unsigned peers = __match_any_sync(act, slot);
  if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(addr_base + slot, n * __popc(peers));
}

template <typename F>
__device__ __forceinline__ void for_candidates(const uint32_t *__restrict__ cand,
                                               const uint32_t *__restrict__ ckey, uint32_t nc,
                                               F &&f) {
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t warps = gridDim.x * (kThreads / 32);
  const uint32_t step = warps * 32 * kCandPer;
  for (uint32_t b0 = (blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * 32 * kCandPer;
       b0 < nc; b0 += step) {
    uint32_t idx[kCandPer], key[kCandPer];
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      const uint32_t i = b0 + u * 32 + lane;
      idx[u] = i < nc ? __ldg(cand + i) : 0xFFFFFFFFu;
      key[u] = i < nc ? __ldg(ckey + i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) f(b0 + u * 32 + lane < nc, idx[u], key[u]);
  }
}

// Histogram of a later digit over the candidates whose decided bits match:
// level 2, bits 10-20 of every candidate; level 3, bits 0-9 of those whose
// top 22 bits match.
template <int LEVEL>
__global__ void __launch_bounds__(kThreads)
    topm_cand_hist_kernel(const uint32_t *__restrict__ cand, const uint32_t *__restrict__ ckey,
                          const TopmState *__restrict__ st, uint32_t *__restrict__ hist) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  constexpr int BINS = LEVEL == 2 ? kBins2 : kBins3;
  __shared__ uint32_t h[BINS];
  for (int i = threadIdx.x; i < BINS; i += kThreads) h[i] = 0;
  __syncthreads();
  const uint32_t nc = st->n_cand, hi = st->prefix >> kShift2;
  for_candidates(cand, ckey, nc, [&](bool valid, uint32_t, uint32_t k) {
    if (LEVEL == 2)
      warp_add(h, static_cast<int>((k >> kShift2) & (kBins2 - 1)), valid);
    else
      warp_add(h, static_cast<int>(k & (kBins3 - 1)), valid && (k >> kShift2) == hi);
  });
  __syncthreads();
  for (int i = threadIdx.x; i < BINS; i += kThreads)
    if (h[i]) atomicAdd(&hist[i], h[i]);
}

// Candidates whose key equals S*, per chunk of kChunk elements of the array.
__global__ void __launch_bounds__(kThreads)
    topm_cand_tie_kernel(const uint32_t *__restrict__ cand, const uint32_t *__restrict__ ckey,
                         const TopmState *__restrict__ st, uint32_t *__restrict__ tiecnt) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  const uint32_t skey = st->prefix;
  for_candidates(cand, ckey, st->n_cand, [&](bool valid, uint32_t idx, uint32_t k) {
    warp_add(tiecnt, static_cast<int>(idx / kChunk), valid && k == skey);
  });
}

// The kept candidates: (key, index) <= (S*, idx*).
__global__ void __launch_bounds__(kThreads)
    topm_cand_keep_kernel(const uint32_t *__restrict__ cand, const uint32_t *__restrict__ ckey,
                          const TopmState *__restrict__ st, RowDiv rd, uint8_t *__restrict__ keep,
                          int32_t *__restrict__ per_head) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  const uint32_t skey = st->prefix, istar = st->idx_star;
  for_candidates(cand, ckey, st->n_cand, [&](bool valid, uint32_t idx, uint32_t k) {
    const bool kept = valid && (k < skey || (k == skey && idx <= istar));
    if (kept) keep[idx] = 1;
    if (per_head)
      warp_add(reinterpret_cast<uint32_t *>(per_head), rd.div(static_cast<int>(idx)), kept);
  });
}

// One CTA of 1024 threads: the last kept candidate.  First the chunk holding
// the k_rem-th tie (candidate with key S*), from an exclusive scan of the
// chunk tie counts (each thread first sums a run); then that tie's index
// idx*, ranking the chunk's ties in index order (four elements a thread).
__global__ void __launch_bounds__(1024)
    topm_tierank_kernel(const uint32_t *__restrict__ tiecnt, int n_chunks,
                        const float *__restrict__ scores, int n, RowDiv rd, int current,
                        TopmState *__restrict__ st) {
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  __shared__ uint32_t s_chunk, s_rank;
  // runs of a multiple of 4 counts, loaded 16 bytes at a time (the counts
  // start 16-byte aligned)
  const int per = ((n_chunks + 1023) / 1024 + 3) & ~3;
  const int lo = threadIdx.x * per, hi = min(n_chunks, lo + per);
  auto quad = [&](int i) {
    if (i + 4 <= hi) return *reinterpret_cast<const uint4 *>(tiecnt + i);
    return make_uint4(i < hi ? tiecnt[i] : 0u, i + 1 < hi ? tiecnt[i + 1] : 0u,
                      i + 2 < hi ? tiecnt[i + 2] : 0u, 0u);
  };
  uint32_t sum = 0;
#pragma unroll 4
  for (int i = lo; i < hi; i += 4) {
    const uint4 v = quad(i);
    sum += v.x + v.y + v.z + v.w;
  }
  const uint32_t r = st->k_rem, skey = st->prefix;
  if (threadIdx.x == 0) s_chunk = s_rank = 0u;  // (rank 0: no index; cannot happen)
  uint32_t run = block_scan_incl<1024>(sum) - sum;
  if (run < r && r <= run + sum) {  // exactly one thread
    for (int i = lo; i < hi; i += 4) {
      const uint4 q = quad(i);
      const uint32_t v[4] = {q.x, q.y, q.z, q.w};
      bool found = false;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (!found && run < r && r <= run + v[u]) {
          s_chunk = st->tie_chunk = static_cast<uint32_t>(i + u);
          s_rank = st->tie_rank = r - run;
          found = true;
        }
        if (!found) run += v[u];
      }
      if (found) break;
    }
  }
  __syncthreads();  // also ends every thread's use of the scan's shared totals
  const uint32_t want = s_rank;
  const int base = static_cast<int>(s_chunk) * kChunk + threadIdx.x * 4;
  uint32_t tie_bits = 0;  // bit e: element base + e is a tie
  int t = base - rd.div(base) * rd.N;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (base + e < n && t != current && score_key(__ldg(scores + base + e)) == skey)
      tie_bits |= 1u << e;
    if (++t == rd.N) t = 0;
  }
  const uint32_t ties = __popc(tie_bits);
  const uint32_t before = block_scan_incl<1024>(ties) - ties;
  if (before < want && want <= before + ties) {  // exactly one thread
    uint32_t bits = tie_bits;
    for (uint32_t k = before + 1; k < want; ++k) bits &= bits - 1;  // drop earlier ties
    st->idx_star = static_cast<uint32_t>(base + __ffs(bits) - 1);
  }
}

// The keep mask when the budget decides it alone.  all = false: only the
// current positions; true: every element.  Kept rows per (layer, head) are
// summed in shared memory, then added once per CTA.
__global__ void __launch_bounds__(kThreads)
    topm_mask_kernel(int n, RowDiv rd, int current, bool all, uint8_t *__restrict__ keep,
                     int32_t *__restrict__ per_head) {
  const int N = rd.N;
  griddep_wait();  // the previous launch of the stream has completed
  griddep_release();
  __shared__ int cnt[kChunk + 2];  // rows of this chunk, relative to its first
  const int cbase = blockIdx.x * kChunk;
  const int row0 = rd.div(cbase);
  const int cend = min(n, cbase + kChunk);
  const int n_rows = rd.div(cend - 1) - row0 + 1;
  if (per_head) {
    for (int i = threadIdx.x; i < n_rows; i += kThreads) cnt[i] = 0;
    __syncthreads();
  }
  const int base = cbase + threadIdx.x * kPerThread;
  int row = rd.div(base);
  int t = base - row * N;
  row -= row0;
  int run_row = -1, run = 0;  // kept count of the current (layer, head) run
  uint32_t bytes[kPerThread / 4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    if (base + e < n) {
      const bool k = all || t == current;
      bytes[e >> 2] |= (k ? 1u : 0u) << (8 * (e & 3));
      if (per_head && k) {
        if (row != run_row) {
          if (run) atomicAdd(&cnt[run_row], run);
          run_row = row;
          run = 0;
        }
        ++run;
      }
    }
    if (++t == N) {
      t = 0;
      ++row;
    }
  }
  if (base + kPerThread <= n) {
    *reinterpret_cast<uint4 *>(keep + base) = make_uint4(bytes[0], bytes[1], bytes[2], bytes[3]);
  } else {
    for (int e = 0; base + e < n; ++e) keep[base + e] = (bytes[e >> 2] >> (8 * (e & 3))) & 1u;
  }
  if (per_head) {
    if (run) atomicAdd(&cnt[run_row], run);
    __syncthreads();
    for (int i = threadIdx.x; i < n_rows; i += kThreads)
      if (cnt[i]) atomicAdd(per_head + row0 + i, cnt[i]);
  }
}

size_t topm_chunks(int64_t n) { return static_cast<size_t>((n + kChunk - 1) / kChunk); }

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

// Workspace: the three histograms, the state, the per-chunk tie counts, then
// the candidate list (an index and a key per element at most), 16-byte
// aligned.
size_t pa_topm_workspace_size(int n_layers, int n_heads, int n_tokens) {
  if (n_layers <= 0 || n_heads <= 0 || n_tokens <= 0) return 0;
  const int64_t n = static_cast<int64_t>(n_layers) * n_heads * n_tokens;
  const size_t head = (kBins1 + kBins2 + kBins3) * sizeof(uint32_t) + sizeof(TopmState) +
                      topm_chunks(n) * sizeof(uint32_t);
  return ((head + 15) & ~size_t(15)) + 2 * static_cast<size_t>(n) * sizeof(uint32_t);
}

int pa_topm_retain(const float *scores, int n_layers, int n_heads, int n_tokens, int current,
                   long long budget, uint8_t *keep, int32_t *kept_per_head, void *workspace,
                   size_t workspace_bytes, pa_stream_t stream) {
  if (!scores || !keep || !workspace) return PA_ERR_NULL;
  if (n_layers <= 0 || n_heads <= 0 || n_tokens <= 0) return PA_ERR_SHAPE;
  const int64_t n = static_cast<int64_t>(n_layers) * n_heads * n_tokens;
  // indices stay 32-bit: the last chunk must end below 2^31
  if (n > (static_cast<int64_t>(1) << 31) - 2 * kChunk || current < 0 || current >= n_tokens)
    return PA_ERR_SHAPE;
  if (budget < 0) return PA_ERR_SHAPE;
  if (workspace_bytes < pa_topm_workspace_size(n_layers, n_heads, n_tokens))
    return PA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(scores) |
       reinterpret_cast<uintptr_t>(keep)) & 15)
    return PA_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t *hist1 = static_cast<uint32_t *>(workspace);
  uint32_t *hist2 = hist1 + kBins1, *hist3 = hist2 + kBins2;
  TopmState *st = reinterpret_cast<TopmState *>(hist3 + kBins3);
  uint32_t *tiecnt = reinterpret_cast<uint32_t *>(st + 1);
  const int n_chunks = static_cast<int>(topm_chunks(n));
  const size_t head = reinterpret_cast<uint8_t *>(tiecnt + n_chunks) -
                      static_cast<uint8_t *>(workspace);
  uint32_t *cand =
      reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + ((head + 15) & ~size_t(15)));
  uint32_t *ckey = cand + n;
  const int64_t n_cand = static_cast<int64_t>(n_layers) * n_heads * (n_tokens - 1);
  const int64_t k = budget - static_cast<int64_t>(n_layers) * n_heads;  // candidates kept
  const int mode = k <= 0 ? 0 : (k >= n_cand ? 1 : 2);
  const int ni = static_cast<int>(n);
  const RowDiv rd = make_rowdiv(n_tokens);
  if (mode != 2) {
    if (kept_per_head &&
        cudaMemsetAsync(kept_per_head, 0, sizeof(int32_t) * n_layers * n_heads, s) != cudaSuccess)
      return PA_ERR_CUDA;
    topm_mask_kernel<<<n_chunks, kThreads, 0, s>>>(ni, rd, current, mode == 1, keep,
                                                   kept_per_head);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int n_zero = kBins1 + kBins2 + kBins3;  // the state follows, set apart
  // Every kernel waits for its predecessor at entry (programmatic dependent
  // launch: only the launch latency overlaps).
  const int grid = n_chunks < sms * 4 ? n_chunks : sms * 4;
  const int cgrid = sms * 4;  // candidate passes: grid-stride over the list
  const dim3 T(kThreads), one(1), T1k(1024);
  const int n_rows = n_layers * n_heads;
  cudaError_t e = launch_pdl(topm_init_kernel, dim3(sms), T, 0, s, hist1, n_zero, tiecnt,
                             n_chunks, kept_per_head, n_rows, st, static_cast<uint32_t>(k));
  int32_t *const no_rows = nullptr;
  const bool long_rows = n_tokens >= kChunk;  // a chunk meets at most two rows
  auto split = long_rows ? topm_split_kernel<true> : topm_split_kernel<false>;
  auto split_redo = long_rows ? topm_split_redo_kernel<true> : topm_split_redo_kernel<false>;
  if (n_chunks >= kSampleStep * 16) {
    // the sampled first digit; the exact one behind it, gated on the counts
    const int n_sampled = (n_chunks + kSampleStep - 1) / kSampleStep;
    const int sgrid = n_sampled < sms * 4 ? n_sampled : sms * 4;
    if (e == cudaSuccess)
      e = launch_pdl(topm_hist1_kernel, dim3(sgrid), T, 0, s, scores, ni, rd, current,
                     hist1, kSampleStep, st, 0);
    if (e == cudaSuccess)
      e = launch_pdl(topm_pick_sample_kernel, one, T1k, 0, s, hist1, st,
                     static_cast<float>(n_cand));
    if (e == cudaSuccess)
      e = launch_pdl(split, dim3(n_chunks), T, 0, s, scores, ni, rd, current,
                     st, keep, kept_per_head, cand, ckey, 1);
    if (e == cudaSuccess)
      e = launch_pdl(topm_hist1_kernel, dim3(grid), T, 0, s, scores, ni, rd, current,
                     hist1, 1, st, 1);
    if (e == cudaSuccess)
      e = launch_pdl(topm_pick_kernel<kBins1>, one, T1k, 0, s, hist1, st, kShift1, 1,
                     kept_per_head, n_rows);
    if (e == cudaSuccess)
      e = launch_pdl(split_redo, dim3(grid), T, 0, s, scores, ni, rd, current,
                     st, keep, kept_per_head, cand, ckey);
  } else {
    if (e == cudaSuccess)
      e = launch_pdl(topm_hist1_kernel, dim3(grid), T, 0, s, scores, ni, rd, current,
                     hist1, 1, st, 0);
    if (e == cudaSuccess)
      e = launch_pdl(topm_pick_kernel<kBins1>, one, T1k, 0, s, hist1, st, kShift1, 0, no_rows,
                     0);
    if (e == cudaSuccess)
      e = launch_pdl(split, dim3(n_chunks), T, 0, s, scores, ni, rd, current,
                     st, keep, kept_per_head, cand, ckey, 0);
  }
  if (e == cudaSuccess)
    e = launch_pdl(topm_cand_hist_kernel<2>, dim3(cgrid), T, 0, s, cand, ckey, st, hist2);
  if (e == cudaSuccess)
    e = launch_pdl(topm_pick_kernel<kBins2>, one, T1k, 0, s, hist2, st, kShift2, 0, no_rows, 0);
  if (e == cudaSuccess)
    e = launch_pdl(topm_cand_hist_kernel<3>, dim3(cgrid), T, 0, s, cand, ckey, st, hist3);
  if (e == cudaSuccess)
    e = launch_pdl(topm_pick_kernel<kBins3>, one, T1k, 0, s, hist3, st, 0, 0, no_rows, 0);
  if (e == cudaSuccess)
    e = launch_pdl(topm_cand_tie_kernel, dim3(cgrid), T, 0, s, cand, ckey, st, tiecnt);
  if (e == cudaSuccess)
    e = launch_pdl(topm_tierank_kernel, one, T1k, 0, s, tiecnt, n_chunks, scores, ni, rd, current,
                   st);
  if (e == cudaSuccess)
    e = launch_pdl(topm_cand_keep_kernel, dim3(cgrid), T, 0, s, cand, ckey, st, rd, keep,
                   kept_per_head);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
