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
// over f (four 8-bit digits, most significant first; each digit one
// histogram pass over the scores plus a one-CTA pick) finds the key S* of the
// K-th candidate and its rank r among the candidates whose key equals S*.
// The kept candidates are then exactly: f < S*, plus the first r with f = S*
// in index order.  The r-th of those is located by counting ties per chunk of
// the array, scanning the counts to find its chunk, and ranking that one
// chunk's ties; with its index idx*, the final pass keeps (f, index) <=
// (S*, idx*) -- a plain comparison per element.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 16;                     // consecutive elements per thread
constexpr int kChunk = kThreads * kPerThread;      // elements per chunk (final passes)

// The state of the select, in the workspace after the histogram.
struct TopmState {
  uint32_t prefix;     // key bits decided so far (S* at the end)
  uint32_t mask;       // which bits are decided
  uint32_t k_rem;      // 1-based rank still to find inside the current bucket
  uint32_t tie_chunk;  // chunk holding the k_rem-th candidate with key S*
  uint32_t tie_rank;   // its 1-based rank among that chunk's ties
  uint32_t idx_star;   // its index: the last kept candidate
  uint32_t pad[2];
};

// Ascending f <=> descending score; -0.0 as 0.0; NaN after every number.
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0xFFFFFFFFu;
  uint32_t u = __float_as_uint(s == 0.f ? 0.f : s);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending order of s
  return ~u;                                        // descending
}

__global__ void __launch_bounds__(kThreads)
    topm_init_kernel(uint32_t *__restrict__ hist, TopmState *__restrict__ st, uint32_t k) {
  hist[threadIdx.x] = 0;
  if (threadIdx.x == 0) *st = TopmState{0u, 0u, k, 0u, 0u, 0u, {0u, 0u}};
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

// Histogram of digit (key >> shift) & 255 over the candidates whose decided
// bits match the prefix.  Each warp counts into its own shared histogram.
__global__ void __launch_bounds__(kThreads)
    topm_hist_kernel(const float *__restrict__ scores, int n, int N, int current,
                     uint32_t *__restrict__ hist, const TopmState *__restrict__ st,
                     int shift) {
  constexpr int NW = kThreads / 32;
  __shared__ uint32_t h[NW][256];
  for (int i = threadIdx.x; i < NW * 256; i += kThreads) h[i / 256][i % 256] = 0;
  __syncthreads();
  const uint32_t prefix = st->prefix, mask = st->mask;
  const int warp = threadIdx.x >> 5;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kChunk;
  for (int64_t cbase = static_cast<int64_t>(blockIdx.x) * kChunk; cbase < n; cbase += stride) {
    const int base = static_cast<int>(cbase) + threadIdx.x * kPerThread;
    float sc[kPerThread];
    load_run(scores, n, base, sc);
    int t = static_cast<int>(static_cast<unsigned>(base) % static_cast<unsigned>(N));
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      uint32_t bin = 256u;  // none
      if (base + e < n && t != current) {
        const uint32_t k = score_key(sc[e]);
        if ((k & mask) == prefix) bin = (k >> shift) & 255u;
      }
      if (bin != 256u) atomicAdd(&h[warp][bin], 1u);
      if (++t == N) t = 0;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += kThreads) {
    uint32_t v = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) v += h[w][i];
    if (v) atomicAdd(&hist[i], v);
  }
}

// One CTA: the bucket holding the k_rem-th key; clears the histogram.
__global__ void __launch_bounds__(kThreads)
    topm_pick_kernel(uint32_t *__restrict__ hist, TopmState *__restrict__ st, int shift) {
  __shared__ uint32_t c[256];
  const int t = threadIdx.x;
  c[t] = hist[t];
  __syncthreads();
  // inclusive scan (Hillis-Steele) over the 256 bins
  for (int o = 1; o < 256; o <<= 1) {
    const uint32_t v = t >= o ? c[t - o] : 0u;
    __syncthreads();
    c[t] += v;
    __syncthreads();
  }
  const uint32_t k = st->k_rem;
  const uint32_t before = t > 0 ? c[t - 1] : 0u;
  if (before < k && k <= c[t]) {  // exactly one bin
    st->k_rem = k - before;
    st->prefix |= static_cast<uint32_t>(t) << shift;
    st->mask |= 0xFFu << shift;
  }
  hist[t] = 0;
}

// Candidates whose key equals S*, per chunk of kChunk elements.
__global__ void __launch_bounds__(kThreads)
    topm_tiecount_kernel(const float *__restrict__ scores, int n, int N, int current,
                         const TopmState *__restrict__ st, uint32_t *__restrict__ tiecnt) {
  const uint32_t skey = st->prefix;
  const int base = blockIdx.x * kChunk + threadIdx.x * kPerThread;
  float sc[kPerThread];
  load_run(scores, n, base, sc);
  int t = static_cast<int>(static_cast<unsigned>(base) % static_cast<unsigned>(N));
  uint32_t cnt = 0;
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    cnt += base + e < n && t != current && score_key(sc[e]) == skey;
    if (++t == N) t = 0;
  }
  __shared__ uint32_t red[kThreads / 32];
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t s = 0;
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
    tiecnt[blockIdx.x] = s;
  }
}

// One CTA of 1024 threads: the chunk holding the k_rem-th tie, from an
// exclusive scan of the chunk tie counts (each thread first sums a run).
__global__ void __launch_bounds__(1024)
    topm_scan_kernel(const uint32_t *__restrict__ tiecnt, int n_chunks,
                     TopmState *__restrict__ st) {
  __shared__ uint32_t c[1024];
  const int per = (n_chunks + 1023) / 1024;
  const int lo = threadIdx.x * per, hi = min(n_chunks, lo + per);
  uint32_t sum = 0;
  for (int i = lo; i < hi; ++i) sum += tiecnt[i];
  c[threadIdx.x] = sum;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const uint32_t u = threadIdx.x >= o ? c[threadIdx.x - o] : 0u;
    __syncthreads();
    c[threadIdx.x] += u;
    __syncthreads();
  }
  const uint32_t r = st->k_rem;
  uint32_t run = c[threadIdx.x] - sum;
  if (run < r && r <= run + sum) {  // exactly one thread
    for (int i = lo; i < hi; ++i) {
      const uint32_t v = tiecnt[i];
      if (run < r && r <= run + v) {
        st->tie_chunk = static_cast<uint32_t>(i);
        st->tie_rank = r - run;
        break;
      }
      run += v;
    }
  }
}

// One CTA: the index of the tie_rank-th candidate with key S* inside chunk
// tie_chunk (index order).
__global__ void __launch_bounds__(kThreads)
    topm_tiefind_kernel(const float *__restrict__ scores, int n, int N, int current,
                        TopmState *__restrict__ st) {
  const uint32_t skey = st->prefix, want = st->tie_rank;
  const int base = static_cast<int>(st->tie_chunk) * kChunk + threadIdx.x * kPerThread;
  float sc[kPerThread];
  load_run(scores, n, base, sc);
  int t = static_cast<int>(static_cast<unsigned>(base) % static_cast<unsigned>(N));
  uint32_t tie_bits = 0;  // bit e: element base + e is a tie
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    if (base + e < n && t != current && score_key(sc[e]) == skey) tie_bits |= 1u << e;
    if (++t == N) t = 0;
  }
  const uint32_t ties = __popc(tie_bits);
  __shared__ uint32_t c[kThreads];
  c[threadIdx.x] = ties;
  __syncthreads();
  for (int o = 1; o < kThreads; o <<= 1) {
    const uint32_t u = threadIdx.x >= o ? c[threadIdx.x - o] : 0u;
    __syncthreads();
    c[threadIdx.x] += u;
    __syncthreads();
  }
  const uint32_t before = c[threadIdx.x] - ties;
  if (before < want && want <= before + ties) {  // exactly one thread
    uint32_t bits = tie_bits;
    for (uint32_t k = before + 1; k < want; ++k) bits &= bits - 1;  // drop earlier ties
    st->idx_star = static_cast<uint32_t>(base + __ffs(bits) - 1);
  }
}

// The keep mask.  mode 0: only the current positions; 1: every element;
// 2: candidates with (key, index) <= (S*, idx*).  Kept rows per (layer,
// head) are summed in shared memory, then added once per CTA.
__global__ void __launch_bounds__(kThreads)
    topm_mask_kernel(const float *__restrict__ scores, int n, int N, int current,
                     const TopmState *__restrict__ st, int mode, uint8_t *__restrict__ keep,
                     int32_t *__restrict__ per_head) {
  __shared__ int cnt[kChunk + 2];  // rows of this chunk, relative to its first
  const uint32_t skey = st->prefix, istar = st->idx_star;
  const int cbase = blockIdx.x * kChunk;
  const int row0 = static_cast<int>(static_cast<unsigned>(cbase) / static_cast<unsigned>(N));
  const int cend = min(n, cbase + kChunk);
  const int n_rows =
      static_cast<int>(static_cast<unsigned>(cend - 1) / static_cast<unsigned>(N)) - row0 + 1;
  if (per_head) {
    for (int i = threadIdx.x; i < n_rows; i += kThreads) cnt[i] = 0;
    __syncthreads();
  }
  const int base = cbase + threadIdx.x * kPerThread;
  float sc[kPerThread];
  load_run(scores, n, base, sc);
  int t = static_cast<int>(static_cast<unsigned>(base) % static_cast<unsigned>(N));
  int row = static_cast<int>(static_cast<unsigned>(base) / static_cast<unsigned>(N)) - row0;
  int run_row = -1, run = 0;  // kept count of the current (layer, head) run
  uint32_t bytes[kPerThread / 4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    if (base + e < n) {
      const uint32_t key = score_key(sc[e]);
      const bool k = t == current || mode == 1 ||
                     (mode == 2 && (key < skey ||
                                    (key == skey && static_cast<uint32_t>(base + e) <= istar)));
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

size_t pa_topm_workspace_size(int n_layers, int n_heads, int n_tokens) {
  if (n_layers <= 0 || n_heads <= 0 || n_tokens <= 0) return 0;
  const int64_t n = static_cast<int64_t>(n_layers) * n_heads * n_tokens;
  return 256 * sizeof(uint32_t) + sizeof(TopmState) + topm_chunks(n) * sizeof(uint32_t);
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
  uint32_t *hist = static_cast<uint32_t *>(workspace);
  TopmState *st = reinterpret_cast<TopmState *>(hist + 256);
  uint32_t *tiecnt = reinterpret_cast<uint32_t *>(st + 1);
  const int n_chunks = static_cast<int>(topm_chunks(n));
  const int64_t n_cand = static_cast<int64_t>(n_layers) * n_heads * (n_tokens - 1);
  const int64_t k = budget - static_cast<int64_t>(n_layers) * n_heads;  // candidates kept
  const int mode = k <= 0 ? 0 : (k >= n_cand ? 1 : 2);
  if (kept_per_head &&
      cudaMemsetAsync(kept_per_head, 0, sizeof(int32_t) * n_layers * n_heads, s) != cudaSuccess)
    return PA_ERR_CUDA;
  topm_init_kernel<<<1, 256, 0, s>>>(hist, st, mode == 2 ? static_cast<uint32_t>(k) : 0u);
  if (mode == 2) {
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = n_chunks < sms * 4 ? n_chunks : sms * 4;
    const int ni = static_cast<int>(n);
    for (int d = 0; d < 4; ++d) {
      const int shift = 24 - 8 * d;
      topm_hist_kernel<<<grid, kThreads, 0, s>>>(scores, ni, n_tokens, current, hist, st,
                                                 shift);
      topm_pick_kernel<<<1, kThreads, 0, s>>>(hist, st, shift);
    }
    topm_tiecount_kernel<<<n_chunks, kThreads, 0, s>>>(scores, ni, n_tokens, current, st,
                                                       tiecnt);
    topm_scan_kernel<<<1, 1024, 0, s>>>(tiecnt, n_chunks, st);
    topm_tiefind_kernel<<<1, kThreads, 0, s>>>(scores, ni, n_tokens, current, st);
  }
  topm_mask_kernel<<<n_chunks, kThreads, 0, s>>>(scores, static_cast<int>(n), n_tokens,
                                                 current, st, mode, keep, kept_per_head);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
