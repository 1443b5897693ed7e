// pa_decode.cu -- decode-step paged GQA attention for sm_103a (CUDA cores).
//
// Computes, per sequence b and query head h, o = softmax(q K^T * scale) V
// over the sequence's cached tokens (ch. 19 "推理系统与性能工程", 19.4.1),
// evaluated page by page with the online-softmax recurrence of 19.6.2
// (running max m, running sum l, unnormalised O).
//
// Work decomposition.  One CTA handles one (sequence, kv head, head tile,
// partition): the GT query heads of a head tile share every K/V page it reads
// (GQA reuse, "吞吐与延迟的系统模型" section 5: the kernel must reuse the shared
// KV for the low-byte bound to hold).  Its NW warps take the partition's
// pages round robin.  Each warp feeds itself: it keeps S pages in flight in
// its own ring of shared-memory stages, filled by 2-D TMA loads (128-byte
// swizzle) that complete on one mbarrier per stage, and issues the load for
// page i+S as soon as page i has been consumed.  No warp waits for another
// until the partition's end, where the warps' (m, l, O) states are merged in
// shared memory with the exponent law of 19.6.2.
//
// Score phase: lane = (token, half of head_dim).  The swizzled tile lets the
// 16 lanes of a half-warp read 16 different K rows without bank conflicts
// while all of them read the same q element (a broadcast).
// Value phase: lane = head_dim / 32 output dims; every lane reads the same V
// row.  Both phases use packed fp32x2 FMAs; K/V elements are unpacked from
// bf16/fp16 once per page and reused by all GT heads.
//
// Scores are kept in log2 units (q is pre-multiplied by scale * log2 e), so
// e^(s - m) is one ex2.  The running max is only moved when a score exceeds it
// by more than kRescaleSlack (a warp vote decides); between moves the
// weights e^(s - m) stay <= 2^kRescaleSlack.  The rescale is exact whatever
// reference max is used, because O and l share it (19.6.2's argument).
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.0f;
constexpr unsigned kFull = 0xffffffffu;

struct DecodeParams {
  const uint16_t *q;
  const int32_t *block_table;
  const int32_t *ctx_lens;
  float *out;
  float *ws;
  int *status;
  float qscale;  // scale * log2(e)
  int n_q_heads, n_kv_heads, group, batch, max_blocks, num_pages;
  int part_pages, n_parts;
};

// Shared-memory plan of one CTA.
template <int D, int GT, int NW, int S>
struct DecodeSmem {
  static constexpr int kBoxBytes = 16 * 128;  // one TMA box: 16 rows x 64 elems
  static constexpr int kBoxes = D / 64;
  static constexpr int kPageBytes = kBoxes * kBoxBytes;  // K (or V) of one page
  static constexpr int kStageBytes = 2 * kPageBytes;     // K tile then V tile
  static constexpr int kStages = NW * S;
  static constexpr int kQStride = D + 8;  // floats per q row; 2nd half +4
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kPOff = kQOff + GT * kQStride * 4;
  static constexpr int kBarOff = kPOff + NW * GT * 16 * 4;
  static constexpr int kBytes = kBarOff + kStages * 8;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-B alignment
  static constexpr int kMergeFloats = NW * GT * (D + 2);
  static_assert(kMergeFloats * 4 <= kQOff, "merge area must fit in the stages");
  static_assert(kStageBytes % 1024 == 0, "swizzled boxes need 1024-B alignment");
};

template <int D, int GT, bool BF16, int NW, int S>
__global__ void __launch_bounds__(NW * 32)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  using L = DecodeSmem<D, GT, NW, S>;
  constexpr int DPL = D / 32;   // output dims per lane
  constexpr int HALF = D / 2;   // dims per half-warp in the score phase
  constexpr int CPH = HALF / 8; // 16-byte chunks per half row

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  float *q_s = reinterpret_cast<float *>(smem + L::kQOff);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int part = blockIdx.x;
  const int n_sub = p.group / GT;
  const int g = blockIdx.y / n_sub;
  const int h0 = g * p.group + (blockIdx.y % n_sub) * GT;
  const int b = blockIdx.z;

  int T = p.ctx_lens[b];
  const int maxT = p.max_blocks * 16;
  if (T < 0 || T > maxT) {
    if (tid == 0) record_error(p.status, PA_ERR_BAD_CTX);
    T = T < 0 ? 0 : maxT;
  }
  const int n_pages = (T + 15) >> 4;
  int pg0 = 0, pg1 = n_pages;
  if (p.part_pages > 0) {
    pg0 = part * p.part_pages;
    pg1 = min(n_pages, pg0 + p.part_pages);
  }
  if (pg0 >= pg1) {
    // Nothing to read.  A single pass owes zeros; with partitions the merge
    // kernel never reads a partition past the sequence's end.
    if (p.n_parts == 1)
      for (int i = tid; i < GT * D; i += NW * 32)
        p.out[(static_cast<size_t>(b) * p.n_q_heads + h0) * D + i] = 0.f;
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < L::kStages; ++s) mbar_init(sbase + L::kBarOff + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- this warp's pages: logical blocks first, first+NW, first+2NW, ...
  const int first = pg0 + warp;
  const int n_i = first < pg1 ? (pg1 - first + NW - 1) / NW : 0;
  const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  auto fetch_id = [&](int i) -> int {
    if (i >= n_i) return 0;
    int id = __ldg(bt_row + first + NW * i);
    if (static_cast<unsigned>(id) >= static_cast<unsigned>(p.num_pages)) {
      record_error(p.status, PA_ERR_BAD_BLOCK);
      id = 0;  // read a page that exists; the result is flagged as invalid
    }
    return id;
  };
  // Lane j holds the page of chunk 32k + j; the next 32 are fetched early.
  int ids_cur = fetch_id(lane);
  int ids_nxt = fetch_id(32 + lane);
  const uint32_t stage0 = sbase + warp * S * L::kStageBytes;
  const uint32_t bar0 = sbase + L::kBarOff + warp * S * 8;
  const int rows_per_page = p.n_kv_heads * 16;

  auto issue = [&](int i) {  // called by the whole warp, i = 0, 1, 2, ...
    if ((i & 31) == 0 && i > 0) {
      ids_cur = ids_nxt;
      ids_nxt = fetch_id(i + 32 + lane);
    }
    const int id = __shfl_sync(kFull, ids_cur, i & 31);
    if (lane == 0) {
      const int s = i % S;
      const uint32_t st = stage0 + s * L::kStageBytes, bar = bar0 + 8 * s;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, L::kStageBytes);
      const int y = id * rows_per_page + g * 16;
#pragma unroll
      for (int bx = 0; bx < L::kBoxes; ++bx) {
        tma_load_2d(st + bx * L::kBoxBytes, &kmap, bx * 64, y, bar);
        tma_load_2d(st + L::kPageBytes + bx * L::kBoxBytes, &vmap, bx * 64, y, bar);
      }
    }
  };

  for (int i = 0; i < S && i < n_i; ++i) issue(i);

  // ---- q of the head tile -> shared memory as fp32 * scale * log2(e)
  {
    const uint16_t *qg = p.q + (static_cast<size_t>(b) * p.n_q_heads + h0) * D;
    for (int e = tid * 8; e < GT * D; e += NW * 32 * 8) {
      const uint4 v = *reinterpret_cast<const uint4 *>(qg + e);
      const int h = e / D, d = e % D;
      float *dst = q_s + h * L::kQStride + d + (d >= HALF ? 4 : 0);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = unpack2<BF16>(w[k]);
        dst[2 * k] = f.x * p.qscale;
        dst[2 * k + 1] = f.y * p.qscale;
      }
    }
  }
  __syncthreads();

  float m[GT], lsum[GT];
  float2 O2[GT][DPL / 2];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    m[h] = -INFINITY;
    lsum[h] = 0.f;
#pragma unroll
    for (int k = 0; k < DPL / 2; ++k) O2[h][k] = make_float2(0.f, 0.f);
  }
  float *p_s = reinterpret_cast<float *>(smem + L::kPOff) + warp * GT * 16;
  const int tok = lane & 15, hf = lane >> 4;
  // score phase: this lane's K row inside a stage
  const uint32_t k_off = (D == 128 ? hf * L::kBoxBytes : 0) + tok * 128;
  // value phase: this lane's dims inside a V row, before the swizzle
  const uint32_t v_off = L::kPageBytes +
                         (D == 128 ? (lane >> 4) * L::kBoxBytes + ((lane & 1) << 3)
                                   : ((lane & 3) << 2));
  const int v_chunk = (D == 128) ? ((lane & 15) >> 1) : (lane >> 2);

  for (int i = 0; i < n_i; ++i) {
    const int s = i % S;
    const uint32_t st = stage0 + s * L::kStageBytes;
    // The verdict is made warp-uniform so that no lane leaves the loop alone.
    if (!__all_sync(kFull, mbar_wait(bar0 + 8 * s, (i / S) & 1))) {
      if (lane == 0) record_error(p.status, PA_ERR_TIMEOUT);
      // Let the other copies this warp has in flight land before leaving.
      for (int j = i + 1; j < n_i && j < i + S; ++j)
        mbar_wait(bar0 + 8 * (j % S), (j / S) & 1);
      break;
    }
    const int t0 = (first + NW * i) * 16;
    const int valid = min(16, T - t0);

    // -- scores s_h(tok) = <q_h, k_tok>, already * scale * log2 e
    float sc[GT];
    {
      float2 acc[GT];
#pragma unroll
      for (int h = 0; h < GT; ++h) acc[h] = make_float2(0.f, 0.f);
      const uint32_t krow = st + k_off;
#pragma unroll
      for (int j = 0; j < CPH; ++j) {
        const int c = (D == 128) ? j : hf * CPH + j;
        const uint4 kv = lds128(krow + ((c ^ (tok & 7)) << 4));
        const float2 k01 = unpack2<BF16>(kv.x), k23 = unpack2<BF16>(kv.y);
        const float2 k45 = unpack2<BF16>(kv.z), k67 = unpack2<BF16>(kv.w);
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          const float *qh = q_s + h * L::kQStride + hf * (HALF + 4) + j * 8;
          const float4 qa = *reinterpret_cast<const float4 *>(qh);
          const float4 qb = *reinterpret_cast<const float4 *>(qh + 4);
          acc[h] = __ffma2_rn(make_float2(qa.x, qa.y), k01, acc[h]);
          acc[h] = __ffma2_rn(make_float2(qa.z, qa.w), k23, acc[h]);
          acc[h] = __ffma2_rn(make_float2(qb.x, qb.y), k45, acc[h]);
          acc[h] = __ffma2_rn(make_float2(qb.z, qb.w), k67, acc[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        float v = acc[h].x + acc[h].y;
        v += __shfl_xor_sync(kFull, v, 16);
        sc[h] = (tok < valid) ? v : -INFINITY;
      }
    }

    // -- online softmax: move the reference max only when needed
    bool need = false;
#pragma unroll
    for (int h = 0; h < GT; ++h) need |= sc[h] > m[h] + kRescaleSlack;
    if (__any_sync(kFull, need)) {
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        float mt = sc[h];
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
        const float mn = fmaxf(m[h], mt);
        const float c = ex2(m[h] - mn);  // 0 on the first page (m = -inf)
        m[h] = mn;
        lsum[h] *= c;
#pragma unroll
        for (int k = 0; k < DPL / 2; ++k)
          O2[h][k] = make_float2(O2[h][k].x * c, O2[h][k].y * c);
      }
    }
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      const float pr = ex2(sc[h] - m[h]);
      lsum[h] += pr;
      if (hf == 0) p_s[h * 16 + tok] = pr;
    }
    __syncwarp();

    // -- O_h += sum_t p_h(t) v_t over the page's valid tokens
    const uint32_t vrow = st + v_off;
    auto pv = [&](int t, const float (&pw)[GT]) {
      const uint32_t addr = vrow + t * 128 + ((v_chunk ^ (t & 7)) << 4);
      if constexpr (D == 128) {
        const uint2 vv = lds64(addr);
        const float2 v01 = unpack2<BF16>(vv.x), v23 = unpack2<BF16>(vv.y);
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          const float2 w2 = make_float2(pw[h], pw[h]);
          O2[h][0] = __ffma2_rn(w2, v01, O2[h][0]);
          O2[h][1] = __ffma2_rn(w2, v23, O2[h][1]);
        }
      } else {
        const float2 v01 = unpack2<BF16>(lds32(addr));
#pragma unroll
        for (int h = 0; h < GT; ++h)
          O2[h][0] = __ffma2_rn(make_float2(pw[h], pw[h]), v01, O2[h][0]);
      }
    };
    if (valid == 16) {
#pragma unroll
      for (int t4 = 0; t4 < 16; t4 += 4) {
        float4 pp[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h)
          pp[h] = *reinterpret_cast<const float4 *>(p_s + h * 16 + t4);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float pw[GT];
#pragma unroll
          for (int h = 0; h < GT; ++h)
            pw[h] = u == 0 ? pp[h].x : u == 1 ? pp[h].y : u == 2 ? pp[h].z : pp[h].w;
          pv(t4 + u, pw);
        }
      }
    } else {
      for (int t = 0; t < valid; ++t) {
        float pw[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) pw[h] = p_s[h * 16 + t];
        pv(t, pw);
      }
    }
    __syncwarp();
    if (i + S < n_i) issue(i + S);
  }

  // ---- l: each token was counted by one lane of each half-warp
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    float v = lsum[h];
    v += __shfl_xor_sync(kFull, v, 8);
    v += __shfl_xor_sync(kFull, v, 4);
    v += __shfl_xor_sync(kFull, v, 2);
    v += __shfl_xor_sync(kFull, v, 1);
    lsum[h] = v;
  }

  // ---- merge the NW warp states (the stages are free once all warps are here)
  __syncthreads();
  float *mer_m = reinterpret_cast<float *>(smem);
  float *mer_l = mer_m + NW * GT;
  float *mer_o = mer_l + NW * GT;
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      mer_m[warp * GT + h] = m[h];
      mer_l[warp * GT + h] = lsum[h];
    }
  }
#pragma unroll
  for (int h = 0; h < GT; ++h)
#pragma unroll
    for (int k = 0; k < DPL / 2; ++k)
      *reinterpret_cast<float2 *>(mer_o + (warp * GT + h) * D + lane * DPL + 2 * k) =
          O2[h][k];
  __syncthreads();

  for (int e = tid; e < GT * D; e += NW * 32) {
    const int h = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mer_m[w * GT + h]);
    float lt = 0.f, o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = ex2(mer_m[w * GT + h] - M);
        lt += f * mer_l[w * GT + h];
        o += f * mer_o[(w * GT + h) * D + d];
      }
    }
    const size_t row = static_cast<size_t>(b) * p.n_q_heads + h0 + h;
    if (p.n_parts == 1) {
      p.out[row * D + d] = lt > 0.f ? o / lt : 0.f;
    } else {
      float *dst = p.ws + (row * p.n_parts + part) * (D + 2);
      dst[d] = o;
      if (d == 0) {
        dst[D] = M * kLn2;  // natural-log units
        dst[D + 1] = lt;
      }
    }
  }
}

// ---- exact merge of partition states: one CTA of head_dim threads per row
template <int D>
__global__ void __launch_bounds__(D)
    merge_kernel(const float *__restrict__ parts, const int32_t *__restrict__ ctx,
                 float *__restrict__ out, int *status, int n_q_heads,
                 int n_parts, int part_tokens) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  long T = ctx[b];
  if (T < 0) {
    if (d == 0 && h == 0) record_error(status, PA_ERR_BAD_CTX);
    T = 0;
  }
  int n_valid = static_cast<int>((T + part_tokens - 1) / part_tokens);
  if (n_valid > n_parts) {
    if (d == 0 && h == 0) record_error(status, PA_ERR_BAD_CTX);
    n_valid = n_parts;
  }
  const size_t row = static_cast<size_t>(b) * n_q_heads + h;
  const float *src = parts + row * n_parts * (D + 2);
  float M = -INFINITY;
  for (int q = 0; q < n_valid; ++q) {
    const float *sp = src + q * (D + 2);
    if (sp[D + 1] > 0.f) M = fmaxf(M, sp[D]);
  }
  float lt = 0.f, o = 0.f;
  if (M != -INFINITY) {
    for (int q = 0; q < n_valid; ++q) {
      const float *sp = src + q * (D + 2);
      const float l = sp[D + 1];
      if (!(l > 0.f)) continue;
      const float f = ex2((sp[D] - M) * kLog2e);
      lt += f * l;
      o += f * sp[d];
    }
  }
  out[row * D + d] = lt > 0.f ? o / lt : 0.f;
}

// Stages per warp: keep about 24 KiB of K/V per warp in flight.
template <int D>
constexpr int stages_per_warp() { return D == 128 ? 3 : 6; }
constexpr int kDecodeWarps = 4;

template <int D, int GT, bool BF16>
int launch_decode_t(const DecodeLaunch &a, cudaStream_t stream) {
  constexpr int NW = kDecodeWarps, S = stages_per_warp<D>();
  using L = DecodeSmem<D, GT, NW, S>;
  auto kern = decode_kernel<D, GT, BF16, NW, S>;
  static uint64_t attr_set = 0;  // one bit per device ordinal
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return PA_ERR_CUDA;
  if (!(attr_set >> dev & 1)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAlloc) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_set |= uint64_t(1) << dev;
  }
  CUtensorMap kmap, vmap;
  const uint64_t rows = static_cast<uint64_t>(a.num_pages) * a.n_kv_heads * 16;
  if (make_rows_map(&kmap, a.k_cache, rows, D, 16) != PA_OK) return PA_ERR_CUDA;
  if (make_rows_map(&vmap, a.v_cache, rows, D, 16) != PA_OK) return PA_ERR_CUDA;
  DecodeParams p;
  p.q = static_cast<const uint16_t *>(a.q);
  p.block_table = a.block_table;
  p.ctx_lens = a.ctx_lens;
  p.out = a.out;
  p.ws = a.workspace;
  p.status = a.status;
  p.qscale = a.scale * kLog2e;
  p.n_q_heads = a.n_q_heads;
  p.n_kv_heads = a.n_kv_heads;
  p.group = a.n_q_heads / a.n_kv_heads;
  p.batch = a.batch;
  p.max_blocks = a.max_blocks;
  p.num_pages = a.num_pages;
  p.part_pages = a.part_pages;
  p.n_parts = a.n_parts;
  const dim3 grid(a.n_parts, a.n_kv_heads * (p.group / GT), a.batch);
  kern<<<grid, NW * 32, L::kAlloc, stream>>>(kmap, vmap, p);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  if (a.n_parts > 1) {
    const dim3 mgrid(a.n_q_heads, a.batch);
    merge_kernel<D><<<mgrid, D, 0, stream>>>(a.workspace, a.ctx_lens, a.out,
                                             a.status, a.n_q_heads, a.n_parts,
                                             a.part_pages * 16);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

template <int D, bool BF16>
int launch_decode_d(const DecodeLaunch &a, cudaStream_t stream) {
  switch (group_tile(a.n_q_heads / a.n_kv_heads)) {
    case 8: return launch_decode_t<D, 8, BF16>(a, stream);
    case 4: return launch_decode_t<D, 4, BF16>(a, stream);
    case 2: return launch_decode_t<D, 2, BF16>(a, stream);
    default: return launch_decode_t<D, 1, BF16>(a, stream);
  }
}

}  // namespace

int launch_decode(const DecodeLaunch &a, cudaStream_t stream) {
  if (a.head_dim == 128)
    return a.bf16 ? launch_decode_d<128, true>(a, stream)
                  : launch_decode_d<128, false>(a, stream);
  return a.bf16 ? launch_decode_d<64, true>(a, stream)
                : launch_decode_d<64, false>(a, stream);
}

int launch_merge(const float *partials, const int32_t *ctx_lens, float *out,
                 int *status, int batch, int n_q_heads, int head_dim,
                 int n_parts, int partition_tokens, cudaStream_t stream) {
  const dim3 grid(n_q_heads, batch);
  if (head_dim == 128)
    merge_kernel<128><<<grid, 128, 0, stream>>>(partials, ctx_lens, out, status,
                                                n_q_heads, n_parts,
                                                partition_tokens);
  else
    merge_kernel<64><<<grid, 64, 0, stream>>>(partials, ctx_lens, out, status,
                                              n_q_heads, n_parts,
                                              partition_tokens);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
