// pa_prefill.cu -- chunked-prefill paged attention (multi-query, causal).
//
// Query i of sequence b (0 <= i < n_new) attends keys 0 .. ctx_lens[b] + i:
// the cached context plus the chunk's own keys up to itself (ch. 19
// "推理系统与性能工程", 19.3.1 prefill; 19.6.3 FlashAttention forward: Q tile
// resident, K/V tiles streamed, running m, l, O, one write of O / l).
//
// Tile plan.  A CTA owns 64 rows = (query, head) pairs of one kv head's GQA
// group: GT heads x 64/GT consecutive queries, so every K/V tile it streams
// serves all GT heads (the group shares the KV, "吞吐与延迟的系统模型" 5).
// K/V tiles are 64 keys = 4 pages, loaded by 2-D TMA (128-byte swizzle) into
// a 2-stage ring; each 16-key slice of a tile is exactly one page.  Four warps
// each own 16 rows.  S = Q K^T and O += P V run on the tensor cores with
// warp-level mma.sync m16n8k16 (bf16/fp16 in, fp32 accumulate), operands
// fetched with ldmatrix from the swizzled tiles; the online softmax runs on
// the accumulator fragments in registers.  P enters P V as two 16-bit terms
// (head + remainder), so the weights keep about 16 significant bits.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

struct PrefillParams {
  const uint16_t *q;
  const int32_t *block_table;
  const int32_t *ctx_lens;
  float *out;
  int *status;
  float qscale;  // scale * log2 e
  int n_new, n_q_heads, n_kv_heads, group, batch, max_blocks, num_pages;
};

template <int D>
struct PrefillSmem {
  static constexpr int kRows = 64;                 // (query, head) rows per CTA
  static constexpr int kKeys = 64;                 // keys per K/V tile (4 pages)
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = 16 * 128;       // one page x 64 dims
  static constexpr int kTileBytes = 4 * kBoxes * kBoxBytes;  // K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = 2;
  static constexpr int kQBoxBytes = kRows * 128;   // 64 rows x 64 dims
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kBarOff = kQOff + kBoxes * kQBoxBytes;
  static constexpr int kBytes = kBarOff + kStages * 8;
  static constexpr int kAlloc = kBytes + 1024;
};

template <int D, int GT, bool BF16>
__global__ void __launch_bounds__(128)
    prefill_mma_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap,
                       const PrefillParams p) {
  using L = PrefillSmem<D>;
  constexpr int BQ = L::kRows / GT;  // queries per CTA
  constexpr int NT = D / 8;          // n-tiles of the output
  constexpr int KS = D / 16;         // k-steps of S = Q K^T

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t qs = sbase + L::kQOff;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int q0 = blockIdx.x * BQ;
  const int n_sub = p.group / GT;
  const int g = blockIdx.y / n_sub;
  const int hbase = g * p.group + (blockIdx.y % n_sub) * GT;
  const int b = blockIdx.z;
  const int nq = min(BQ, p.n_new - q0);  // real queries in this tile

  int ctx = p.ctx_lens[b];
  const int maxT = p.max_blocks * 16;
  if (ctx < 0 || ctx + p.n_new > maxT) {
    if (tid == 0) record_error(p.status, PA_ERR_BAD_CTX);
    ctx = max(0, min(ctx, maxT - p.n_new));
  }
  const int total = ctx + p.n_new;           // tokens held by the sequence
  const int kmax = ctx + q0 + nq - 1;        // last key any row of this CTA sees
  const int n_tiles = kmax / L::kKeys + 1;
  const int n_pages = (total + 15) >> 4;

  if (tid == 0) {
    for (int s = 0; s < L::kStages; ++s) mbar_init(sbase + L::kBarOff + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Warp 0 issues the tile loads; lane j keeps the page ids of pages 32k + j.
  const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  auto fetch_id = [&](int pg) -> int {
    if (pg >= n_pages) return 0;  // past the sequence: masked, any page will do
    int id = __ldg(bt_row + pg);
    if (static_cast<unsigned>(id) >= static_cast<unsigned>(p.num_pages)) {
      record_error(p.status, PA_ERR_BAD_BLOCK);
      id = 0;
    }
    return id;
  };
  int ids_cur = 0, ids_nxt = 0, ids_base = -32;
  const int rows_per_page = p.n_kv_heads * 16;
  auto issue = [&](int t) {  // warp 0 only, t = 0, 1, 2, ...
    const int pg0 = t * 4;
    if (pg0 >= ids_base + 32) {  // pages advance by 4 per tile: rotate
      if (ids_base < 0) {
        ids_cur = fetch_id(lane);
        ids_nxt = fetch_id(32 + lane);
        ids_base = 0;
      } else {
        ids_cur = ids_nxt;
        ids_base += 32;
        ids_nxt = fetch_id(ids_base + 32 + lane);
      }
    }
    int ids[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) ids[j] = __shfl_sync(kFull, ids_cur, (pg0 + j) & 31);
    if (lane == 0) {
      const int s = t % L::kStages;
      const uint32_t st = sbase + s * L::kStageBytes, bar = sbase + L::kBarOff + 8 * s;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, L::kStageBytes);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int y = ids[j] * rows_per_page + g * 16;
#pragma unroll
        for (int bx = 0; bx < L::kBoxes; ++bx) {
          const uint32_t off = (j * L::kBoxes + bx) * L::kBoxBytes;
          tma_load_2d(st + off, &kmap, bx * 64, y, bar);
          tma_load_2d(st + L::kTileBytes + off, &vmap, bx * 64, y, bar);
        }
      }
    }
  };
  if (warp == 0) {
    issue(0);
    if (n_tiles > 1) issue(1);
  }

  // ---- Q tile -> shared memory (row r = query r / GT, head r % GT), swizzled
  {
    constexpr int CH = D / 8;  // 16-byte chunks per row
    for (int e = tid; e < L::kRows * CH; e += 128) {
      const int r = e / CH, c = e % CH;
      const int qi = r / GT, h = r % GT;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (qi < nq) {
        const size_t off =
            ((static_cast<size_t>(b) * p.n_new + q0 + qi) * p.n_q_heads + hbase + h) * D +
            c * 8;
        v = *reinterpret_cast<const uint4 *>(p.q + off);
      }
      const uint32_t addr =
          qs + (c / 8) * L::kQBoxBytes + r * 128 + (((c % 8) ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
                   "r"(v.y), "r"(v.z), "r"(v.w));
    }
  }
  __syncthreads();

  // Q fragments stay in registers for the whole key loop.
  uint32_t qa[KS][4];
  {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int c = 2 * kk + (lane >> 4);
      const uint32_t addr =
          qs + (c / 8) * L::kQBoxBytes + r * 128 + (((c % 8) ^ (r & 7)) << 4);
      ldsm_x4(addr, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }
  }

  // Rows of this thread in the accumulator fragments: r_lo and r_lo + 8.
  const int r_lo = warp * 16 + (lane >> 2);
  const int lim_lo = ctx + q0 + r_lo / GT;        // last key row r_lo may see
  const int lim_hi = ctx + q0 + (r_lo + 8) / GT;
  const int warp_lim = ctx + q0 + min((warp * 16 + 15) / GT, nq - 1);
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  bool timed_out = false;
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % L::kStages;
    const uint32_t st = sbase + s * L::kStageBytes;
    if (!timed_out &&
        !__all_sync(kFull, mbar_wait(sbase + L::kBarOff + 8 * s, (t / L::kStages) & 1))) {
      if (lane == 0) record_error(p.status, PA_ERR_TIMEOUT);
      // the next tile may already be in flight: let it land before giving up
      if (t + 1 < n_tiles)
        mbar_wait(sbase + L::kBarOff + 8 * ((t + 1) % L::kStages),
                  ((t + 1) / L::kStages) & 1);
      timed_out = true;
    }
    const int key0 = t * L::kKeys;
    // V rows past the last key any row sees may hold non-finite junk; P is
    // zero there, but 0 * inf is NaN, so clear them.
    if (key0 + L::kKeys - 1 > kmax) {
      for (int e = tid; e < L::kKeys * (D / 8); e += 128) {
        const int r = e / (D / 8), c = e % (D / 8);
        if (key0 + r > kmax) {
          const uint32_t addr = st + L::kTileBytes +
                                ((r >> 4) * L::kBoxes + c / 8) * L::kBoxBytes +
                                (r & 15) * 128 + (((c % 8) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0));
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
    }
    if (!timed_out && key0 <= warp_lim) {
      // ---- S = Q K^T for this warp's 16 rows x 64 keys
      float sacc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // 16 keys = page j of the tile
        const int rr = (lane >> 4) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int c = 2 * kk + ((lane >> 3) & 1);
          const uint32_t addr = st + (j * L::kBoxes + c / 8) * L::kBoxBytes + rr * 128 +
                                (((c % 8) ^ (rr & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma16816<BF16>(sacc[2 * j], qa[kk], b0, b1);
          mma16816<BF16>(sacc[2 * j + 1], qa[kk], b2, b3);
        }
      }
      // ---- scale, causal mask, online softmax (two rows per thread)
      float tmax_lo = -INFINITY, tmax_hi = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key0 + n * 8 + (lane & 3) * 2 + e;
          const float slo = sacc[n][e] * p.qscale, shi = sacc[n][2 + e] * p.qscale;
          sacc[n][e] = key <= lim_lo ? slo : -INFINITY;
          sacc[n][2 + e] = key <= lim_hi ? shi : -INFINITY;
          tmax_lo = fmaxf(tmax_lo, sacc[n][e]);
          tmax_hi = fmaxf(tmax_hi, sacc[n][2 + e]);
        }
      }
      tmax_lo = fmaxf(tmax_lo, __shfl_xor_sync(kFull, tmax_lo, 1));
      tmax_lo = fmaxf(tmax_lo, __shfl_xor_sync(kFull, tmax_lo, 2));
      tmax_hi = fmaxf(tmax_hi, __shfl_xor_sync(kFull, tmax_hi, 1));
      tmax_hi = fmaxf(tmax_hi, __shfl_xor_sync(kFull, tmax_hi, 2));
      const float mn_lo = fmaxf(m_lo, tmax_lo), mn_hi = fmaxf(m_hi, tmax_hi);
      // A row whose keys are all masked in this tile keeps m = -inf only if it
      // has seen nothing yet, which cannot happen (key 0 is in tile 0).
      const float c_lo = mn_lo == -INFINITY ? 1.f : ex2(m_lo - mn_lo);
      const float c_hi = mn_hi == -INFINITY ? 1.f : ex2(m_hi - mn_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      l_lo *= c_lo;
      l_hi *= c_hi;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= c_lo;
        o[n][1] *= c_lo;
        o[n][2] *= c_hi;
        o[n][3] *= c_hi;
      }
      // P as the A operand (k-step j covers keys 16j..16j+15), split into a
      // 16-bit head and a 16-bit remainder so that P V keeps ~16 significant
      // bits: a single bf16 rounding of P perturbs each weight by up to 2^-9,
      // which with few keys moves O by more than the 2e-3 bound allows.
      uint32_t pa[4][4], pb[4][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float p0 = ex2(sacc[n][0] - (m_lo == -INFINITY ? 0.f : m_lo));
        const float p1 = ex2(sacc[n][1] - (m_lo == -INFINITY ? 0.f : m_lo));
        const float p2 = ex2(sacc[n][2] - (m_hi == -INFINITY ? 0.f : m_hi));
        const float p3 = ex2(sacc[n][3] - (m_hi == -INFINITY ? 0.f : m_hi));
        l_lo += p0 + p1;
        l_hi += p2 + p3;
        const uint32_t h01 = pack2<BF16>(p0, p1), h23 = pack2<BF16>(p2, p3);
        const float2 r01 = unpack2<BF16>(h01), r23 = unpack2<BF16>(h23);
        pa[n >> 1][(n & 1) * 2 + 0] = h01;
        pa[n >> 1][(n & 1) * 2 + 1] = h23;
        pb[n >> 1][(n & 1) * 2 + 0] = pack2<BF16>(p0 - r01.x, p1 - r01.y);
        pb[n >> 1][(n & 1) * 2 + 1] = pack2<BF16>(p2 - r23.x, p3 - r23.y);
      }
      // ---- O += P V
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int rr = (lane & 7) + ((lane >> 3) & 1) * 8;  // key row within page j
#pragma unroll
        for (int nn = 0; nn < NT / 2; ++nn) {
          const int c = 2 * nn + (lane >> 4);
          const uint32_t addr = st + L::kTileBytes + (j * L::kBoxes + c / 8) * L::kBoxBytes +
                                rr * 128 + (((c % 8) ^ (rr & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma16816<BF16>(o[2 * nn], pa[j], b0, b1);
          mma16816<BF16>(o[2 * nn + 1], pa[j], b2, b3);
          mma16816<BF16>(o[2 * nn], pb[j], b0, b1);
          mma16816<BF16>(o[2 * nn + 1], pb[j], b2, b3);
        }
      }
    }
    // every warp is done with stage s; a timeout anywhere stops new loads
    const bool stop = __syncthreads_or(timed_out);
    if (stop) break;
    if (warp == 0 && t + L::kStages < n_tiles) issue(t + L::kStages);
  }

  // ---- O / l, one write
  l_lo += __shfl_xor_sync(kFull, l_lo, 1);
  l_lo += __shfl_xor_sync(kFull, l_lo, 2);
  l_hi += __shfl_xor_sync(kFull, l_hi, 1);
  l_hi += __shfl_xor_sync(kFull, l_hi, 2);
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
  const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = r_lo + half * 8;
    const int qi = r / GT, h = r % GT;
    if (qi >= nq) continue;
    const float inv = half ? inv_hi : inv_lo;
    float *dst = p.out +
                 ((static_cast<size_t>(b) * p.n_new + q0 + qi) * p.n_q_heads + hbase + h) * D +
                 (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      *reinterpret_cast<float2 *>(dst + n * 8) =
          make_float2(o[n][half * 2] * inv, o[n][half * 2 + 1] * inv);
  }
}

template <int D, int GT, bool BF16>
int launch_prefill_t(const PrefillLaunch &a, cudaStream_t stream) {
  using L = PrefillSmem<D>;
  auto kern = prefill_mma_kernel<D, GT, BF16>;
  static uint64_t attr_set = 0;
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
  PrefillParams p;
  p.q = static_cast<const uint16_t *>(a.q);
  p.block_table = a.block_table;
  p.ctx_lens = a.ctx_lens;
  p.out = a.out;
  p.status = a.status;
  p.qscale = a.scale * kLog2e;
  p.n_new = a.n_new;
  p.n_q_heads = a.n_q_heads;
  p.n_kv_heads = a.n_kv_heads;
  p.group = a.n_q_heads / a.n_kv_heads;
  p.batch = a.batch;
  p.max_blocks = a.max_blocks;
  p.num_pages = a.num_pages;
  constexpr int BQ = L::kRows / GT;
  const dim3 grid((a.n_new + BQ - 1) / BQ, a.n_kv_heads * (p.group / GT), a.batch);
  kern<<<grid, 128, L::kAlloc, stream>>>(kmap, vmap, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <int D, bool BF16>
int launch_prefill_d(const PrefillLaunch &a, cudaStream_t stream) {
  switch (group_tile(a.n_q_heads / a.n_kv_heads)) {
    case 8: return launch_prefill_t<D, 8, BF16>(a, stream);
    case 4: return launch_prefill_t<D, 4, BF16>(a, stream);
    case 2: return launch_prefill_t<D, 2, BF16>(a, stream);
    default: return launch_prefill_t<D, 1, BF16>(a, stream);
  }
}

}  // namespace

int launch_prefill(const PrefillLaunch &a, cudaStream_t stream) {
  if (a.head_dim == 128)
    return a.bf16 ? launch_prefill_d<128, true>(a, stream)
                  : launch_prefill_d<128, false>(a, stream);
  return a.bf16 ? launch_prefill_d<64, true>(a, stream)
                : launch_prefill_d<64, false>(a, stream);
}

}  // namespace pa
