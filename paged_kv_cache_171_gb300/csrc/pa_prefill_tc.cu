// pa_prefill_tc.cu -- chunked-prefill paged attention on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Query i of sequence b (0 <= i < n_new) attends keys 0 .. ctx_lens[b] + i
// (ch. 19 "推理系统与性能工程", 19.3.1 prefill; 19.6.3 FlashAttention forward:
// the Q tile stays on chip, K/V tiles stream through, running m, l, O, one
// write of O / l; 19.6.2 online softmax).
//
// Tile plan.  A CTA owns M = 128 rows = (query, head) pairs of one kv head's
// GQA group (GT heads x 128/GT consecutive queries), so every K/V tile serves
// the whole group ("吞吐与延迟的系统模型" 5).  Row r lives in TMEM lane r and is
// owned by thread r of the four consumer warps.  K/V tiles are 128 keys =
// 8 pages; a producer warp loads them page by page with 2-D TMA (128-byte
// swizzle) into two K and two V stages laid out as the canonical K-major
// (K) and MN-major (V) operand tiles.  Per tile j:
//   S_j   = Q K_j^T            tcgen05.mma, M=128 N=128 K=head_dim, into TMEM
//   softmax on S_j rows        thread r: its row from TMEM, mask, max, ex2
//   P_j   -> shared memory     two 16-bit terms (head + remainder) so the
//                              weights keep ~16 significant bits
//   O    += P_j V_j            tcgen05.mma, M=128 N=head_dim K=128, in TMEM
// S_{j+1} is issued as soon as S_j has been read, so it overlaps the softmax
// of tile j; the softmax of tile j+1 overlaps P V of tile j.  The running max
// moves only when a row's max exceeds it by more than 8 (log2 units); O in
// TMEM is then rescaled in place by its row's thread.
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 8.0f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kRows = 128;      // M: (query, head) rows per CTA
constexpr int kKeys = 128;      // keys per K/V tile (8 pages)
constexpr int kConsumers = 256; // eight consumer warps, two threads per row
constexpr int kThreads = kConsumers + 32;  // + one producer warp

struct TcParams {
  const uint16_t *q;
  const int32_t *block_table;
  const int32_t *ctx_lens;
  float *out;
  int *status;
  float qscale;  // scale * log2 e
  int n_new, n_q_heads, n_kv_heads, group, batch, max_blocks, num_pages;
};

// Shared memory (offsets from a 1024-aligned base).  Operand tiles are
// stored as 64-column blocks of [rows][128 B] with the 128-byte swizzle.
template <int D>
struct TcSmem {
  static constexpr int kColBlk = kRows * 128;   // one 64-column block, 128 rows
  static constexpr int kQBytes = (D / 64) * kColBlk;
  static constexpr int kKVBytes = (D / 64) * kColBlk;  // 128 keys x D
  static constexpr int kPBytes = 2 * kColBlk;           // 128 rows x 128 keys
  static constexpr int kQ = 0;
  static constexpr int kK0 = kQ + kQBytes;
  static constexpr int kV0 = kK0 + 2 * kKVBytes;
  static constexpr int kPhi = kV0 + 2 * kKVBytes;
  static constexpr int kPlo = kPhi + kPBytes;
  static constexpr int kBars = kPlo + kPBytes;  // 12 mbarriers
  static constexpr int kXchg = kBars + 12 * 8;  // per-row halves: max, sum
  static constexpr int kSlot = kXchg + 2 * kRows * 4;  // TMEM address, abort flag
  static constexpr int kBytes = kSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
};

// mbarrier indices
enum { kBarK = 0, kBarV = 2, kBarKFree = 4, kBarVFree = 6, kBarS = 8, kBarO = 9 };

__device__ __forceinline__ uint32_t swz128(int r, int c) {  // row r, 16-B chunk c < 8
  return r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Named barrier over the consumer warps, OR-reducing a flag.
__device__ __forceinline__ bool consumers_sync_or(bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<int>(v)), "r"(kConsumers)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b,
                                             uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// Producer warp: loads K_t and V_t (8 pages each) for t = 0 .. n_tiles-1.
// Stage t & 1 of K (V) is refilled once the MMA that read it for tile t-2,
// S_{t-2} (P V_{t-2}), has completed (its commit arrives on the free barrier).
template <int D>
__device__ __forceinline__ void produce_tiles(const CUtensorMap *kmap, const CUtensorMap *vmap,
                                              uint32_t sb, const int32_t *bt_row,
                                              int n_pages, int n_tiles, int num_pages,
                                              int y_page, int y_head, int *status,
                                              volatile int *abort_flag, int lane) {
  using L = TcSmem<D>;
  constexpr int kBoxes = D / 64;
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  int issued[2] = {0, 0};  // K tiles, V tiles whose loads were issued
  for (int t = 0; t < n_tiles; ++t) {
    int id = 0;  // lane j < 8: page 8t + j (past the sequence: page 0, masked)
    const int pg = 8 * t + (lane & 7);
    if (lane < 8 && pg < n_pages) {
      id = __ldg(bt_row + pg);
      if (static_cast<unsigned>(id) >= static_cast<unsigned>(num_pages)) {
        record_error(status, PA_ERR_BAD_BLOCK);
        id = 0;
      }
    }
    const int s = t & 1;
    bool stop = false;
    for (int which = 0; which < 2 && !stop; ++which) {  // K, then V
      if (t >= 2) {
        const int fb = (which ? kBarVFree : kBarKFree) + s;
        if (!__all_sync(kFull, mbar_wait(bar(fb), ((t - 2) >> 1) & 1)) || *abort_flag) {
          stop = true;
          break;
        }
      }
      const uint32_t full = bar((which ? kBarV : kBarK) + s);
      const uint32_t dst0 = sb + (which ? L::kV0 : L::kK0) + s * L::kKVBytes;
      if (lane == 0) mbar_arrive_expect_tx(full, L::kKVBytes);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int idj = __shfl_sync(kFull, id, j);
        if (lane == 0) {
          const int y = idj * y_page + y_head;
#pragma unroll
          for (int bx = 0; bx < kBoxes; ++bx)
            tma_load_2d(dst0 + bx * L::kColBlk + j * 2048, which ? vmap : kmap, bx * 64, y,
                        full);
        }
      }
      issued[which] = t + 1;
    }
    if (stop) break;
  }
  // Every issued copy lands before the CTA can leave (consumers wait for them
  // on the normal path; this covers an aborted one).
  for (int which = 0; which < 2; ++which)
    for (int t = issued[which] >= 2 ? issued[which] - 2 : 0; t < issued[which]; ++t)
      mbar_wait(bar((which ? kBarV : kBarK) + (t & 1)), (t >> 1) & 1);
}

template <int D, int GT, bool BF16>
__device__ __forceinline__ void consume_tiles(uint32_t sb, uint32_t tS, uint32_t tO,
                                              const TcParams &p, int b, int q0, int hbase,
                                              int nq, int ctx, int kmax, int n_tiles,
                                              volatile int *abort_flag, int tid, int warp,
                                              int lane);

// Consumer warps 0-7 (threads r and r + 128 share row r % 128); thread 0 also
// issues the MMAs.  Warp 8 produces the K/V tiles.
template <int D, int GT, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const TcParams p) {
  using L = TcSmem<D>;
  constexpr int BQ = kRows / GT;   // queries per CTA

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int q0 = blockIdx.x * BQ;
  const int n_sub = p.group / GT;
  const int g = blockIdx.y / n_sub;
  const int hbase = g * p.group + (blockIdx.y % n_sub) * GT;
  const int b = blockIdx.z;
  const int nq = min(BQ, p.n_new - q0);  // real queries in this CTA

  int ctx = p.ctx_lens[b];
  const int maxT = p.max_blocks * 16;
  if (ctx < 0 || ctx + p.n_new > maxT) {
    if (tid == 0) record_error(p.status, PA_ERR_BAD_CTX);
    ctx = max(0, min(ctx, maxT - p.n_new));
  }
  const int kmax = ctx + q0 + nq - 1;  // last key any row of this CTA sees
  const int n_tiles = kmax / kKeys + 1;
  const int n_pages = (ctx + p.n_new + 15) >> 4;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kSlot + 4);

  if (tid == 0) {
    for (int i = 0; i < 10; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tc::alloc(sb + L::kSlot, 256);  // S: columns 0-127, O: 128 .. 128+D-1
    tc::relinquish();
  }
  // Q tile: row r = query r / GT, head r % GT (zeros past the chunk's end)
  if (tid < kConsumers) {
    for (int e = tid; e < kRows * (D / 8); e += kConsumers) {
      const int r = e / (D / 8), c = e % (D / 8);
      const int qi = r / GT, hh = r % GT;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (qi < nq)
        v = *reinterpret_cast<const uint4 *>(
            p.q + ((static_cast<size_t>(b) * p.n_new + q0 + qi) * p.n_q_heads + hbase + hh) * D +
            c * 8);
      st_shared_v4(sb + L::kQ + (c >> 3) * L::kColBlk + swz128(r, c), v.x, v.y, v.z, v.w);
    }
    fence_proxy_async_smem();  // generic stores -> read by the tensor cores
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kSlot);
  const uint32_t tS = tmem, tO = tmem + 128;

  if (warp == kConsumers / 32) {
    produce_tiles<D>(&kmap, &vmap, sb, p.block_table + static_cast<size_t>(b) * p.max_blocks,
                     n_pages, n_tiles, p.num_pages, p.n_kv_heads * 16, g * 16, p.status,
                     abort_flag, lane);
  } else {
    consume_tiles<D, GT, BF16>(sb, tS, tO, p, b, q0, hbase, nq, ctx, kmax, n_tiles,
                               abort_flag, tid, warp, lane);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::dealloc(tmem, 256);
  }
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

template <int D, int GT, bool BF16>
__device__ __forceinline__ void consume_tiles(uint32_t sb, uint32_t tS, uint32_t tO,
                                              const TcParams &p, int b, int q0, int hbase,
                                              int nq, int ctx, int kmax, int n_tiles,
                                              volatile int *abort_flag, int tid, int warp,
                                              int lane) {
  using L = TcSmem<D>;
  constexpr int KSQ = D / 16;
  constexpr int HK = kKeys / 2;  // S columns (keys) per thread
  constexpr int HD = D / 2;      // O columns per thread
  constexpr uint32_t kIdS = tc::idesc_f16(BF16, kRows, kKeys, false, false);
  constexpr uint32_t kIdO = tc::idesc_f16(BF16, kRows, D, false, true);
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  // Two threads per row: warps w and w + 4 reach the same TMEM lanes; `half`
  // picks keys [64 half, 64 half + 64) of S and columns [HD half, +HD) of O.
  const int half = warp >> 2;
  const int r = ((warp & 3) << 5) + lane, qi = r / GT, hh = r % GT;
  const int lim = min(ctx + q0 + qi, kmax);  // last key row r sees
  const int lim_all = ctx + q0;              // every row sees keys <= this
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t x_mine = sb + L::kXchg + (half * kRows + r) * 4;
  const uint32_t x_peer = sb + L::kXchg + ((half ^ 1) * kRows + r) * 4;
  int issued_s = 0, issued_o = 0;  // thread 0's MMA groups, for a drain on error

  auto issue_s = [&](int t) {  // S_t = Q K_t^T, one thread
    const uint32_t kst = sb + L::kK0 + (t & 1) * L::kKVBytes;
#pragma unroll
    for (int kk = 0; kk < KSQ; ++kk) {
      const uint32_t off = (kk >> 2) * L::kColBlk + (kk & 3) * 32;
      tc::mma_f16(tS, tc::smem_desc_sw128(sb + L::kQ + off, 16, 1024),
                  tc::smem_desc_sw128(kst + off, 16, 1024), kIdS, kk > 0);
    }
    tc::commit(bar(kBarS));
    tc::commit(bar(kBarKFree + (t & 1)));
    ++issued_s;
  };
  auto issue_pv = [&](int t) {  // O += P_hi V_t + P_lo V_t, one thread
    const uint32_t vst = sb + L::kV0 + (t & 1) * L::kKVBytes;
#pragma unroll
    for (int ph = 0; ph < 2; ++ph) {
      const uint32_t pb = sb + (ph ? L::kPlo : L::kPhi);
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk)
        tc::mma_f16(tO, tc::smem_desc_sw128(pb + (kk >> 2) * L::kColBlk + (kk & 3) * 32, 16, 1024),
                    tc::smem_desc_sw128(vst + kk * 2048, L::kColBlk, 1024), kIdO,
                    (t > 0 || kk > 0 || ph > 0) ? 1u : 0u);
    }
    tc::commit(bar(kBarO));
    tc::commit(bar(kBarVFree + (t & 1)));
    ++issued_o;
  };

  bool bad = false;
  if (tid == 0) {
    if (mbar_wait(bar(kBarK), 0)) issue_s(0);
    else bad = true;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j < n_tiles; ++j) {
    const int key0 = j * kKeys;
    const int kbase = key0 + half * HK;
    // ---- my half of S_j's row -> registers, scaled and masked, half max
    if (!mbar_wait(bar(kBarS), j & 1)) bad = true;
    tc::fence_after_sync();
    uint32_t sr[HK];
#pragma unroll
    for (int cb = 0; cb < HK / 32; ++cb)
      tc::ld32(tS + lane_base + half * HK + cb * 32,
               *reinterpret_cast<uint32_t(*)[32]>(sr + cb * 32));
    tc::wait_ld();
    float hmax = -INFINITY;
    if (key0 + kKeys - 1 <= lim_all) {  // no key of this tile is masked
#pragma unroll
      for (int c = 0; c < HK; ++c) {
        const float v = __uint_as_float(sr[c]) * p.qscale;
        sr[c] = __float_as_uint(v);
        hmax = fmaxf(hmax, v);
      }
    } else {
#pragma unroll
      for (int c = 0; c < HK; ++c) {
        const float v = (kbase + c <= lim) ? __uint_as_float(sr[c]) * p.qscale : -INFINITY;
        sr[c] = __float_as_uint(v);
        hmax = fmaxf(hmax, v);
      }
    }
    st_shared_f32(x_mine, hmax);
    tc::fence_before_sync();
    if (consumers_sync_or(bad)) { bad = true; break; }  // S buffer, K stage free
    if (tid == 0 && j + 1 < n_tiles) {
      tc::fence_after_sync();
      if (mbar_wait(bar(kBarK + ((j + 1) & 1)), ((j + 1) >> 1) & 1)) issue_s(j + 1);
      else bad = true;
    }

    // ---- row max from both halves; lazy rescale decision (same in both)
    const float tmax = fmaxf(hmax, ld_shared_f32(x_peer));
    const bool need = tmax > m + kSlack;
    float corr = 1.f;
    if (need) {
      const float mn = fmaxf(m, tmax);
      corr = ex2(m - mn);  // 0 on the first tile (m = -inf)
      m = mn;
      l *= corr;
    }
    // ---- P V_{j-1} done: O is stable and the P buffers are free
    if (j > 0) {
      if (!mbar_wait(bar(kBarO), (j - 1) & 1)) bad = true;
      tc::fence_after_sync();
      if (__any_sync(kFull, need)) {
#pragma unroll
        for (int cb = 0; cb < HD / 32; ++cb) {
          uint32_t o[32];
          tc::ld32(tO + lane_base + half * HD + cb * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
          tc::st32(tO + lane_base + half * HD + cb * 32, o);
        }
        tc::wait_st();
      }
    }
    // ---- P = e^(s - m) as head + remainder: my 64 keys = 64-column block `half`
#pragma unroll
    for (int ch = 0; ch < HK / 8; ++ch) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float p0 = ex2(__uint_as_float(sr[ch * 8 + 2 * k]) - m);
        const float p1 = ex2(__uint_as_float(sr[ch * 8 + 2 * k + 1]) - m);
        l += p0 + p1;
        hi[k] = pack2<BF16>(p0, p1);
        const float2 hr = unpack2<BF16>(hi[k]);
        lo[k] = pack2<BF16>(p0 - hr.x, p1 - hr.y);
      }
      const uint32_t off = half * L::kColBlk + swz128(r, ch);
      st_shared_v4(sb + L::kPhi + off, hi[0], hi[1], hi[2], hi[3]);
      st_shared_v4(sb + L::kPlo + off, lo[0], lo[1], lo[2], lo[3]);
    }
    // ---- V rows past the last key any row sees may hold non-finite junk;
    // P is 0 there but 0 * inf is NaN inside the MMA, so clear them.
    if (key0 + kKeys - 1 > kmax) {
      if (!mbar_wait(bar(kBarV + (j & 1)), (j >> 1) & 1)) bad = true;
      const uint32_t vst = sb + L::kV0 + (j & 1) * L::kKVBytes;
      const int first = kmax - key0 + 1;
      for (int e = tid; e < (kKeys - first) * (D / 8); e += kConsumers) {
        const int rr = first + e / (D / 8), c = e % (D / 8);
        st_shared_v4(vst + (c >> 3) * L::kColBlk + swz128(rr, c), 0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    if (consumers_sync_or(bad)) { bad = true; break; }
    if (tid == 0) {
      tc::fence_after_sync();
      if (mbar_wait(bar(kBarV + (j & 1)), (j >> 1) & 1)) issue_pv(j);
      else bad = true;
    }
  }

  // ---- O / l, one write per row (each thread its HD columns)
  if (!bad && !mbar_wait(bar(kBarO), (n_tiles - 1) & 1)) bad = true;
  tc::fence_after_sync();
  st_shared_f32(x_mine, l);
  if (consumers_sync_or(bad)) {
    if (tid == 0) {
      record_error(p.status, PA_ERR_TIMEOUT);
      *abort_flag = 1;
      // let the MMAs in flight finish before the tensor memory is freed
      if (issued_s) mbar_wait(bar(kBarS), (issued_s - 1) & 1);
      if (issued_o) mbar_wait(bar(kBarO), (issued_o - 1) & 1);
    }
    return;
  }
  const float lt = l + ld_shared_f32(x_peer);
  const float inv = lt > 0.f ? 1.f / lt : 0.f;
  float *dst = p.out +
               ((static_cast<size_t>(b) * p.n_new + q0 + qi) * p.n_q_heads + hbase + hh) * D +
               half * HD;
#pragma unroll
  for (int cb = 0; cb < HD / 32; ++cb) {
    uint32_t o[32];
    tc::ld32(tO + lane_base + half * HD + cb * 32, o);
    tc::wait_ld();
    if (qi < nq) {
#pragma unroll
      for (int k = 0; k < 32; k += 4)
        *reinterpret_cast<float4 *>(dst + cb * 32 + k) =
            make_float4(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                        __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
    }
  }
}

template <int D, int GT, bool BF16>
int launch_tc_t(const PrefillLaunch &a, cudaStream_t stream) {
  using L = TcSmem<D>;
  auto kern = prefill_tc_kernel<D, GT, BF16>;
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
  TcParams p;
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
  constexpr int BQ = kRows / GT;
  const dim3 grid((a.n_new + BQ - 1) / BQ, a.n_kv_heads * (p.group / GT), a.batch);
  kern<<<grid, kThreads, L::kAlloc, stream>>>(kmap, vmap, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <int D, bool BF16>
int launch_tc_d(const PrefillLaunch &a, cudaStream_t stream) {
  switch (group_tile(a.n_q_heads / a.n_kv_heads)) {
    case 8: return launch_tc_t<D, 8, BF16>(a, stream);
    case 4: return launch_tc_t<D, 4, BF16>(a, stream);
    case 2: return launch_tc_t<D, 2, BF16>(a, stream);
    default: return launch_tc_t<D, 1, BF16>(a, stream);
  }
}

}  // namespace

int launch_prefill(const PrefillLaunch &a, cudaStream_t stream) {
  if (a.head_dim == 128)
    return a.bf16 ? launch_tc_d<128, true>(a, stream) : launch_tc_d<128, false>(a, stream);
  return a.bf16 ? launch_tc_d<64, true>(a, stream) : launch_tc_d<64, false>(a, stream);
}

}  // namespace pa
