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
// the whole group ("吞吐与延迟的系统模型" 5).  K/V tiles are 128 keys = 8 pages,
// loaded page by page with 2-D TMA (128-byte swizzle) into a ring of K and V
// stages laid out as the canonical K-major (K) and MN-major (V) operand
// tiles.  Per tile j:
//   S_j   = Q K_j^T           tcgen05.mma, M=128 N=128 K=head_dim, A and B in
//                             shared memory, into TMEM buffer j&1 (two
//                             buffers: S_{j+1} is computed while tile j's
//                             softmax runs)
//   softmax                   row r is shared by two threads; each owns one
//                             half of every tile's keys with its own running
//                             (m, l) and its own accumulator O_half
//   P_j   -> TMEM             written over the S_j columns its thread has
//                             just read, as two 16-bit terms (head +
//                             remainder) so the weights keep ~16 significant
//                             bits
//   O_A  += P_j[:, :64] V_j[:64],  O_B += P_j[:, 64:] V_j[64:]
//                             tcgen05.mma with A in TMEM, B in shared memory
// The halves are merged once at the end with the exponent law of 19.6.2.
//
// Warp roles: eight consumer warps (softmax), one load warp (TMA), one MMA
// warp (a single issuing thread).  Every hand-off is an mbarrier: TMA
// transaction counts, tcgen05.commit arrivals, and one arrival per consumer
// warp when its half of P_j is in TMEM.  The running max moves only when a
// score exceeds it by more than 8 (log2 units); the thread then rescales its
// accumulator row in TMEM.  Every wait is bounded and gives up early once
// another role has raised the CTA's abort flag.
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 8.0f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kRows = 128;       // M: (query, head) rows per CTA
constexpr int kKeys = 128;       // keys per K/V tile (8 pages)
constexpr int kConsumers = 256;  // eight consumer warps, two threads per row
constexpr int kLoadWarp = kConsumers / 32;
constexpr int kMmaWarp = kLoadWarp + 1;
constexpr int kThreads = kConsumers + 64;

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
  static constexpr int kStages = D == 128 ? 3 : 4;     // K and V ring depth
  static constexpr int kColBlk = kRows * 128;          // one 64-column block, 128 rows
  static constexpr int kQBytes = (D / 64) * kColBlk;
  static constexpr int kKVBytes = (D / 64) * kColBlk;  // 128 keys x D
  static constexpr int kQ = 0;
  static constexpr int kK0 = kQ + kQBytes;
  static constexpr int kV0 = kK0 + kStages * kKVBytes;
  static constexpr int kBars = kV0 + kStages * kKVBytes;
  static constexpr int kSlot = kBars + 24 * 8;  // TMEM address, abort flag
  static constexpr int kBytes = kSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
  static_assert(2 * kRows * 8 <= kKVBytes, "final exchange must fit in one K stage");
};

// mbarrier indices
enum {
  kBarK = 0,        // K stage s landed (TMA transaction count), s < 4
  kBarV = 4,        // V stage s landed
  kBarKFree = 8,    // K stage s read by its S MMAs (commit)
  kBarVFree = 12,   // V stage s read by both halves' P V MMAs (commit)
  kBarS = 16,       // S_t ready in TMEM buffer t&1 (commit), per buffer
  kBarO = 18,       // P V_t of key half h done (commit), per half
  kBarPReady = 20,  // P_t of key half h in TMEM (one arrival per warp), per half
  kNumBars = 22
};

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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Bounded wait on one mbarrier phase that also gives up once another role has
// raised the abort flag.  Warp-wide callers combine the result with
// __all_sync.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

__device__ __forceinline__ void raise_abort(int *status, volatile int *abort_flag) {
  record_error(status, PA_ERR_TIMEOUT);
  *abort_flag = 1;
}

// Load warp: K_t and V_t into stage t % kStages, each once the MMAs that
// read the stage's previous tile have completed.  Lane j < 8 copies page j
// of the tile (one box per 64 columns).  Page ids come in 32-page windows
// held one per lane, fetched one window ahead and checked when used.
template <int D>
__device__ __forceinline__ void load_tiles(const CUtensorMap *kmap, const CUtensorMap *vmap,
                                           uint32_t sb, const int32_t *bt_row, int n_pages,
                                           int n_tiles, int num_pages, int y_page, int y_head,
                                           int *status, volatile int *abort_flag, int lane) {
  using L = TcSmem<D>;
  constexpr int S = L::kStages;
  constexpr int kBoxes = D / 64;
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  auto load_window = [&](int w) {
    const int pg = 32 * w + lane;
    return pg < n_pages ? __ldg(bt_row + pg) : 0;  // past the end: page 0, masked
  };
  if (lane == 0) {
    prefetch_tensormap(kmap);
    prefetch_tensormap(vmap);
  }
  int wcur = load_window(0), wnext = load_window(1);
  auto load_tile = [&](int which, int t, int idj) {
    const int s = t % S;
    const uint32_t full = bar((which ? kBarV : kBarK) + s);
    const uint32_t dst0 = sb + (which ? L::kV0 : L::kK0) + s * L::kKVBytes;
    if (lane == 0) mbar_arrive_expect_tx(full, L::kKVBytes);
    __syncwarp();
    if (lane < 8) {
#pragma unroll
      for (int bx = 0; bx < kBoxes; ++bx)
        tma_load_2d(dst0 + bx * L::kColBlk + lane * 2048, which ? vmap : kmap, bx * 64,
                    idj * y_page + y_head, full);
    }
  };
  int issued = 0;
  bool failed = false;
  for (int t = 0; t < n_tiles; ++t) {
    if (t > 0 && (t & 3) == 0) {  // the tile starts a new 32-page window
      wcur = wnext;
      wnext = load_window((t >> 2) + 1);
    }
    int idj = __shfl_sync(kFull, wcur, 8 * (t & 3) + (lane & 7));
    if (lane < 8 && static_cast<unsigned>(idj) >= static_cast<unsigned>(num_pages)) {
      record_error(status, PA_ERR_BAD_BLOCK);
      idj = 0;
    }
    const int par = ((t / S) - 1) & 1;
    if (t >= S && !__all_sync(kFull, wait_or_abort(bar(kBarKFree + t % S), par, abort_flag))) {
      failed = true;
      break;
    }
    load_tile(0, t, idj);
    if (t >= S && !__all_sync(kFull, wait_or_abort(bar(kBarVFree + t % S), par, abort_flag))) {
      issued = 2 * t + 1;
      failed = true;
      break;
    }
    load_tile(1, t, idj);
    issued = 2 * t + 2;
  }
  if (failed) {
    if (lane == 0) raise_abort(status, abort_flag);
    // Copies in flight still land in shared memory: wait for them.
    for (int i = issued - 1; i >= 0 && i >= issued - 2 * S; --i) {
      const int t = i >> 1;
      mbar_wait(bar(((i & 1) ? kBarV : kBarK) + t % S), (t / S) & 1);
    }
  }
}

// MMA warp (lane 0 issues): S_0, S_1, then per tile t
//   O_0 += P_t V_t (keys 0-63), O_1 += P_t V_t (keys 64-127), S_{t+2}.
// S_{t+2} goes after P V_t because it overwrites P_t in TMEM buffer t&1;
// tcgen05 MMAs of one thread run in issue order.
template <int D, bool BF16>
__device__ __forceinline__ void mma_tiles(uint32_t sb, uint32_t tS, uint32_t tO, int n_tiles,
                                          int *status, volatile int *abort_flag, int lane) {
  using L = TcSmem<D>;
  constexpr int S = L::kStages;
  constexpr int KSQ = D / 16;
  constexpr uint32_t kIdS = tc::idesc_f16(BF16, kRows, kKeys, false, false);
  constexpr uint32_t kIdO = tc::idesc_f16(BF16, kRows, D, false, true);
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  // Descriptors of stage 0 / the Q tile; other stages and K steps add their
  // byte offset >> 4 to the address field.
  const uint64_t dq = tc::smem_desc_sw128(sb + L::kQ, 16, 1024);
  const uint64_t dk = tc::smem_desc_sw128(sb + L::kK0, 16, 1024);
  const uint64_t dv = tc::smem_desc_sw128(sb + L::kV0, L::kColBlk, 1024);
  uint32_t last_bar = 0, last_par = 0;  // most recent commit (for the failure path)
  bool failed = false;

  auto issue_s = [&](int t) {
    if (!__all_sync(kFull, wait_or_abort(bar(kBarK + t % S), (t / S) & 1, abort_flag)))
      return false;
    tc::fence_after_sync();
    if (lane == 0) {
      const uint64_t kst = dk + static_cast<uint64_t>((t % S) * L::kKVBytes >> 4);
#pragma unroll
      for (int kk = 0; kk < KSQ; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::kColBlk + (kk & 3) * 32) >> 4);
        tc::mma_f16(tS + (t & 1) * kKeys, dq + off, kst + off, kIdS, kk > 0);
      }
      tc::commit(bar(kBarS + (t & 1)));
      tc::commit(bar(kBarKFree + t % S));
    }
    __syncwarp();
    last_bar = bar(kBarS + (t & 1));
    last_par = (t >> 1) & 1;
    return true;
  };
  auto issue_pv = [&](int t, int h) {
    if (!__all_sync(kFull, wait_or_abort(bar(kBarPReady + h), t & 1, abort_flag))) return false;
    if (h == 0 &&
        !__all_sync(kFull, wait_or_abort(bar(kBarV + t % S), (t / S) & 1, abort_flag)))
      return false;
    tc::fence_after_sync();
    if (lane == 0) {
      const uint64_t vst = dv + static_cast<uint64_t>((t % S) * L::kKVBytes >> 4);
      const uint32_t pa = tS + (t & 1) * kKeys + 64 * h;  // this half's P: hi, then lo
#pragma unroll
      for (int ph = 0; ph < 2; ++ph) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_f16_tmem_a(tO + h * D, pa + 32 * ph + 8 * kk,
                             vst + static_cast<uint64_t>(((4 * h + kk) * 2048) >> 4), kIdO,
                             (t > 0 || kk > 0 || ph > 0) ? 1u : 0u);
      }
      tc::commit(bar(kBarO + h));
      if (h == 1) tc::commit(bar(kBarVFree + t % S));
    }
    __syncwarp();
    last_bar = bar(kBarO + h);
    last_par = t & 1;
    return true;
  };

  bool any = false;
  if (!issue_s(0)) failed = true;
  else any = true;
  if (!failed && n_tiles > 1 && !issue_s(1)) failed = true;
  for (int t = 0; t < n_tiles && !failed; ++t) {
    if (!issue_pv(t, 0) || !issue_pv(t, 1) || (t + 2 < n_tiles && !issue_s(t + 2)))
      failed = true;
  }
  if (failed) {
    if (lane == 0) raise_abort(status, abort_flag);
    // Nothing this warp started may still run when the CTA leaves.
    if (any) mbar_wait(last_bar, last_par);
  }
}

// Consumer warps 0-7: threads r and r + 128 share row r % 128; warps w and
// w + 4 reach the same TMEM lanes.  `half` owns keys [64 half, 64 half + 64)
// of every tile, with its own running (m, l) and its own accumulator O_half.
template <int D, int GT, bool BF16>
__device__ __forceinline__ void consume_tiles(uint32_t sb, uint32_t tS, uint32_t tO,
                                              const TcParams &p, int b, int q0, int hbase,
                                              int nq, int ctx, int kmax, int n_tiles,
                                              volatile int *abort_flag, int tid, int warp,
                                              int lane) {
  using L = TcSmem<D>;
  constexpr int S = L::kStages;
  constexpr int HK = kKeys / 2;  // keys of each tile this thread owns
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  const int half = warp >> 2;
  const int r = ((warp & 3) << 5) + lane, qi = r / GT, hh = r % GT;
  const int lim = min(ctx + q0 + qi, kmax);  // last key row r sees
  const int lim_all = ctx + q0;              // every row sees keys <= this
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tOh = tO + half * D + lane_base;  // this half's accumulator row

  bool bad = false;
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j < n_tiles; ++j) {
    const int key0 = j * kKeys;
    const int kbase = key0 + half * HK;
    // my 64 columns of buffer j&1: S_j, then P_j (head terms, remainder terms)
    const uint32_t tSj = tS + (j & 1) * kKeys + half * HK + lane_base;
    if (!__all_sync(kFull, wait_or_abort(bar(kBarS + (j & 1)), (j >> 1) & 1, abort_flag))) {
      bad = true;
      break;
    }
    tc::fence_after_sync();
    uint32_t sr[HK];
    tc::ld32(tSj, *reinterpret_cast<uint32_t(*)[32]>(sr));
    tc::ld32(tSj + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
    tc::wait_ld();

    // ---- scale, mask, max of my keys; lazy move of my reference max
    float tmax = -INFINITY;
    if (key0 + kKeys - 1 <= lim_all) {  // no key of this tile is masked
#pragma unroll
      for (int c = 0; c < HK; ++c) {
        const float v = __uint_as_float(sr[c]) * p.qscale;
        sr[c] = __float_as_uint(v);
        tmax = fmaxf(tmax, v);
      }
    } else {
#pragma unroll
      for (int c = 0; c < HK; ++c) {
        const float v = (kbase + c <= lim) ? __uint_as_float(sr[c]) * p.qscale : -INFINITY;
        sr[c] = __float_as_uint(v);
        tmax = fmaxf(tmax, v);
      }
    }
    const bool need = tmax > m + kSlack;
    float corr = 1.f;
    if (need) {
      const float mn = fmaxf(m, tmax);
      corr = ex2(m - mn);  // 0 while m was still -inf
      m = mn;
      l *= corr;
    }
    // ---- P = e^(s - m) as head + remainder, into the columns S_j came from
    const bool live = m != -INFINITY;  // nothing seen yet: every weight is 0
    {
      uint32_t phi[HK / 2], plo[HK / 2];
#pragma unroll
      for (int k = 0; k < HK / 2; ++k) {
        const float p0 = live ? ex2(__uint_as_float(sr[2 * k]) - m) : 0.f;
        const float p1 = live ? ex2(__uint_as_float(sr[2 * k + 1]) - m) : 0.f;
        l += p0 + p1;
        phi[k] = pack2<BF16>(p0, p1);
        const float2 hr = unpack2<BF16>(phi[k]);
        plo[k] = pack2<BF16>(p0 - hr.x, p1 - hr.y);
      }
      tc::st32(tSj, phi);
      tc::st32(tSj + 32, plo);
    }
    // ---- P V_{j-1} of my half done: my accumulator is stable (and the MMA
    // warp has taken P_{j-1}, so this warp's next arrival starts a new phase)
    if (j > 0) {
      if (!__all_sync(kFull, wait_or_abort(bar(kBarO + half), (j - 1) & 1, abort_flag))) {
        bad = true;
        break;
      }
      tc::fence_after_sync();
      if (__any_sync(kFull, need)) {
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          tc::ld32(tOh + cb * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
          tc::st32(tOh + cb * 32, o);
        }
      }
    }
    tc::wait_st();
    // ---- V rows past the last key any row sees may hold non-finite junk;
    // P is 0 there but 0 * inf is NaN inside the MMA, so clear them (each half
    // clears the rows its own P V reads).
    if (key0 + kKeys - 1 > kmax) {
      if (!__all_sync(kFull, wait_or_abort(bar(kBarV + j % S), (j / S) & 1, abort_flag))) {
        bad = true;
        break;
      }
      const uint32_t vst = sb + L::kV0 + (j % S) * L::kKVBytes;
      const int first = max(kmax - key0 + 1, half * HK);
      const int htid = tid & (kConsumers / 2 - 1);
      for (int e = htid; e < (half * HK + HK - first) * (D / 8); e += kConsumers / 2) {
        const int rr = first + e / (D / 8), c = e % (D / 8);
        st_shared_v4(vst + (c >> 3) * L::kColBlk + swz128(rr, c), 0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();  // cleared V rows -> read by the tensor cores
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarPReady + half));  // one arrival per warp
  }
  tc::wait_st();
  if (!bad)
    bad = !__all_sync(kFull, wait_or_abort(bar(kBarO), (n_tiles - 1) & 1, abort_flag));
  if (!bad)
    bad = !__all_sync(kFull, wait_or_abort(bar(kBarO + 1), (n_tiles - 1) & 1, abort_flag));
  tc::fence_after_sync();

  // ---- merge the two halves once (exponent law) and write O / l.  Every
  // K/V copy has landed and been read by now, so K stage 0 carries the
  // exchange.
  const uint32_t x_mine = sb + L::kK0 + (half * kRows + r) * 8;
  const uint32_t x_peer = sb + L::kK0 + ((half ^ 1) * kRows + r) * 8;
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(x_mine), "f"(m), "f"(l) : "memory");
  if (consumers_sync_or(bad)) {
    if (tid == 0) raise_abort(p.status, abort_flag);
    return;
  }
  float m2, l2;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(m2), "=f"(l2) : "r"(x_peer) : "memory");
  const float mA = half ? m2 : m, lA = half ? l2 : l;  // keys [0, 64) of each tile
  const float mB = half ? m : m2, lB = half ? l : l2;  // keys [64, 128)
  const float M = fmaxf(mA, mB);
  const float fA = mA == -INFINITY ? 0.f : ex2(mA - M);
  const float fB = mB == -INFINITY ? 0.f : ex2(mB - M);
  const float lt = lA * fA + lB * fB;
  const float sA = lt > 0.f ? fA / lt : 0.f, sB = lt > 0.f ? fB / lt : 0.f;
  float *dst = p.out +
               ((static_cast<size_t>(b) * p.n_new + q0 + qi) * p.n_q_heads + hbase + hh) * D +
               half * (D / 2);
#pragma unroll
  for (int cb = 0; cb < D / 64; ++cb) {  // my D/2 output columns
    uint32_t oa[32], ob[32];
    tc::ld32(tO + lane_base + half * (D / 2) + cb * 32, oa);
    tc::ld32(tO + D + lane_base + half * (D / 2) + cb * 32, ob);
    tc::wait_ld();
    if (qi < nq) {
#pragma unroll
      for (int k = 0; k < 32; k += 4)
        *reinterpret_cast<float4 *>(dst + cb * 32 + k) = make_float4(
            __uint_as_float(oa[k]) * sA + __uint_as_float(ob[k]) * sB,
            __uint_as_float(oa[k + 1]) * sA + __uint_as_float(ob[k + 1]) * sB,
            __uint_as_float(oa[k + 2]) * sA + __uint_as_float(ob[k + 2]) * sB,
            __uint_as_float(oa[k + 3]) * sA + __uint_as_float(ob[k + 3]) * sB);
    }
  }
}

template <int D, int GT, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const TcParams p) {
  using L = TcSmem<D>;
  constexpr int BQ = kRows / GT;  // queries per CTA

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
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(bar(i), (i == kBarPReady || i == kBarPReady + 1) ? kConsumers / 64 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // S_0: columns 0-127, S_1: 128-255, O_A: 256 .. 256+D-1, O_B: 256+D .. 256+2D-1
    tc::alloc(sb + L::kSlot, 512);
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
  const uint32_t tS = tmem, tO = tmem + 2 * kKeys;

  if (warp == kLoadWarp) {
    load_tiles<D>(&kmap, &vmap, sb, p.block_table + static_cast<size_t>(b) * p.max_blocks,
                  n_pages, n_tiles, p.num_pages, p.n_kv_heads * 16, g * 16, p.status,
                  abort_flag, lane);
  } else if (warp == kMmaWarp) {
    mma_tiles<D, BF16>(sb, tS, tO, n_tiles, p.status, abort_flag, lane);
  } else {
    consume_tiles<D, GT, BF16>(sb, tS, tO, p, b, q0, hbase, nq, ctx, kmax, n_tiles,
                               abort_flag, tid, warp, lane);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::dealloc(tmem, 512);
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
