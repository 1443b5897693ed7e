// pa_prefill_tc.cu -- chunked-prefill paged attention on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Query i of sequence b (0 <= i < n_new) attends keys 0 .. ctx_lens[b] + i
// (ch. 19 "推理系统与性能工程", 19.3.1 prefill; 19.6.3 FlashAttention forward:
// the Q tile stays on chip, K/V tiles stream through, running m, l, O, one
// write of O / l; 19.6.2 online softmax).
//
// Tile plan.  A CTA owns two row tiles, A and B, of 128 rows each; a row is
// a (query, head) pair of one kv head's GQA group (GT heads x 128/GT
// consecutive queries), and B holds the 128/GT queries after A's.  Every K/V
// tile therefore serves 256 rows ("吞吐与延迟的系统模型" 5).  K/V tiles are 128
// keys = 8 pages, loaded page by page with 2-D TMA (128-byte swizzle) into
// rings of K and V stages laid out as the canonical K-major (K) and MN-major
// (V) operand tiles.  For each row tile x and key tile j:
//   S_x   = Q_x K_j^T          tcgen05.mma M=128 N=128 K=head_dim, operands in
//                              shared memory, accumulator in TMEM
//   softmax                    one thread per row, all 128 keys of the tile
//   P_x   -> TMEM              written over S_x as one 16-bit term, or as
//                              two (head + remainder, ~16 bits) where the
//                              rounding of one term could matter (below)
//   O_x  += P_x V_j            tcgen05.mma with A in TMEM, B in shared memory
// The tensor pipe alternates between the two row tiles: while tile A's
// softmax runs it computes P_B V_j and S_B for the next key tile, and the
// other way round.  The softmax warpgroups enforce that ping-pong: B's
// softmax of key tile j starts once A has handed over P_A(j), and A's of
// tile j+1 once B has handed over P_B(j).  Left to themselves the two tiles
// fall into lockstep (their S MMAs finish together), both softmaxes then
// share the SM sub-partitions while the tensor pipe idles, and a key tile
// takes the sum of both phases instead of the larger.
//
// Warp roles: warps 0 and 1 issue the MMAs of row tiles A and B (one thread
// each), warps 2 and 3 the K and V TMA loads, warps 4-7 are tile A's softmax
// and 8-11 tile B's.  Every hand-off is an
// mbarrier.  MMAs of one thread run in issue order, so once S_x for key tile
// j has completed, P_x V_{j-1} has too: the softmax may rescale O_x then,
// and S_x may overwrite P_x.  The running max moves only when a score
// exceeds it by more than 8 (log2 units).  Every wait is bounded and gives up
// early once another role has raised the CTA's abort flag.
//
// Interleaved key tiles.  When a CTA's queries fit in row tile A (a short
// chunk, e.g. speculative verify: gamma drafted tokens x GT heads <= 128
// rows) row tile B takes the same rows, and the two tiles split the key
// tiles: A the even ones, B the odd ones, so one tile's softmax overlaps the
// other's MMAs.  Each tile keeps its own (m, l, O) over its keys; at the end
// B hands (m, l) to A through shared memory, A reads both O's from TMEM (its
// lanes hold the same rows of O_A and O_B) and merges the two states exactly:
// O = 2^(m_A - m) O_A + 2^(m_B - m) O_B, l likewise, m = max(m_A, m_B).  Both
// tiles read Q_A, and Q_B's bytes go to a third V stage.  A stage then serves
// the two row tiles in turn, so its full and free barriers are kept per (row
// tile, stage): each is used every lcm(2, stages) tiles by one waiter, in
// order, and its phase parity stays exact.
//
// One or two terms of P.  Rounding a weight p to 16 bits changes it by at
// most 2^-9 p (bf16), and the output row by sum_t w_t d_t v_t (w = p / l,
// |d_t| <= 2^-9): on short or peaked rows that can exceed the 2e-3 absolute
// bound, so there P keeps a remainder term.  A row tile's key tile j takes
// one term when, in every row, the tile's largest weight is below 1/16 of
// the weight l already accumulated over the tiles before it.  Then
// sum over such tiles of sum_t w_t^2 <= max_j (pmax_j / l) <= 1/16, and the
// rounding error of the single-term tiles has an rms of at most
// 2^-9 / sqrt(3) * rms(v) / 4.  The first tile of every row tile (l = 0)
// and any tile that holds a new dominant key take two terms.  The four
// warps of a softmax warpgroup vote per key tile: each posts its warp's
// vote and arrives on an mbarrier after the head terms of its first 32
// keys, and reads the four votes after those of the first 64, so the
// vote's latency hides behind work that both modes share.  One thread tells the
// MMA warp, which then issues the remainder's P V MMAs or not.  Long diffuse
// rows take one term on most tiles: half the P V MMAs and half the P stores
// to tensor memory.
//
// Split rows.  When an interleaved tile has at most 64 real rows, rows
// r + 64 of Q repeat rows r, so lanes r and r + 64 of S hold the same scores
// and their softmax threads compute the same weights.  Lane r writes the head
// term of P and lane r + 64 the remainder, into the same 64 columns: one
// P V pass over 128 keys (8 MMAs, not 16) accumulates both, and the row's
// output is the sum of O's lanes r and r + 64.
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 8.0f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kRows = 128;       // rows per row tile (the MMA's M)
constexpr int kKeys = 128;       // keys per K/V tile (8 pages)
// Warp roles: warps 0 and 1 issue the MMAs of row tiles A and B, warps 2
// and 3 the K and V copies, warps 4-7 and 8-11 are the two softmax
// warpgroups (TMEM lanes are reached by warp index mod 4).
constexpr int kKLoadWarp = 2, kVLoadWarp = 3;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kThreads = 12 * 32;

struct TcParams {
  const uint16_t *q;
  const int32_t *block_table;
  const int32_t *ctx_lens;
  float *out;
  int *status;
  float qscale;     // |scale| * log2 e, at least 1e-30
  uint32_t qsign;   // 0x80008000 when scale < 0 (folded into Q), else 0
  int n_new, n_q_heads, n_kv_heads, group, batch, max_blocks, num_pages;
  // Key-range partitions: n_parts > 1 splits each sequence's keys into
  // ranges of part_tiles key tiles.  With ws set, every CTA writes its rows'
  // partial states (O, m, l) to ws [batch][n_new][n_q_heads][ws_slots]
  // [head_dim + 4] (slot = its range) for a merge instead of O / l to out.
  float *ws;
  int part_tiles, n_parts, ws_slots;
  // shared_ctx >= 0: every query of a sequence attends the same keys
  // 0 .. shared_ctx - 1 (ctx_lens unused, no causal mask): the forks of a
  // shared prefix, queried once for all of them.
  int shared_ctx;
};

// Shared memory (offsets from a 1024-aligned base).  Operand tiles are
// stored as 64-column blocks of [rows][128 B] with the 128-byte swizzle.
template <int D>
struct TcSmem {
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kColBlk = kRows * 128;          // one 64-column block, 128 rows
  static constexpr int kQBytes = (D / 64) * kColBlk;   // one row tile of Q
  static constexpr int kKVBytes = (D / 64) * kColBlk;  // 128 keys x D
  static constexpr int kQ = 0;                         // Q_A, then Q_B
  static constexpr int kK0 = kQ + 2 * kQBytes;
  static constexpr int kV0 = kK0 + kKStages * kKVBytes;
  static constexpr int kBars = kV0 + kVStages * kKVBytes;
  // TMEM address, abort flag, then the P mode of row tiles A and B (1: one
  // term) for the key tile their softmax handed over last
  static constexpr int kSlot = kBars + 48 * 8;
  static constexpr int kML = kSlot + 16;        // interleaved: B's (m, l) per row
  static constexpr int kVote = kML + kRows * 8;  // per softmax warp: one term fits its rows
  static constexpr int kBytes = kVote + 8 * 4;
  // Interleaved key tiles: Q_A only, then the K and V rings.
  static constexpr int kKStagesIl = D == 128 ? 3 : 4;
  static constexpr int kVStagesIl = D == 128 ? 3 : 4;
  static constexpr int kK0Il = kQ + kQBytes;
  static constexpr int kV0Il = kK0Il + kKStagesIl * kKVBytes;
  static_assert(kV0Il + kVStagesIl * kKVBytes <= kBars, "interleaved rings overflow");
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
};

// mbarrier indices.  Stage barriers come in two sets of 4 (stage s < 4):
// full barriers use set 0 alone unless interleaved (then set t mod 2); free
// barriers use set x, the row tile that read the stage.
enum {
  kBarK = 0,        // K stage s landed (TMA transaction count), at 4 set + s
  kBarV = 8,        // V stage s landed
  kBarKFree = 16,   // K stage s read by row tile x's S MMA (commit), at 16 + 4 x + s
  kBarVFree = 24,   // V stage s read by row tile x's P V MMAs, at 24 + 4 x + s
  kBarS = 32,       // S_x of the next key tile in TMEM (commit), per row tile
  kBarP = 34,       // keys [64 h, 64 h + 64) of P_x in TMEM, at 34 + 2 x + h
                    // (one arrival per warp of x's warpgroup)
  kBarO = 38,       // the last P_x V done (commit, once), per row tile
  kBarVZ = 40,      // the last V tile's rows past the final key are cleared
  kBarDrain = 41,   // an MMA warp's own drain on its failure path, per row tile
  kBarVote = 43,    // the four warps of softmax warpgroup x have voted (one
                    // arrival each), per row tile
  kNumBars = 45
};
static_assert(kNumBars <= 48, "barrier space");

// Stage bookkeeping for key tile t in a ring of S stages: its stage, the
// barrier set of its full barrier, and the parity of its use of that
// barrier.  Interleaved, a barrier of set t mod 2 serves every lcm(2, S)-th
// tile.
template <bool IL>
struct Ring {
  int S;
  __device__ __forceinline__ int stage(int t) const { return t % S; }
  __device__ __forceinline__ int full(int t) const { return (IL ? 4 * (t & 1) : 0) + t % S; }
  __device__ __forceinline__ uint32_t parity(int t) const {
    return static_cast<uint32_t>(t / (IL && (S & 1) ? 2 * S : S)) & 1;
  }
};

__device__ __forceinline__ uint32_t swz128(int r, int c) {  // row r, 16-B chunk c < 8
  return r * 128 + (((c & 7) ^ (r & 7)) << 4);
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

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Bounded wait on one mbarrier phase that also gives up once another role has
// raised the abort flag.
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
// Warp-wide form: true only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          volatile int *abort_flag) {
  return __all_sync(kFull, wait_or_abort(bar, parity, abort_flag));
}

__device__ __forceinline__ void raise_abort(int *status, volatile int *abort_flag) {
  record_error(status, PA_ERR_TIMEOUT);
  *abort_flag = 1;
}

// Per-CTA work description shared by all roles.  Key tiles are counted
// from t0, the first tile of the CTA's key range (0 without partitions).
struct TcWork {
  int b, g, hbase, q0;  // batch, kv head, first q head, first query of tile A
  int ctx;              // cached tokens of sequence b
  int part, t0;         // key-range partition, its first key tile
  int qx[2];            // first query of row tiles A and B
  int nq[2];            // real queries in row tiles A and B (B may have none)
  int n_tiles[2];       // key tiles of the range each row tile visits (0: none)
  int kmax;             // last key any row of the CTA sees (absolute)
  int n_kv_tiles;       // key tiles loaded = max(n_tiles), or their sum when il
  bool il;              // interleaved: B has A's rows; tile x takes tiles t = x mod 2
  bool sr;              // split rows (interleaved, <= 64 real rows): rows r + 64 repeat r
};

// Load warps: one copies K, the other V.  Tile t goes into stage t % kStages
// of its ring once the MMAs that read the stage's previous tile have
// completed.  Lane j < 8 copies page j of the tile (one box per 64 columns).
// Page ids come in 32-page windows held one per lane, fetched one window
// ahead and checked when used.  The V warp then clears the rows of the last
// V tile past the final key: P is 0 there, but 0 * (non-finite junk) is NaN
// in the MMA.
template <int D, bool IL>
__device__ __forceinline__ void load_tiles(bool is_v, const CUtensorMap *map, uint32_t sb,
                                           const int32_t *bt_row, int n_pages, const TcWork &w,
                                           int num_pages, int y_page, int *status,
                                           volatile int *abort_flag, int lane) {
  using L = TcSmem<D>;
  const int S = IL ? (is_v ? L::kVStagesIl : L::kKStagesIl) : (is_v ? L::kVStages : L::kKStages);
  const Ring<IL> rg{S};
  const int bar_full = is_v ? kBarV : kBarK, bar_free = is_v ? kBarVFree : kBarKFree;
  const uint32_t ring = sb + (IL ? (is_v ? L::kV0Il : L::kK0Il) : (is_v ? L::kV0 : L::kK0));
  constexpr int kBoxes = D / 64;
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  auto load_window = [&](int win) {
    const int pg = 32 * win + lane;
    return pg < n_pages ? __ldg(bt_row + pg) : 0;  // past the end: page 0, masked
  };
  if (lane == 0) prefetch_tensormap(map);
  const int y_head = w.g * 16;
  int wcur = load_window(w.t0 >> 2), wnext = load_window((w.t0 >> 2) + 1);
  const int n = w.n_kv_tiles;
  int issued = 0;
  bool ok = true;
  for (int t = 0; t < n; ++t) {  // t counts the range's tiles; ta is absolute
    const int ta = w.t0 + t;
    if (t > 0 && (ta & 3) == 0) {  // the tile starts a new 32-page window
      wcur = wnext;
      wnext = load_window((ta >> 2) + 1);
    }
    int idj = __shfl_sync(kFull, wcur, 8 * (ta & 3) + (lane & 7));
    if (lane < 8 && static_cast<unsigned>(idj) >= static_cast<unsigned>(num_pages)) {
      record_error(status, PA_ERR_BAD_BLOCK);
      idj = 0;
    }
    // the stage's previous tile, t - S, must be released by every row tile
    // that used it (interleaved: by row tile (t - S) mod 2 alone)
    if (IL) {
      const int tp = t - S;
      if (tp >= 0) ok = warp_wait(bar(bar_free + 4 * (tp & 1) + rg.stage(tp)), rg.parity(tp), abort_flag);
    } else {
      for (int x = 0; x < 2 && ok && t >= S; ++x)
        if (t - S < w.n_tiles[x])
          ok = warp_wait(bar(bar_free + 4 * x + t % S), ((t / S) - 1) & 1, abort_flag);
    }
    if (!ok) break;
    const uint32_t full = bar(bar_full + rg.full(t));
    const uint32_t dst0 = ring + rg.stage(t) * L::kKVBytes;
    if (lane == 0) mbar_arrive_expect_tx(full, L::kKVBytes);
    __syncwarp();
    if (lane < 8) {
#pragma unroll
      for (int bx = 0; bx < kBoxes; ++bx)
        tma_load_2d(dst0 + bx * L::kColBlk + lane * 2048, map, bx * 64, idj * y_page + y_head,
                    full);
    }
    ++issued;
  }
  const int key0 = (w.t0 + n - 1) * kKeys;
  const int first = w.kmax - key0 + 1;  // first row of the last V tile no row sees
  if (is_v && ok && n > 0 && first < kKeys) {
    const int t = n - 1;
    if ((ok = warp_wait(bar(kBarV + rg.full(t)), rg.parity(t), abort_flag))) {
      const uint32_t vst = ring + rg.stage(t) * L::kKVBytes;
      for (int e = lane; e < (kKeys - first) * (D / 8); e += 32) {
        const int rr = first + e / (D / 8), c = e % (D / 8);
        st_shared_v4(vst + (c >> 3) * L::kColBlk + swz128(rr, c), 0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();  // generic stores -> read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarVZ));
    }
  }
  if (!ok) {
    if (lane == 0) raise_abort(status, abort_flag);
    // Copies in flight still land in shared memory: wait for them.
    for (int t = issued > S ? issued - S : 0; t < issued; ++t)
      mbar_wait(bar(bar_full + rg.full(t)), rg.parity(t));
  }
}

// MMA warps: warp x (lane 0) issues row tile x's MMAs,
//   S_x(0), then per key tile t:  P_x(t) V_t (two key halves), S_x(t+1)
// S_x(t+1) goes after P_x(t) V_t because it overwrites P_x in TMEM; MMAs of
// one thread run in issue order.  With one issuing warp per row tile the
// tensor pipe takes work from whichever tile is ready, so one tile's
// barrier waits and softmax do not stall the other's MMAs.  Interleaved, the
// j-th key tile of row tile x is t = 2 j + x and both tiles read Q_A.
template <int D, bool BF16, bool IL, bool SR>
__device__ __forceinline__ void mma_tiles(int x, uint32_t sb, uint32_t tmem, const TcWork &w,
                                          int *status, volatile int *abort_flag,
                                          const volatile int *mode_x, int lane) {
  using L = TcSmem<D>;
  constexpr int SK = IL ? L::kKStagesIl : L::kKStages, SV = IL ? L::kVStagesIl : L::kVStages;
  const Ring<IL> rk{SK}, rv{SV};
  constexpr int kStep = IL ? 2 : 1;
  constexpr int KSQ = D / 16;
  constexpr uint32_t kIdS = tc::idesc_f16(BF16, kRows, kKeys, false, false);
  constexpr uint32_t kIdO = tc::idesc_f16(BF16, kRows, D, false, true);
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  // Descriptors of this tile's Q and of stage 0; other stages and K steps add
  // their byte offset >> 4 to the address field.
  const uint64_t dq = tc::smem_desc_sw128(sb + L::kQ + (IL ? 0 : x * L::kQBytes), 16, 1024);
  const uint64_t dk0 = tc::smem_desc_sw128(sb + (IL ? L::kK0Il : L::kK0), 16, 1024);
  const uint64_t dv0 = tc::smem_desc_sw128(sb + (IL ? L::kV0Il : L::kV0), L::kColBlk, 1024);
  const uint32_t tSx = tmem + x * kKeys, tOx = tmem + 2 * kKeys + x * D;
  const int n = w.n_kv_tiles, nx = w.n_tiles[x];
  const int last_first = w.kmax - (w.t0 + n - 1) * kKeys + 1;
  const bool cleared = last_first < kKeys;  // the last V tile waits for the clearing

  auto s_mma = [&](int t) {  // S_x = Q_x K_t^T; then K stage t % SK is free for x
    if (lane == 0) {
      const uint64_t dk = dk0 + static_cast<uint64_t>(((t % SK) * L::kKVBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < KSQ; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::kColBlk + (kk & 3) * 32) >> 4);
        tc::mma_f16(tSx, dq + off, dk + off, kIdS, kk > 0);
      }
      tc::commit(bar(kBarS + x));
      tc::commit(bar(kBarKFree + 4 * x + t % SK));
    }
    __syncwarp();
  };
  // O_x += P_x[:, keys of half h] V_t[keys of half h].  P_x in TMEM: head
  // terms in columns 0-63 (two keys per column), remainders in 64-127.
  // Split rows: the remainders are in rows 64-127 of the same columns, so
  // one pass; else one or two passes as the softmax decided for the tile.
  auto pv_mma = [&](int j, int t, int h, int n_ph) {  // the j-th key tile of x is t
    if (lane == 0) {
      const uint64_t dv = dv0 + static_cast<uint64_t>(((t % SV) * L::kKVBytes) >> 4);
      const uint32_t pa = tSx + 32 * h;
#pragma unroll
      for (int ph = 0; ph < 2; ++ph) {
        if (ph >= n_ph) break;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_f16_tmem_a(tOx, pa + 64 * ph + 8 * kk,
                             dv + static_cast<uint64_t>(((4 * h + kk) * 2048) >> 4), kIdO,
                             (j > 0 || h > 0 || ph > 0 || kk > 0) ? 1u : 0u);
      }
      if (h == 1) {
        tc::commit(bar(kBarVFree + 4 * x + t % SV));
        if (j == nx - 1) tc::commit(bar(kBarO + x));
      }
    }
    __syncwarp();
  };

  bool ok = true;
  const int tx = IL ? x : 0;  // x's first key tile
  if (nx > 0 && (ok = warp_wait(bar(kBarK + rk.full(tx)), rk.parity(tx), abort_flag))) {
    tc::fence_after_sync();
    s_mma(tx);
  }
  for (int j = 0; j < nx && ok; ++j) {
    const int t = tx + kStep * j;
    int n_ph = 1;
    for (int h = 0; h < 2 && ok; ++h) {
      if (!(ok = warp_wait(bar(kBarP + 2 * x + h), j & 1, abort_flag))) break;
      if (h == 0) {
        // written before the softmax's first hand-off of this tile (the
        // barrier's acquire makes it visible); rewritten only after S_x of
        // a later tile, which is issued below
        if (!SR) n_ph = *mode_x ? 1 : 2;
        ok = (t == n - 1 && cleared) ? warp_wait(bar(kBarVZ), 0, abort_flag)
                                     : warp_wait(bar(kBarV + rv.full(t)), rv.parity(t), abort_flag);
        if (!ok) break;
      }
      tc::fence_after_sync();
      pv_mma(j, t, h, n_ph);
    }
    const int tn = t + kStep;
    if (ok && j + 1 < nx &&
        (ok = warp_wait(bar(kBarK + rk.full(tn)), rk.parity(tn), abort_flag))) {
      tc::fence_after_sync();
      s_mma(tn);
    }
  }
  if (!ok) {
    if (lane == 0) {
      raise_abort(status, abort_flag);
      tc::commit(bar(kBarDrain + x));  // arrives once every MMA issued so far is done
    }
    __syncwarp();
    mbar_wait(bar(kBarDrain + x), 0);
  }
}

// Named barriers of the softmax warps.  Barrier 1 joins warps 4-11 and
// returns whether any thread passed true; barrier 2 joins warps 4-7.
__device__ __forceinline__ bool softmax_pair_sync_any(bool c) {
  uint32_t any;
  asm volatile(
      "{\n\t.reg .pred q, p;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 256, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(any)
      : "r"(static_cast<uint32_t>(c))
      : "memory");
  return any != 0;
}
__device__ __forceinline__ void softmax_group_sync() {
  asm volatile("bar.sync 2, 128;" ::: "memory");
}
// Softmax warpgroup x (warps 4 + 4 x .. 7 + 4 x): lane l of warp w owns TMEM
// lane r = 32 (w % 4) + l of row tile x, i.e. row rr = r (split rows:
// r mod 64): query qx[x] + rr / GT, head hbase + rr % GT.
template <int D, int GT, bool BF16, bool IL, bool SR>
__device__ __forceinline__ void softmax_tiles(uint32_t sb, uint32_t tmem, const TcParams &p,
                                              const TcWork &w, volatile int *abort_flag,
                                              volatile int *mode_x, volatile int *votes,
                                              float *ml, float *scratch, int x, int warp,
                                              int lane) {
  using L = TcSmem<D>;
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  const int r = ((warp & 3) << 5) + lane, rr = SR ? (r & 63) : r;
  const int qi = rr / GT, hh = rr % GT;
  const bool rem = SR && r >= 64;  // this warp writes the remainder terms
  const int qx0 = w.qx[x];
  const bool shared = p.shared_ctx >= 0;  // every row sees keys < ctx
  const int kmax_x = shared ? w.ctx - 1 : w.ctx + qx0 + w.nq[x] - 1;
  const int lim = shared ? kmax_x : min(w.ctx + qx0 + qi, kmax_x);  // last key row r sees
  const int lim_all = shared ? kmax_x : w.ctx + qx0;  // every row of x sees keys <= this
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tSx = tmem + x * kKeys + lane_base;      // S_x, then P_x
  const uint32_t tOx = tmem + 2 * kKeys + x * D + lane_base;
  const float qs = p.qscale;
  const int nt = w.n_tiles[x];

  bool bad = false;
  float m = -INFINITY;
  float2 lp = make_float2(0.f, 0.f);  // running sums of the even and odd keys
  for (int j = 0; j < nt; ++j) {
    // ping-pong: wait for the other tile's turn before this one (where the
    // other tile has that many key tiles)
    const int jo = j - 1 + x;
    if (jo >= 0 && jo < w.n_tiles[x ^ 1]) {
      if (!warp_wait(bar(kBarP + 2 * (x ^ 1)), jo & 1, abort_flag) ||
          !warp_wait(bar(kBarP + 2 * (x ^ 1) + 1), jo & 1, abort_flag)) {
        bad = true;
        break;
      }
    }
    if (!warp_wait(bar(kBarS + x), j & 1, abort_flag)) {
      bad = true;
      break;
    }
    tc::fence_after_sync();
    uint32_t s[kKeys];
#pragma unroll
    for (int cb = 0; cb < kKeys / 32; ++cb)
      tc::ld32(tSx + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(s + cb * 32));
    tc::wait_ld();

    // ---- mask, max of the raw scores, lazy move of the reference max
    const int key0 = (w.t0 + (IL ? 2 * j + x : j)) * kKeys;
    if (key0 + kKeys - 1 > lim_all) {
      const int last = lim - key0;  // keys past this one are masked for row r
#pragma unroll
      for (int c = 0; c < kKeys; ++c)
        if (c > last) s[c] = __float_as_uint(-INFINITY);
    }
    float t0 = -INFINITY, t1 = -INFINITY, t2 = -INFINITY, t3 = -INFINITY;
#pragma unroll
    for (int c = 0; c < kKeys; c += 8) {
      t0 = max3(t0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
      t1 = max3(t1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
      t2 = max3(t2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
      t3 = max3(t3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
    }
    const float cand = fmaxf(fmaxf(t0, t1), fmaxf(t2, t3)) * qs;
    const bool need = cand > m + kSlack;
    float corr = 1.f;
    if (need) {
      const float mn = fmaxf(m, cand);
      corr = ex2(m - mn);  // 0 while m was still -inf
      m = mn;
      lp = __fmul2_rn(lp, make_float2(corr, corr));
    }
    // ---- this row's vote: one term of P for this key tile if the tile's
    // largest weight 2^(cand - m) is below 1/16 of the weight of the earlier
    // tiles (NaN while m = -inf: two terms); the warpgroup votes below
    const bool fine = 16.f * ex2(cand - m) < lp.x + lp.y;
    const float nm = m == -INFINITY ? 0.f : -m;  // nothing seen yet: weights are 0
    const float2 qs2 = make_float2(qs, qs), nm2 = make_float2(nm, nm);

    auto head = [&](int ch, int k, uint32_t &hi) {  // packed fp32x2: one instruction per pair
      const float2 e = __ffma2_rn(make_float2(__uint_as_float(s[32 * ch + 2 * k]),
                                              __uint_as_float(s[32 * ch + 2 * k + 1])),
                                  qs2, nm2);
      const float2 pp = make_float2(ex2(e.x), ex2(e.y));
      lp = __fadd2_rn(lp, pp);
      hi = pack2<BF16>(pp.x, pp.y);
      return pp;
    };
    auto rem_of = [&](float2 pp, uint32_t hi) {  // the remainder p - head, exact before rounding
      const float2 d = __ffma2_rn(unpack2<BF16>(hi), make_float2(-1.f, -1.f), pp);
      return pack2<BF16>(d.x, d.y);
    };
    // After chunk ch's stores: the O rescale (once per tile, before the
    // first P V of the tile) and the hand-off of each 64-key half.
    auto after_chunk = [&](int ch) {
      if (ch == 1 && j > 0 && __any_sync(kFull, need)) {
        // the max moved: rescale this row of O_x before the first P V of
        // this tile (P_x V_{j-1} has completed: S_x was issued after it)
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          tc::ld32(tOx + cb * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
          tc::st32(tOx + cb * 32, o);
        }
      }
      if (ch & 1) {
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarP + 2 * x + (ch >> 1)));  // one arrival per warp
      }
    };
    // ---- P = 2^(s qs - m) over the S columns, keys 32 ch .. 32 ch + 31 per
    // chunk; each half of the keys is handed to the MMA warp as soon as it
    // is written.  Kind 0: head + remainder, 1: one term, 2: split rows (the
    // warps of rows 0-63 store the head term, those of rows 64-127 the
    // remainder, into the same columns).  Each kind is its own unrolled loop.
    auto tile_p = [&](auto kind, int ch0) {  // chunks ch0 .. 3
      constexpr int K = decltype(kind)::value;
#pragma unroll
      for (int ch = 0; ch < kKeys / 32; ++ch) {
        if (ch < ch0) continue;
        uint32_t phi[16], plo[16];
        if constexpr (K == 2) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 pp = head(ch, k, phi[k]);
            if (rem) plo[k] = rem_of(pp, phi[k]);
          }
          tc::st16(tSx + 16 * ch, rem ? plo : phi);
        } else if constexpr (K == 1) {
#pragma unroll
          for (int k = 0; k < 16; ++k) head(ch, k, phi[k]);
          tc::st16(tSx + 16 * ch, phi);
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) plo[k] = rem_of(head(ch, k, phi[k]), phi[k]);
          tc::st16(tSx + 16 * ch, phi);
          tc::st16(tSx + 64 + 16 * ch, plo);
        }
        after_chunk(ch);
      }
    };
    if constexpr (SR) {
      tile_p(std::integral_constant<int, 2>{}, 0);
    } else {
      // Keys 0-63: head terms first (both modes need them; the weights stay
      // in s for a remainder), the warp's vote posted after the first 32
      // and the four votes read after all 64, so that neither the vote's
      // latency nor a branch on its outcome holds up the exponentials.
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t phi[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 pp = head(ch, k, phi[k]);
          s[32 * ch + 2 * k] = __float_as_uint(pp.x);
          s[32 * ch + 2 * k + 1] = __float_as_uint(pp.y);
        }
        tc::st16(tSx + 16 * ch, phi);
        if (ch == 0) {
          const bool wfine = __all_sync(kFull, fine);
          if (lane == 0) {
            votes[4 * x + (warp & 3)] = wfine ? 1 : 0;
            mbar_arrive(bar(kBarVote + x));
          }
        }
      }
      if (!warp_wait(bar(kBarVote + x), j & 1, abort_flag)) {
        bad = true;
        if (lane == 0) raise_abort(p.status, abort_flag);
        break;
      }
      const bool one = votes[4 * x] & votes[4 * x + 1] & votes[4 * x + 2] & votes[4 * x + 3];
      if ((warp & 3) == 0 && lane == 0) *mode_x = one ? 1 : 0;
      if (!one) {  // remainders of keys 0-63 from the kept weights
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t plo[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 pp = make_float2(__uint_as_float(s[32 * ch + 2 * k]),
                                          __uint_as_float(s[32 * ch + 2 * k + 1]));
            plo[k] = rem_of(pp, pack2<BF16>(pp.x, pp.y));
          }
          tc::st16(tSx + 64 + 16 * ch, plo);
        }
      }
      after_chunk(1);  // the O rescale, then keys 0-63 go to the MMA warp
      if (one)
        tile_p(std::integral_constant<int, 1>{}, 2);
      else
        tile_p(std::integral_constant<int, 0>{}, 2);
    }
  }
  tc::wait_st();
  if (nt == 0) return;
  if (!bad) bad = !warp_wait(bar(kBarO + x), 0, abort_flag);
  if (bad && lane == 0) raise_abort(p.status, abort_flag);
  float l = lp.x + lp.y, ca = 1.f, cb = 0.f;
  if (IL) {
    // both warpgroups always meet here, failed or not, and all of them take
    // the same decision
    if (x == 1) {
      ml[2 * r] = m;
      ml[2 * r + 1] = l;
    }
    if (softmax_pair_sync_any(bad || *abort_flag) || x == 1) return;
    const float mb = ml[2 * r], lb = ml[2 * r + 1];
    const float mn = fmaxf(m, mb);
    if (mn != -INFINITY) {  // else no key reached this row: O and l stay 0
      ca = ex2(m - mn);
      cb = ex2(mb - mn);
    }
    m = mn;
    l = ca * l + cb * lb;
  } else if (bad) {
    return;
  }
  tc::fence_after_sync();

  // ---- O / l for this row, or the row's partial state for this key range
  const bool split = p.ws != nullptr;
  const float inv = split ? 1.f : (l > 0.f ? 1.f / l : 0.f);
  const size_t row =
      (static_cast<size_t>(w.b) * p.n_new + qx0 + qi) * p.n_q_heads + w.hbase + hh;
  float *dst = split ? p.ws + (row * p.ws_slots + w.part) * (D + 4) : p.out + row * D;
  // columns 32 c .. 32 c + 31 of this lane's O (interleaved: both tiles' merged)
  auto load_o = [&](int c, uint32_t (&o)[32]) {
    tc::ld32(tOx + c * 32, o);
    if (IL) {  // O_A 2^(m_A - m) + O_B 2^(m_B - m); O_B is D columns to the right
      uint32_t ob[32];
      tc::ld32(tOx + D + c * 32, ob);
      tc::wait_ld();
#pragma unroll
      for (int k = 0; k < 32; ++k)
        o[k] = __float_as_uint(ca * __uint_as_float(o[k]) + cb * __uint_as_float(ob[k]));
    } else {
      tc::wait_ld();
    }
  };
  // Split rows: lane rr + 64 hands its part of O to lane rr through shared
  // memory (Q_A's space, free once every S MMA has completed); float4 k of
  // row rr sits at slot k ^ (rr mod 8).
  auto scr = [&](int k4) { return scratch + rr * D + ((k4 ^ (rr & 7)) << 2); };
  if (SR) {
    if (rem) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        load_o(c, o);
#pragma unroll
        for (int k = 0; k < 32; k += 4)
          *reinterpret_cast<float4 *>(scr(c * 8 + k / 4)) =
              make_float4(__uint_as_float(o[k]), __uint_as_float(o[k + 1]),
                          __uint_as_float(o[k + 2]), __uint_as_float(o[k + 3]));
      }
    }
    softmax_group_sync();  // warps 4-7: all reach it (the decision above is shared)
    if (rem) return;
  }
  if (split && qi < w.nq[x])
    *reinterpret_cast<float2 *>(dst + D) = make_float2(m * kLn2, l);  // natural-log m
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    load_o(c, o);
    if (SR) {
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 t = *reinterpret_cast<const float4 *>(scr(c * 8 + k / 4));
        o[k] = __float_as_uint(__uint_as_float(o[k]) + t.x);
        o[k + 1] = __float_as_uint(__uint_as_float(o[k + 1]) + t.y);
        o[k + 2] = __float_as_uint(__uint_as_float(o[k + 2]) + t.z);
        o[k + 3] = __float_as_uint(__uint_as_float(o[k + 3]) + t.w);
      }
    }
    if (qi < w.nq[x]) {
#pragma unroll
      for (int k = 0; k < 32; k += 4)
        *reinterpret_cast<float4 *>(dst + c * 32 + k) =
            make_float4(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                        __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
    }
  }
}

template <int D, int GT, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const TcParams p) {
  using L = TcSmem<D>;
  constexpr int BQ = kRows / GT;  // queries per row tile

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + L::kBars + 8 * i; };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_release();
  griddep_wait();  // inputs may come from the previous kernel in the stream

  TcWork w;
  const int n_sub = p.group / GT;
  w.b = blockIdx.z;
  w.g = blockIdx.y / n_sub;
  w.hbase = w.g * p.group + (blockIdx.y % n_sub) * GT;
  w.part = blockIdx.x % p.n_parts;
  w.q0 = (blockIdx.x / p.n_parts) * 2 * BQ;
  w.t0 = w.part * p.part_tiles;  // part_tiles = every tile when n_parts is 1
  const bool shared = p.shared_ctx >= 0;
  const int maxT = p.max_blocks * 16;
  int ctx;
  if (shared) {
    ctx = p.shared_ctx;  // checked against the table on the host (at least 1 key)
  } else {
    ctx = p.ctx_lens[w.b];
    if (ctx < 0 || ctx + p.n_new > maxT) {
      if (tid == 0) record_error(p.status, PA_ERR_BAD_CTX);
      ctx = max(0, min(ctx, maxT - p.n_new));
    }
  }
  w.ctx = ctx;
  w.kmax = -1;
  for (int x = 0; x < 2; ++x) {
    w.nq[x] = max(0, min(BQ, p.n_new - (w.q0 + x * BQ)));
    // last key a row of x sees
    const int kx = shared ? ctx - 1 : ctx + w.q0 + x * BQ + w.nq[x] - 1;
    const int t_end = min(kx / kKeys + 1, w.t0 + p.part_tiles);
    w.n_tiles[x] = w.nq[x] > 0 ? max(0, t_end - w.t0) : 0;
    if (w.nq[x] > 0) w.kmax = max(w.kmax, kx);
  }
  w.n_kv_tiles = max(w.n_tiles[0], w.n_tiles[1]);
  // B idle and A with at least two key tiles: interleave (B gets the odd ones)
  w.il = w.nq[1] == 0 && w.n_tiles[0] >= 2;
  w.qx[0] = w.q0;
  w.qx[1] = w.il ? w.q0 : w.q0 + BQ;
  if (w.il) {
    w.nq[1] = w.nq[0];
    w.n_tiles[1] = w.n_tiles[0] / 2;
    w.n_tiles[0] -= w.n_tiles[1];
  }
  w.sr = w.il && w.nq[0] * GT <= kRows / 2;
  const int n_pages = (ctx + (shared ? 0 : p.n_new) + 15) >> 4;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kSlot + 4);
  volatile int *mode = reinterpret_cast<volatile int *>(smem + L::kSlot + 8);  // [2]
  volatile int *votes = reinterpret_cast<volatile int *>(smem + L::kVote);     // [2][4]

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(bar(i), ((i >= kBarP && i < kBarP + 4) || i >= kBarVote) ? 4 : 1);
    *abort_flag = 0;
    mode[0] = mode[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // S_A: columns 0-127, S_B: 128-255, O_A: 256 .. 256+D-1, O_B: 256+D .. 256+2D-1
    tc::alloc(sb + L::kSlot, 512);
    tc::relinquish();
  }
  // Q tiles: row r of tile x = query qx[x] + r / GT, head hbase + r % GT
  // (zeros past the chunk's end; the sign of a negative scale folded in).
  // Interleaved, only Q_A is loaded: Q_B's space belongs to the K ring.
  if (warp >= kSoftmaxWarp0 && !(w.il && warp >= kSoftmaxWarp0 + 4)) {
    // A thread's loads all go out before its first store (each store is a
    // compiler barrier), so they cost one memory round trip, not sixteen.
    const int x = (warp - kSoftmaxWarp0) >> 2;
    constexpr int kPer = kRows * (D / 8) / 128;  // 16-byte chunks per thread
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = (tid & 127) + 128 * k, r = e / (D / 8), c = e % (D / 8);
      const int rr = w.sr ? (r & 63) : r;  // split rows: rows 64-127 repeat 0-63
      const int qi = rr / GT, hh = rr % GT;
      v[k] = make_uint4(0, 0, 0, 0);
      if (qi < w.nq[x])
        v[k] = __ldg(reinterpret_cast<const uint4 *>(
            p.q +
            ((static_cast<size_t>(w.b) * p.n_new + w.qx[x] + qi) * p.n_q_heads + w.hbase +
             hh) * D + c * 8));
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = (tid & 127) + 128 * k, r = e / (D / 8), c = e % (D / 8);
      st_shared_v4(sb + L::kQ + x * L::kQBytes + (c >> 3) * L::kColBlk + swz128(r, c),
                   v[k].x ^ p.qsign, v[k].y ^ p.qsign, v[k].z ^ p.qsign, v[k].w ^ p.qsign);
    }
    fence_proxy_async_smem();  // generic stores -> read by the tensor cores
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kSlot);

  if (warp == kKLoadWarp || warp == kVLoadWarp) {
    const bool is_v = warp == kVLoadWarp;
    const int32_t *bt_row = p.block_table + static_cast<size_t>(w.b) * p.max_blocks;
    if (w.il)
      load_tiles<D, true>(is_v, is_v ? &vmap : &kmap, sb, bt_row, n_pages, w, p.num_pages,
                          p.n_kv_heads * 16, p.status, abort_flag, lane);
    else
      load_tiles<D, false>(is_v, is_v ? &vmap : &kmap, sb, bt_row, n_pages, w, p.num_pages,
                           p.n_kv_heads * 16, p.status, abort_flag, lane);
  } else if (warp < 2) {
    const volatile int *mode_x = mode + warp;
    if (w.sr)
      mma_tiles<D, BF16, true, true>(warp, sb, tmem, w, p.status, abort_flag, mode_x, lane);
    else if (w.il)
      mma_tiles<D, BF16, true, false>(warp, sb, tmem, w, p.status, abort_flag, mode_x, lane);
    else
      mma_tiles<D, BF16, false, false>(warp, sb, tmem, w, p.status, abort_flag, mode_x, lane);
  } else if (warp >= kSoftmaxWarp0) {
    float *ml = reinterpret_cast<float *>(smem + L::kML);
    float *scratch = reinterpret_cast<float *>(smem + L::kQ);
    const int x = (warp - kSoftmaxWarp0) >> 2;
    if (w.sr)
      softmax_tiles<D, GT, BF16, true, true>(sb, tmem, p, w, abort_flag, mode + x, votes, ml,
                                             scratch, x, warp, lane);
    else if (w.il)
      softmax_tiles<D, GT, BF16, true, false>(sb, tmem, p, w, abort_flag, mode + x, votes, ml,
                                              scratch, x, warp, lane);
    else
      softmax_tiles<D, GT, BF16, false, false>(sb, tmem, p, w, abort_flag, mode + x, votes, ml,
                                               scratch, x, warp, lane);
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
  static ContextCache<bool> smem_set;  // contexts where the limit is set
  if (set_smem_limit(kern, L::kAlloc, smem_set) != PA_OK) return PA_ERR_CUDA;
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
  // The kernel takes the maximum of the raw scores, so it needs a positive
  // factor: a negative scale flips the sign of Q instead (exact in 16 bits),
  // and a zero scale becomes a factor small enough that every weight is 1.
  p.qscale = fmaxf(fabsf(a.scale) * kLog2e, 1e-30f);
  p.qsign = a.scale < 0.f ? 0x80008000u : 0u;
  p.n_new = a.n_new;
  p.n_q_heads = a.n_q_heads;
  p.n_kv_heads = a.n_kv_heads;
  p.group = a.n_q_heads / a.n_kv_heads;
  p.batch = a.batch;
  p.max_blocks = a.max_blocks;
  p.num_pages = a.num_pages;
  p.ws = a.workspace;
  p.n_parts = a.n_parts > 1 ? a.n_parts : 1;
  p.part_tiles = a.n_parts > 1 ? a.part_tokens / kKeys : (a.max_blocks * 16 + kKeys - 1) / kKeys;
  p.ws_slots = a.ws_slots > 0 ? a.ws_slots : p.n_parts;
  p.shared_ctx = a.shared_ctx;
  constexpr int BQ = kRows / GT;
  const dim3 grid(((a.n_new + 2 * BQ - 1) / (2 * BQ)) * p.n_parts,
                  a.n_kv_heads * (p.group / GT), a.batch);
  if (launch_pdl(kern, grid, dim3(kThreads), L::kAlloc, stream, kmap, vmap, p) != cudaSuccess)
    return PA_ERR_CUDA;
  if (p.n_parts > 1 && a.merge)
    return launch_merge_rows(a.workspace, a.ctx_lens, a.out, a.status, a.batch, a.n_q_heads,
                             D, p.n_parts, a.part_tokens, a.n_new, stream);
  return PA_OK;
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
