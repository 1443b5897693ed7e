// pa_decode.cu -- decode-step paged GQA attention for sm_103a.
//
// Computes, per sequence b and query head h, o = softmax(q K^T * scale) V
// over the sequence's cached tokens (ch. 19 "推理系统与性能工程", 19.4.1),
// evaluated page by page with the online-softmax recurrence of 19.6.2
// (running max m, running sum l, unnormalised O).
//
// Work decomposition.  One CTA handles one (sequence, kv head, head tile,
// key range): the GT query heads of a head tile share every K/V page it reads
// (GQA reuse, "吞吐与延迟的系统模型" section 5: the kernel must reuse the shared
// KV for the low-byte bound to hold).  Its NW warps take the range's pages
// round robin (one partition per CTA), or each warp owns whole consecutive
// partitions (short partitions).  Each warp feeds itself: it keeps S pages in
// flight in its own ring of shared-memory stages, filled by 2-D TMA loads
// (128-byte swizzle) that complete on one mbarrier per stage, and issues the
// load for page i+S as soon as page i has been consumed.  No warp waits for
// another until the range's end, where the warps' (m, l, O) states are merged
// in shared memory with the exponent law of 19.6.2.  A sequence cut over
// several CTAs leaves one partial state per CTA; the last CTA of its
// (sequence, head tile) to finish (an arrival counter) merges them all with
// the same law, so no second kernel waits for the whole grid.  (When one CTA
// holds all of a sequence's partitions, its warps write each partition's
// state and the CTA folds them itself.)
//
// Per-page math, chosen by the group tile:
//  * GT = 1 (MHA): CUDA cores.  Score phase lane = (token, half of head_dim):
//    the swizzled tile lets 16 lanes read 16 different K rows without bank
//    conflicts while sharing each q element; value phase lane = head_dim/32
//    output dims.  Packed fp32x2 FMAs.
//  * GT >= 2 (GQA): the group's q K^T (GT heads x 16 keys x head_dim) and
//    P V are dense contractions, so they run on the tensor cores as warp-level
//    mma.sync m16n8k16 with the heads as rows (padded to 16).  K and V
//    fragments come straight from the swizzled page tiles with ldmatrix; q
//    stays in registers.  On CUDA cores every lane would re-read all GT q rows
//    from shared memory for every page, which made that path shared-memory
//    bound at GT = 8; this way shared-memory traffic is the K/V bytes alone.
//    P enters P V as two 16-bit terms (head + remainder) so the weights keep
//    ~16 significant bits.
//
// Scores are kept in log2 units (scale * log2 e folded in), so e^(s - m) is
// one ex2.  The running max is only moved when a score exceeds it by more than
// kRescaleSlack (a warp vote decides); between moves the weights e^(s - m)
// stay <= 2^kRescaleSlack.  The rescale is exact whatever reference max is
// used, because O and l share it (19.6.2's argument).
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
  float *ws;   // split: partial states [B][Hq][n_parts][D + 4]
  int *ctr;    // split: arrivals per (sequence, head tile), zero at launch
  int *status;
  float qscale;  // scale * log2(e)
  int n_q_heads, n_kv_heads, group, batch, max_blocks, num_pages;
  int part_pages, n_parts;
  int warp_parts;  // > 0: each warp owns this many whole partitions
  int sink, window;  // window >= 0: only the first `sink` and the last
                     // `window` keys of each sequence are attended
  // Single pass only: with part set, each row's state (O unnormalised,
  // m in natural-log units, l) goes to slot part_slot of part
  // [row][part_stride][D + 4] instead of O / l to out (the own keys of a
  // cascade decode, merged with the shared prefix's states afterwards).
  float *part;
  int part_stride, part_slot;
  // Fused append (k_new set): the step's token of sequence b sits at
  // position ctx_lens[b] - 1; its rows k_new/v_new [B][Hkv][D] are written
  // into the cache at that position, and attended from there.
  const uint16_t *k_new, *v_new;
  uint16_t *k_cache, *v_cache;
};

// The keys a sequence's query attends, as a list of virtual pages.  Without
// a window every page 0 .. ceil(T/16) - 1 in order.  With an attention sink
// of S keys and a window of W keys (S + W < T): the sink pages
// 0 .. ceil(S/16) - 1, then the window pages floor((T-W)/16) .. ceil(T/16) - 1;
// a page holding both the sink's end and the window's start appears twice,
// each time with its own key range.  Virtual page v covers keys
// [16 lp + lo, 16 lp + hi) of logical page lp.
struct KeySet {
  int T, n_s, s_end, wf, w_lo, n_v;
  __device__ void init(int T_, int sink, int window) {
    T = T_;
    if (window < 0 || sink + window >= T) {  // every key
      n_s = n_v = (T + 15) >> 4;
      s_end = T;
      wf = 0;
      w_lo = T;
    } else {
      s_end = sink;
      n_s = (sink + 15) >> 4;
      w_lo = T - window;
      wf = w_lo >> 4;
      n_v = n_s + (window > 0 ? ((T + 15) >> 4) - wf : 0);
    }
  }
  __device__ int logical(int v) const { return v < n_s ? v : wf + (v - n_s); }
  __device__ void range(int v, int &lo, int &hi) const {
    if (v < n_s) {
      lo = 0;
      hi = min(16, s_end - 16 * v);
    } else {
      const int lp = wf + (v - n_s);
      lo = max(0, w_lo - 16 * lp);
      hi = min(16, T - 16 * lp);
    }
  }
};

// Shared-memory plan of one CTA.
template <int D, int GT, int NW, int S, bool MMA>
struct DecodeSmem {
  static constexpr int kBoxBytes = 16 * 128;  // one TMA box: 16 rows x 64 elems
  static constexpr int kBoxes = D / 64;
  static constexpr int kPageBytes = kBoxes * kBoxBytes;  // K (or V) of one page
  static constexpr int kStageBytes = 2 * kPageBytes;     // K tile then V tile
  static constexpr int kStages = NW * S;
  static constexpr int kQStride = D + 8;  // CUDA-core path: floats per q row
  // q: fp32 rows (CUDA cores) or a swizzled 16-row bf16/fp16 tile (MMA)
  static constexpr int kQBytes = MMA ? 16 * D * 2 : GT * kQStride * 4;
  static constexpr int kPBytes = MMA ? 0 : NW * GT * 16 * 4;
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kBarOff = kPOff + kPBytes;
  static constexpr int kBytes = kBarOff + kStages * 8;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-B alignment
  static constexpr int kMergeFloats = NW * GT * (D + 2);
  static_assert(kMergeFloats * 4 <= kQOff, "merge area must fit in the stages");
  static_assert(kStageBytes % 1024 == 0, "swizzled boxes need 1024-B alignment");
};

// Byte offset of 16-byte chunk c (0 .. D/8-1) of row r in a tile stored as
// 64-column boxes of `box_rows` rows with the TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int r, int c, int box_rows) {
  return (c >> 3) * (box_rows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// One warp's ring of S page stages and the page ids that feed it.  Chunk i
// of the warp is logical block first + stride * i of the sequence (stride NW
// when the CTA's warps share a partition, 1 when a warp owns whole ones).
template <int D, int NW, int S>
struct PageRing {
  static constexpr int kBoxBytes = 16 * 128;
  static constexpr int kBoxes = D / 64;
  static constexpr int kPageBytes = kBoxes * kBoxBytes;
  static constexpr int kStageBytes = 2 * kPageBytes;
  uint32_t stage0, bar0;
  const int32_t *bt_row;
  int *status;
  int first, stride, n_i, num_pages, y_page, y_head;
  int ids_cur, ids_nxt;
  KeySet ks;  // chunk i is virtual page first + stride * i of this key set
  // Fused append: logical page patch_lp (-1: none), row patch_row gets the
  // step's token; lane l < 16 holds 16-byte chunk l of its K row, lane
  // 16 + l chunk l of its V row.
  int patch_lp, patch_row;
  uint4 patch_val;

  // The raw table entry; checked only when it is used, so the load's latency
  // is hidden behind the 32 chunks that come first.
  __device__ int fetch_id(int i) {
    return i < n_i ? __ldg(bt_row + ks.logical(first + stride * i)) : 0;
  }
  // Lane j holds the page of chunk 32k + j; the next 32 are fetched early.
  __device__ void start(int lane) {
    ids_cur = fetch_id(lane);
    ids_nxt = fetch_id(32 + lane);
  }
  __device__ int page(int i) const { return first + stride * i; }
  __device__ uint32_t stage(int i) const { return stage0 + (i % S) * kStageBytes; }
  __device__ uint32_t bar(int i) const { return bar0 + 8 * (i % S); }
  __device__ uint32_t parity(int i) const { return (i / S) & 1; }
  // Called by the whole warp with i = 0, 1, 2, ... in order.
  __device__ void issue(int i, int lane, const CUtensorMap *kmap, const CUtensorMap *vmap) {
    if ((i & 31) == 0 && i > 0) {
      ids_cur = ids_nxt;
      ids_nxt = fetch_id(i + 32 + lane);
    }
    int id = __shfl_sync(kFull, ids_cur, i & 31);
    if (lane == 0) {
      if (static_cast<unsigned>(id) >= static_cast<unsigned>(num_pages)) {
        record_error(status, PA_ERR_BAD_BLOCK);
        id = 0;  // read a page that exists; the result is flagged as invalid
      }
      const uint32_t st = stage(i), b = bar(i);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(b, kStageBytes);
      const int y = id * y_page + y_head;
#pragma unroll
      for (int bx = 0; bx < kBoxes; ++bx) {
        tma_load_2d(st + bx * kBoxBytes, kmap, bx * 64, y, b);
        tma_load_2d(st + kPageBytes + bx * kBoxBytes, vmap, bx * 64, y, b);
      }
    }
  }
  // Warp-uniform wait for chunk i; on a timeout, records it, lets the other
  // copies in flight land, and returns false.  The page holding a fused
  // append's token gets the token's rows written over the copy (which may
  // predate their write to the cache); the next copy into the stage is
  // ordered after these stores by issue()'s proxy fence.
  __device__ bool wait(int i, int lane) {
    if (__all_sync(kFull, mbar_wait(bar(i), parity(i)))) {
      if (patch_lp >= 0 && ks.logical(page(i)) == patch_lp) {
        const int c = lane & 15;
        if (c < D / 8) {
          const uint32_t a = stage(i) + (lane >= 16 ? kPageBytes : 0) + swz(patch_row, c, 16);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(patch_val.x),
                       "r"(patch_val.y), "r"(patch_val.z), "r"(patch_val.w)
                       : "memory");
        }
        __syncwarp();
      }
      return true;
    }
    if (lane == 0) record_error(status, PA_ERR_TIMEOUT);
    for (int j = i + 1; j < n_i && j < i + S; ++j) mbar_wait(bar(j), parity(j));
    return false;
  }
};

// ---------------------------------------------------------------------------
// CUDA-core page loop (GT = 1, or any GT): per-warp (m, l, O) in registers.
// Chunks [i_begin, i_end) of the warp's ring; false if a wait ran out.
template <int D, int GT, bool BF16, int NW, int S, class Ring>
__device__ __forceinline__ bool pages_cuda_core(Ring &ring, int i_begin, int i_end,
                                                const CUtensorMap *kmap,
                                                const CUtensorMap *vmap,
                                                const float *q_s, float *p_s, int T,
                                                int lane, float (&m)[GT],
                                                float (&lsum)[GT],
                                                float2 (&O2)[GT][D / 64]) {
  constexpr int DPL = D / 32;
  constexpr int HALF = D / 2;
  constexpr int CPH = HALF / 8;
  constexpr int QS = D + 8;
  const int tok = lane & 15, hf = lane >> 4;
  const uint32_t k_off = (D == 128 ? hf * Ring::kBoxBytes : 0) + tok * 128;
  const uint32_t v_off = Ring::kPageBytes +
                         (D == 128 ? (lane >> 4) * Ring::kBoxBytes + ((lane & 1) << 3)
                                   : ((lane & 3) << 2));
  const int v_chunk = (D == 128) ? ((lane & 15) >> 1) : (lane >> 2);

  bool ok = true;
  for (int i = i_begin; i < i_end; ++i) {
    if (!ring.wait(i, lane)) { ok = false; break; }
    const uint32_t st = ring.stage(i);
    int lo, valid;  // keys [lo, valid) of the page are attended
    ring.ks.range(ring.page(i), lo, valid);

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
          const float *qh = q_s + h * QS + hf * (HALF + 4) + j * 8;
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
        sc[h] = (tok >= lo && tok < valid) ? v : -INFINITY;
      }
    }

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

    const uint32_t vrow = st + v_off;
    auto pv = [&](int t, const float(&pw)[GT]) {
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
    if (lo == 0 && valid == 16) {
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
      // V rows outside the attended keys are never read.
      for (int t = lo; t < valid; ++t) {
        float pw[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) pw[h] = p_s[h * 16 + t];
        pv(t, pw);
      }
    }
    __syncwarp();
    if (i + S < ring.n_i) ring.issue(i + S, lane, kmap, vmap);
  }
#pragma unroll
  for (int h = 0; h < GT; ++h) {  // each token was counted once per half-warp
    float v = lsum[h];
    v += __shfl_xor_sync(kFull, v, 8);
    v += __shfl_xor_sync(kFull, v, 4);
    v += __shfl_xor_sync(kFull, v, 2);
    v += __shfl_xor_sync(kFull, v, 1);
    lsum[h] = v;
  }
  return ok;
}

// ---------------------------------------------------------------------------
// Tensor-core page loop (GT >= 2).  Row r = lane / 4 of the score
// accumulators is query head r of the tile (rows >= GT are padding); this
// lane holds keys k0, k0+1, k0+8, k0+9 of the page (k0 = 2 * (lane % 4)).
// In P V the A operand's rows 0-7 carry the 16-bit head terms of P and rows
// 8-15 (padding in S) the remainder terms, so one MMA does both: o[n][0..1]
// accumulate head r's output dims 8n + k0, 8n + k0 + 1 from the head terms,
// o[n][2..3] the same dims from the remainders; the two are summed when the
// state leaves registers.
template <int D, int GT, bool BF16, int NW, int S, class Ring>
__device__ __forceinline__ bool pages_mma(Ring &ring, int i_begin, int i_end,
                                          const CUtensorMap *kmap,
                                          const CUtensorMap *vmap, uint32_t qs,
                                          float qscale, int T, int lane, float &m_r,
                                          float &l_r, float (&o)[D / 8][4]) {
  constexpr int KS = D / 16;
  constexpr int NT = D / 8;
  uint32_t qa[KS][4];
  {
    const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
      ldsm_x4(qs + swz(r, 2 * kk + (lane >> 4), 16), qa[kk][0], qa[kk][1], qa[kk][2],
              qa[kk][3]);
  }
  const bool real = (lane >> 2) < GT;
  const int k0 = 2 * (lane & 3);
  const int rk = ((lane >> 4) << 3) + (lane & 7);       // K ldmatrix row
  const int rv = (lane & 7) + (((lane >> 3) & 1) << 3);  // V ldmatrix row

  bool ok = true;
  for (int i = i_begin; i < i_end; ++i) {
    if (!ring.wait(i, lane)) { ok = false; break; }
    const uint32_t st = ring.stage(i);
    int lo, valid;  // keys [lo, valid) of the page are attended
    ring.ks.range(ring.page(i), lo, valid);
    if (valid < 16) {
      // V rows past the attended keys may hold non-finite junk (past the
      // sequence end), and 0 * inf is NaN inside the MMA: clear them in the
      // stage (the next TMA overwrites it).
      const int n = (16 - valid) * (D / 8);
      for (int e = lane; e < n; e += 32) {
        const int r = valid + e / (D / 8), c = e % (D / 8);
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                         st + Ring::kPageBytes + swz(r, c, 16)),
                     "r"(0));
      }
      fence_proxy_async_smem();
      __syncwarp();
    }

    float sacc[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(st + swz(rk, 2 * kk + ((lane >> 3) & 1), 16), b0, b1, b2, b3);
      mma16816<BF16>(sacc[0], qa[kk], b0, b1);
      mma16816<BF16>(sacc[1], qa[kk], b2, b3);
    }
    float s[4] = {sacc[0][0] * qscale, sacc[0][1] * qscale, sacc[1][0] * qscale,
                  sacc[1][1] * qscale};
    const int keys[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      s[j] = (real && keys[j] >= lo && keys[j] < valid) ? s[j] : -INFINITY;
    const float tmax = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
    if (__any_sync(kFull, tmax > m_r + kRescaleSlack)) {
      float mt = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 1));
      mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
      const float mn = fmaxf(m_r, mt);
      const float c = mn == -INFINITY ? 1.f : ex2(m_r - mn);
      m_r = mn;
      l_r *= c;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= c;
        o[n][1] *= c;
        o[n][2] *= c;
        o[n][3] *= c;
      }
    }
    float p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) p[j] = real ? ex2(s[j] - m_r) : 0.f;
    l_r += (p[0] + p[1]) + (p[2] + p[3]);
    const uint32_t h01 = pack2<BF16>(p[0], p[1]), h89 = pack2<BF16>(p[2], p[3]);
    const float2 r01 = unpack2<BF16>(h01), r89 = unpack2<BF16>(h89);
    // rows 0-7: head terms, rows 8-15: remainders of the same weights
    const uint32_t pa[4] = {h01, pack2<BF16>(p[0] - r01.x, p[1] - r01.y), h89,
                            pack2<BF16>(p[2] - r89.x, p[3] - r89.y)};
#pragma unroll
    for (int nn = 0; nn < NT / 2; ++nn) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(st + Ring::kPageBytes + swz(rv, 2 * nn + (lane >> 4), 16), b0, b1, b2, b3);
      mma16816<BF16>(o[2 * nn], pa, b0, b1);
      mma16816<BF16>(o[2 * nn + 1], pa, b2, b3);
    }
    __syncwarp();
    if (i + S < ring.n_i) ring.issue(i + S, lane, kmap, vmap);
  }
  l_r += __shfl_xor_sync(kFull, l_r, 1);
  l_r += __shfl_xor_sync(kFull, l_r, 2);
  return ok;
}

// One CTA holds every partition of its (sequence, head tile), and its warps
// have written their partitions' states to the workspace: after a barrier the
// CTA folds partitions 0 .. n_valid - 1 of its GT rows into the output (the
// exponent law of 19.6.2).
template <int D, int GT, int NW>
__device__ __forceinline__ void merge_own_partitions(const DecodeParams &p, size_t row0,
                                                     int n_valid, int tid) {
  __syncthreads();
  constexpr int Q4 = D / 4;
  for (int e = tid; e < GT * Q4; e += NW * 32) {
    const float *base = p.ws + (row0 + e / Q4) * p.n_parts * (D + 4);
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < n_valid; ++c) {
      const float *sp = base + static_cast<size_t>(c) * (D + 4);
      const float2 ml = *reinterpret_cast<const float2 *>(sp + D);
      const float4 o4 = reinterpret_cast<const float4 *>(sp)[e % Q4];
      if (ml.y > 0.f) {  // a partition whose keys all had weight 0 adds nothing
        const float mp = ml.x * kLog2e, mn = fmaxf(m, mp);
        const float a = ex2(m - mn), f = ex2(mp - mn);  // a = 0 at m = -inf
        acc = make_float4(acc.x * a + o4.x * f, acc.y * a + o4.y * f, acc.z * a + o4.z * f,
                          acc.w * a + o4.w * f);
        l = l * a + ml.y * f;
        m = mn;
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    reinterpret_cast<float4 *>(p.out + (row0 + e / Q4) * D)[e % Q4] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
}

// ---------------------------------------------------------------------------
// SPLIT: several CTAs per (sequence, head tile), merged by the last to finish
// (a separate instantiation, so one CTA per (sequence, head tile) carries
// none of that code).
template <int D, int GT, bool BF16, int NW, int S, bool MMA, bool SPLIT>
__global__ void __launch_bounds__(NW * 32)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  using L = DecodeSmem<D, GT, NW, S, MMA>;
  using Ring = PageRing<D, NW, S>;
  constexpr int HALF = D / 2;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_release();
  griddep_wait();  // inputs may come from the previous kernel in the stream
  const int n_sub = p.group / GT;
  const int g = blockIdx.y / n_sub;
  const int h0 = g * p.group + (blockIdx.y % n_sub) * GT;
  const int b = blockIdx.z;
  const int ppw = p.warp_parts;  // > 0: every warp owns ppw whole partitions

  int T = p.ctx_lens[b];
  const int maxT = p.max_blocks * 16;
  const bool t_ok = T >= 0 && T <= maxT;  // a clamped length stores no token
  if (!t_ok) {
    if (tid == 0) record_error(p.status, PA_ERR_BAD_CTX);
    T = T < 0 ? 0 : maxT;
  }
  KeySet ks;
  ks.init(T, p.sink, p.window);
  const int n_pages = ks.n_v;  // virtual pages of the attended keys
  // Pages per CTA (0: all of them), this CTA's pages, and how many CTAs of
  // this (sequence, head tile) have any: those, and only those, arrive at
  // the merge.
  const int cta_pages = ppw > 0 ? NW * ppw * p.part_pages : p.part_pages;
  int pg0 = 0, pg1 = n_pages;
  if (cta_pages > 0) {
    pg0 = blockIdx.x * cta_pages;
    pg1 = min(n_pages, pg0 + cta_pages);
  }
  const int n_active = cta_pages > 0 ? (n_pages + cta_pages - 1) / cta_pages : 1;
  if (pg0 >= pg1) {
    // Nothing to read.  An empty sequence owes zeros (CTA 0 writes them), or
    // an empty state (O = 0, m = -inf, l = 0).
    if (blockIdx.x == 0) {
      for (int i = tid; i < GT * (D + 4); i += NW * 32) {
        const size_t row = static_cast<size_t>(b) * p.n_q_heads + h0 + i / (D + 4);
        const int d = i % (D + 4);
        if (!p.part) {
          if (d < D) p.out[row * D + d] = 0.f;
        } else if (d < D + 2) {
          p.part[(row * p.part_stride + p.part_slot) * (D + 4) + d] = d == D ? -INFINITY : 0.f;
        }
      }
    }
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < L::kStages; ++s) mbar_init(sbase + L::kBarOff + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();

  Ring ring;
  ring.stage0 = sbase + warp * S * L::kStageBytes;
  ring.bar0 = sbase + L::kBarOff + warp * S * 8;
  ring.bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  ring.status = p.status;
  if (ppw > 0) {  // warp w: partitions blockIdx.x * NW * ppw + w * ppw + [0, ppw)
    ring.first = pg0 + warp * ppw * p.part_pages;
    ring.stride = 1;
    ring.n_i = max(0, min(pg1, ring.first + ppw * p.part_pages) - ring.first);
  } else {        // warp w: pages pg0 + w, pg0 + w + NW, ...
    ring.first = pg0 + warp;
    ring.stride = NW;
    ring.n_i = ring.first < pg1 ? (pg1 - ring.first + NW - 1) / NW : 0;
  }
  ring.num_pages = p.num_pages;
  ring.ks = ks;
  ring.y_page = p.n_kv_heads * 16;
  ring.y_head = g * 16;
  ring.patch_lp = -1;
  if (p.k_new && pg1 == n_pages) {
    // Fused append: this CTA holds the last page, which holds key T - 1.
    ring.patch_lp = (T - 1) >> 4;
    ring.patch_row = (T - 1) & 15;
    const int c = lane & 15;
    const uint16_t *src = (lane >= 16 ? p.v_new : p.k_new) +
                          (static_cast<size_t>(b) * p.n_kv_heads + g) * D + c * 8;
    ring.patch_val = make_uint4(0u, 0u, 0u, 0u);
    if (c < D / 8) ring.patch_val = __ldg(reinterpret_cast<const uint4 *>(src));
    if (t_ok && warp == 0 && blockIdx.y % n_sub == 0) {
      // one CTA per (sequence, kv head) writes the rows into the cache
      int id = __ldg(ring.bt_row + ring.patch_lp);
      if (static_cast<unsigned>(id) >= static_cast<unsigned>(p.num_pages)) {
        if (lane == 0) record_error(p.status, PA_ERR_BAD_BLOCK);
      } else if (c < D / 8) {
        const size_t row = (static_cast<size_t>(id) * p.n_kv_heads + g) * 16 + ring.patch_row;
        *reinterpret_cast<uint4 *>((lane >= 16 ? p.v_cache : p.k_cache) + row * D + c * 8) =
            ring.patch_val;
      }
    }
  }
  ring.start(lane);
  for (int i = 0; i < S && i < ring.n_i; ++i) ring.issue(i, lane, &kmap, &vmap);

  // ---- q of the head tile -> shared memory (overlaps the first copies)
  const uint16_t *qg = p.q + (static_cast<size_t>(b) * p.n_q_heads + h0) * D;
  if constexpr (MMA) {
    const uint32_t qs = sbase + L::kQOff;
    for (int e = tid; e < 16 * (D / 8); e += NW * 32) {
      const int r = e / (D / 8), c = e % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < GT) v = *reinterpret_cast<const uint4 *>(qg + r * D + c * 8);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(qs + swz(r, c, 16)),
                   "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
    }
  } else {
    float *q_s = reinterpret_cast<float *>(smem + L::kQOff);
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

  const size_t row0 = static_cast<size_t>(b) * p.n_q_heads + h0;
  float *mer_m = reinterpret_cast<float *>(smem);
  float *mer_l = mer_m + NW * GT;
  float *mer_o = mer_l + NW * GT;
  if constexpr (MMA) {
    const int r = lane >> 2, k0 = 2 * (lane & 3);
    float m_r, l_r, o[D / 8][4];
    auto reset = [&] {
      m_r = -INFINITY;
      l_r = 0.f;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    };
    if (!SPLIT && ppw > 0) {
      // ---- one CTA holds every partition: each one's state goes from
      // registers to the workspace, then the CTA folds them into the output
      for (int k = 0; k < ppw && k * p.part_pages < ring.n_i; ++k) {
        reset();
        const bool ok = pages_mma<D, GT, BF16, NW, S>(
            ring, k * p.part_pages, min(ring.n_i, (k + 1) * p.part_pages), &kmap, &vmap,
            sbase + L::kQOff, p.qscale, T, lane, m_r, l_r, o);
        const int part = (ring.first / p.part_pages) + k;
        if (r < GT) {
          float *dst = p.ws + ((row0 + r) * p.n_parts + part) * (D + 4);
#pragma unroll
          for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<float2 *>(dst + n * 8 + k0) =
                make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
          if ((lane & 3) == 0) *reinterpret_cast<float2 *>(dst + D) = make_float2(m_r * kLn2, l_r);
        }
        if (!ok) break;
      }
      merge_own_partitions<D, GT, NW>(p, row0, (n_pages + p.part_pages - 1) / p.part_pages, tid);
      return;
    } else {
      // ---- one range per warp (a warp that owns partitions walks them as one)
      reset();
      pages_mma<D, GT, BF16, NW, S>(ring, 0, ring.n_i, &kmap, &vmap, sbase + L::kQOff,
                                    p.qscale, T, lane, m_r, l_r, o);
      __syncthreads();  // every warp is done with its stages
      if (r < GT) {
        if ((lane & 3) == 0) {
          mer_m[warp * GT + r] = m_r;
          mer_l[warp * GT + r] = l_r;
        }
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
          *reinterpret_cast<float2 *>(mer_o + (warp * GT + r) * D + n * 8 + k0) =
              make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
      }
    }
  } else {
    constexpr int DPL = D / 32;
    float m[GT], lsum[GT];
    float2 O2[GT][D / 64];
    auto reset = [&] {
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        m[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int k = 0; k < D / 64; ++k) O2[h][k] = make_float2(0.f, 0.f);
      }
    };
    float *p_s = reinterpret_cast<float *>(smem + L::kPOff) + warp * GT * 16;
    const float *q_s = reinterpret_cast<const float *>(smem + L::kQOff);
    if (!SPLIT && ppw > 0) {  // as in the tensor-core path
      for (int k = 0; k < ppw && k * p.part_pages < ring.n_i; ++k) {
        reset();
        const bool ok = pages_cuda_core<D, GT, BF16, NW, S>(
            ring, k * p.part_pages, min(ring.n_i, (k + 1) * p.part_pages), &kmap, &vmap, q_s,
            p_s, T, lane, m, lsum, O2);
        const int part = (ring.first / p.part_pages) + k;
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          float *dst = p.ws + ((row0 + h) * p.n_parts + part) * (D + 4);
#pragma unroll
          for (int kk = 0; kk < DPL / 2; ++kk)
            *reinterpret_cast<float2 *>(dst + lane * DPL + 2 * kk) = O2[h][kk];
          if (lane == 0) *reinterpret_cast<float2 *>(dst + D) = make_float2(m[h] * kLn2, lsum[h]);
        }
        if (!ok) break;
      }
      merge_own_partitions<D, GT, NW>(p, row0, (n_pages + p.part_pages - 1) / p.part_pages, tid);
      return;
    } else {
      reset();
      pages_cuda_core<D, GT, BF16, NW, S>(ring, 0, ring.n_i, &kmap, &vmap, q_s, p_s, T, lane,
                                          m, lsum, O2);
      __syncthreads();  // every warp is done with its stages
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
    }
  }

  // ---- merge the NW warp states: final output, or this CTA's partial state
  // (slot blockIdx.x of the row: the partition, or the CTA's partitions)
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
    const size_t row = row0 + h;
    if constexpr (!SPLIT) {
      if (!p.part) {
        p.out[row * D + d] = lt > 0.f ? o / lt : 0.f;
      } else {
        float *dst = p.part + (row * p.part_stride + p.part_slot) * (D + 4);
        dst[d] = o;
        if (d == 0) {
          dst[D] = M * kLn2;  // natural-log units
          dst[D + 1] = lt;
        }
      }
    } else {
      float *dst = p.ws + (row * p.n_parts + blockIdx.x) * (D + 4);
      dst[d] = o;
      if (d == 0) {
        dst[D] = M * kLn2;  // natural-log units
        dst[D + 1] = lt;
      }
    }
  }

  if constexpr (SPLIT) {
    // ---- the last of the n_active CTAs of this (sequence, head tile) to
    // finish merges all their states (the same exponent law).  One
    // thread arrives with an acquire-release add once the CTA's partial
    // stores are issued (release: they are visible before the arrival
    // counts; acquire: the last arrival sees every other CTA's), the barrier
    // extending it to the CTA.
    __shared__ int s_last;
    __syncthreads();
    const int grp = blockIdx.z * gridDim.y + blockIdx.y;
    if (tid == 0) s_last = atomic_add_acq_rel_gpu(p.ctr + grp, 1) == n_active - 1;
    __syncthreads();
    if (!s_last) return;
    // Thread t folds (row, float4 of head_dim) pairs t, t + 128, ... over the
    // CTAs' states, loading 8 of them before folding any, so n CTAs cost
    // about n / 8 round trips to L2.
    const int n_valid = n_active;
    constexpr int Q4 = D / 4, kPairs = (GT * Q4 + NW * 32 - 1) / (NW * 32), kBatch = 8;
    float mm[kPairs], ll[kPairs];
    float4 acc[kPairs];
#pragma unroll
    for (int j = 0; j < kPairs; ++j) {
      mm[j] = -INFINITY;
      ll[j] = 0.f;
      acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int c0 = 0; c0 < n_valid; c0 += kBatch) {
      float2 ml[kPairs][kBatch];
      float4 o4[kPairs][kBatch];
#pragma unroll
      for (int j = 0; j < kPairs; ++j) {
        const int e = tid + j * NW * 32;
        const float *base = p.ws + (row0 + e / Q4) * p.n_parts * (D + 4);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          ml[j][u] = make_float2(-INFINITY, 0.f);
          if (e < GT * Q4 && c0 + u < n_valid) {
            const float *sp = base + static_cast<size_t>(c0 + u) * (D + 4);
            ml[j][u] = __ldcg(reinterpret_cast<const float2 *>(sp + D));
            o4[j][u] = __ldcg(reinterpret_cast<const float4 *>(sp) + e % Q4);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kPairs; ++j)
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (ml[j][u].y > 0.f) {  // a CTA whose keys all had weight 0 adds nothing
            const float mp = ml[j][u].x * kLog2e;
            const float mn = fmaxf(mm[j], mp);
            const float a = ex2(mm[j] - mn), f = ex2(mp - mn);  // a = 0 at m = -inf
            acc[j].x = acc[j].x * a + o4[j][u].x * f;
            acc[j].y = acc[j].y * a + o4[j][u].y * f;
            acc[j].z = acc[j].z * a + o4[j][u].z * f;
            acc[j].w = acc[j].w * a + o4[j][u].w * f;
            ll[j] = ll[j] * a + ml[j][u].y * f;
            mm[j] = mn;
          }
        }
    }
#pragma unroll
    for (int j = 0; j < kPairs; ++j) {
      const int e = tid + j * NW * 32;
      if (e < GT * Q4) {
        const float inv = ll[j] > 0.f ? 1.f / ll[j] : 0.f;
        reinterpret_cast<float4 *>(p.out + (row0 + e / Q4) * D)[e % Q4] =
            make_float4(acc[j].x * inv, acc[j].y * inv, acc[j].z * inv, acc[j].w * inv);
      }
    }
    if (tid == 0) p.ctr[grp] = 0;  // left as the next call's clear finds it
  }
}

// Clears a split pa_decode's arrival counters after every earlier kernel in
// the stream (one of them may still be counting on the same workspace).
__global__ void clear_counters_kernel(int *ctr, int n) {
  griddep_release();
  griddep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    ctr[i] = 0;
}

// ---------------------------------------------------------------------------
// Exact merge of partition states (the exponent law: M = max m_p,
// l = sum e^(m_p - M) l_p, o = sum e^(m_p - M) O_p / l), one CTA of 128
// threads per row.  A row is (sequence b, query i < q_len, head h), stored at
// (b q_len + i) n_q_heads + h; it saw T = ctx[b] keys (decode), or
// ctx[b] + i + 1 (prefill: query i of a chunk that follows ctx[b] cached
// tokens), so its partitions 0 .. ceil(T / part_tokens) - 1 hold states; or
// (mode 2, a cascade decode) every one of its n_parts slots holds a state,
// possibly empty (l = 0).  Thread (sl, qd) owns a float4 of head_dim
// and every SL-th partition, and folds its partitions into a running
// (m, l, O) with the same law as it reads them, so all its loads are
// independent and a row costs about one memory round trip; the SL slices
// then fold through shared memory.
template <int D>
__global__ void __launch_bounds__(128)
    merge_kernel(const float *__restrict__ parts, const int32_t *__restrict__ ctx,
                 float *__restrict__ out, int *status, int n_q_heads, int n_parts,
                 int part_tokens, int prefill) {
  constexpr int W = D + 4, Q = D / 4, SL = 128 / Q;
  __shared__ float2 sml[SL];
  __shared__ __align__(16) float sacc[SL][D];
  const int h = blockIdx.x % n_q_heads, i = blockIdx.x / n_q_heads, b = blockIdx.y;
  const int q_len = gridDim.x / n_q_heads, tid = threadIdx.x;
  griddep_release();
  griddep_wait();
  int n_valid = n_parts;
  if (prefill != 2) {
    long T = ctx[b];
    if (T < 0) {
      if (tid == 0 && blockIdx.x == 0) record_error(status, PA_ERR_BAD_CTX);
      T = 0;
    }
    if (prefill) T += i + 1;
    n_valid = static_cast<int>((T + part_tokens - 1) / part_tokens);
    if (n_valid > n_parts) {
      if (tid == 0 && blockIdx.x == 0) record_error(status, PA_ERR_BAD_CTX);
      n_valid = n_parts;
    }
  }
  const size_t row = (static_cast<size_t>(b) * q_len + i) * n_q_heads + h;
  const float *base = parts + row * static_cast<size_t>(n_parts) * W;

  const int qd = tid % Q, sl = tid / Q;
  float m = -INFINITY, l = 0.f;  // m in log2 units
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int q = sl; q < n_valid; q += SL) {
    const float *sp = base + static_cast<size_t>(q) * W;
    const float2 ml = __ldg(reinterpret_cast<const float2 *>(sp + D));
    const float4 o4 = __ldg(reinterpret_cast<const float4 *>(sp) + qd);
    if (ml.y > 0.f) {  // an empty partition (l = 0) contributes nothing
      const float mp = ml.x * kLog2e;
      const float mn = fmaxf(m, mp);
      const float a = ex2(m - mn), c = ex2(mp - mn);  // a = 0 while m = -inf
      acc.x = acc.x * a + o4.x * c;
      acc.y = acc.y * a + o4.y * c;
      acc.z = acc.z * a + o4.z * c;
      acc.w = acc.w * a + o4.w * c;
      l = l * a + ml.y * c;
      m = mn;
    }
  }
  *reinterpret_cast<float4 *>(&sacc[sl][4 * qd]) = acc;
  if (qd == 0) sml[sl] = make_float2(m, l);
  __syncthreads();
  if (tid < Q) {
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < SL; ++k) M = fmaxf(M, sml[k].x);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    float lt = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < SL; ++k) {
        const float f = ex2(sml[k].x - M);  // 0 for a slice that saw nothing
        const float4 v = *reinterpret_cast<const float4 *>(&sacc[k][4 * tid]);
        t.x += f * v.x;
        t.y += f * v.y;
        t.z += f * v.z;
        t.w += f * v.w;
        lt += f * sml[k].y;
      }
    }
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    reinterpret_cast<float4 *>(out + row * D)[tid] =
        make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
  }
}

// Stages per warp: about 24 KiB of K/V per warp in the ring.
template <int D>
constexpr int stages_per_warp() { return D == 128 ? 3 : 6; }

template <int D, int GT, bool BF16>
int launch_decode_t(const DecodeLaunch &a, cudaStream_t stream) {
  constexpr int NW = kDecodeWarps, S = stages_per_warp<D>();
  constexpr bool MMA = GT >= 2;
  using L = DecodeSmem<D, GT, NW, S, MMA>;
  const int gx = a.warp_parts > 0 ? (a.n_parts + NW * a.warp_parts - 1) / (NW * a.warp_parts)
                                  : a.n_parts;
  const bool split = gx > 1;  // else one CTA per (sequence, head tile)
  auto kern = split ? decode_kernel<D, GT, BF16, NW, S, MMA, true>
                    : decode_kernel<D, GT, BF16, NW, S, MMA, false>;
  static ContextCache<bool> smem_set[2];  // per variant: contexts where the limit is set
  if (set_smem_limit(kern, L::kAlloc, smem_set[split]) != PA_OK) return PA_ERR_CUDA;
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
  p.ctr = nullptr;
  p.qscale = a.scale * kLog2e;
  p.n_q_heads = a.n_q_heads;
  p.n_kv_heads = a.n_kv_heads;
  p.group = a.n_q_heads / a.n_kv_heads;
  p.batch = a.batch;
  p.max_blocks = a.max_blocks;
  p.num_pages = a.num_pages;
  p.part_pages = a.part_pages;
  p.n_parts = a.n_parts;
  p.warp_parts = a.warp_parts;
  p.sink = a.sink;
  p.window = a.window;
  p.part = a.part;
  p.part_stride = a.part_stride;
  p.part_slot = a.part_slot;
  p.k_new = static_cast<const uint16_t *>(a.k_new);
  p.v_new = static_cast<const uint16_t *>(a.v_new);
  p.k_cache = static_cast<uint16_t *>(const_cast<void *>(a.k_cache));
  p.v_cache = static_cast<uint16_t *>(const_cast<void *>(a.v_cache));
  const dim3 grid(gx, a.n_kv_heads * (p.group / GT), a.batch);
  if (split) {
    p.ctr = reinterpret_cast<int *>(reinterpret_cast<char *>(a.workspace) +
                                    decode_counters_offset(a.batch, a.n_q_heads, a.n_parts, D));
    if (launch_clear_counters(p.ctr, static_cast<int>(grid.y * grid.z), stream) != PA_OK)
      return PA_ERR_CUDA;
  }
  if (launch_pdl(kern, grid, dim3(NW * 32), L::kAlloc, stream, kmap, vmap, p) != cudaSuccess)
    return PA_ERR_CUDA;
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

int launch_clear_counters(int *ctr, int n, cudaStream_t stream) {
  return launch_pdl(clear_counters_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, ctr,
                    n) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

int launch_merge(const float *partials, const int32_t *ctx_lens, float *out,
                 int *status, int batch, int n_q_heads, int head_dim,
                 int n_parts, int partition_tokens, cudaStream_t stream) {
  const dim3 grid(n_q_heads, batch);
  if (head_dim == 128)
    merge_kernel<128><<<grid, 128, 0, stream>>>(partials, ctx_lens, out, status,
                                                n_q_heads, n_parts, partition_tokens, 0);
  else
    merge_kernel<64><<<grid, 128, 0, stream>>>(partials, ctx_lens, out, status,
                                               n_q_heads, n_parts, partition_tokens, 0);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_merge_all(const float *partials, float *out, int *status, int n_rows, int n_q_heads,
                     int head_dim, int n_slots, cudaStream_t stream) {
  const dim3 grid(n_q_heads * n_rows, 1);
  const cudaError_t e =
      head_dim == 128
          ? launch_pdl(merge_kernel<128>, grid, dim3(128), 0, stream, partials,
                       static_cast<const int32_t *>(nullptr), out, status, n_q_heads, n_slots, 1, 2)
          : launch_pdl(merge_kernel<64>, grid, dim3(128), 0, stream, partials,
                       static_cast<const int32_t *>(nullptr), out, status, n_q_heads, n_slots, 1, 2);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_merge_rows(const float *partials, const int32_t *ctx_lens, float *out, int *status,
                      int batch, int n_q_heads, int head_dim, int n_parts,
                      int partition_tokens, int n_new, cudaStream_t stream) {
  const dim3 grid(n_q_heads * n_new, batch);
  const cudaError_t e =
      head_dim == 128
          ? launch_pdl(merge_kernel<128>, grid, dim3(128), 0, stream, partials, ctx_lens, out,
                       status, n_q_heads, n_parts, partition_tokens, 1)
          : launch_pdl(merge_kernel<64>, grid, dim3(128), 0, stream, partials, ctx_lens, out,
                       status, n_q_heads, n_parts, partition_tokens, 1);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
