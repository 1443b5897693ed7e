/*
 * pa_oracle.c -- TEST INFRASTRUCTURE, not product code.
 *
 * A plain, slow, float64 CPU oracle for paged GQA attention.  Only the test
 * suite, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load it.
 * It shares no source, header, table or helper with the CUDA library; it has
 * its own 16-bit float decoders and its own gather through the block table.
 *
 * What it computes, and the passage each function follows:
 *
 *  - Attention for one decode query (ch. 19 "推理系统与性能工程", 19.4.1):
 *    o = softmax(q . K^T * scale) . V over every cached token of the sequence.
 *  - The numerically stable softmax (same chapter, 19.6.2, first display):
 *    softmax(x)_i = e^(x_i - m) / sum_j e^(x_j - m) with m = max_j x_j.
 *  - The online-softmax recurrence over blocks B_1, B_2, ... (19.6.2, three
 *    steps: running max, rescale factor c = e^(m_k - m_{k+1}), rebased l, O).
 *  - PagedAttention's block table (19.7.3): logical token t of a sequence lives
 *    in physical block block_table[b][t / P] at slot t % P.
 *  - GQA sharing of KV heads ("吞吐与延迟的系统模型", section 4 and 5): h_q query
 *    heads read h_kv < h_q KV heads.  The pages do not fix the head mapping;
 *    the plainest reading is contiguous groups, q head h -> kv head h / G with
 *    G = h_q / h_kv, which makes h_kv = h_q the identity (MHA).
 *  - Exact merge of partial (m, l, O) states of disjoint chunks: the exponent
 *    law e^(a+b) = e^a e^b that 19.6.2 uses to justify the rescale, applied to
 *    two already-summarised chunks instead of one new block.
 *  - KV append: a decode step writes one new K and one new V row per layer
 *    and head ("吞吐与延迟的系统模型", section 4, the 2LBd_kv b_kv write term).
 *  - Chunked prefill over the cache: query i of a chunk of new tokens sees
 *    every cached key plus the new keys up to and including its own
 *    (causal prefill, 19.3.1; FlashAttention forward, 19.6.3).
 *
 * Data layout it reads (chosen by the library, documented there):
 *   q        [batch, n_q_heads, head_dim]           16-bit floats (bit patterns)
 *   k_cache  [num_pages, n_kv_heads, page_size, head_dim]
 *   v_cache  same
 *   block_table int32 [batch, max_blocks]
 *   ctx_lens int32 [batch]
 * Results are written as double.
 *
 * Every function returns 0 on success and -1 when an index it would follow
 * (a block-table entry, a context length) is out of range; it never reads
 * outside the buffers it was given.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 0, OR_F16 = 1 };

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double or_dec_bf16(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double or_dec_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25);   /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

static double or_dec(uint16_t h, int dtype) {
  return dtype == OR_BF16 ? or_dec_bf16(h) : or_dec_f16(h);
}

/* Exposed so the pins can check the decoders against numpy's own casts. */
double oracle_decode_half(uint16_t h, int dtype) { return or_dec(h, dtype); }

static void or_set_threads(int n_threads) {
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

typedef struct {
  const uint16_t *k_cache, *v_cache;
  const int32_t *block_table;
  int n_kv_heads, head_dim, page_size, max_blocks, num_pages, dtype;
} or_cache;

/* Address of the K (or V) row of logical token t of sequence b, kv head g,
 * or NULL when the block table points outside the pool. */
static const uint16_t *or_row(const or_cache *c, const uint16_t *base, int b,
                              int g, long t) {
  long blk = t / c->page_size;
  long slot = t % c->page_size;
  if (blk < 0 || blk >= c->max_blocks) return NULL;
  int32_t page = c->block_table[(long)b * c->max_blocks + blk];
  if (page < 0 || page >= c->num_pages) return NULL;
  size_t off = (((size_t)page * c->n_kv_heads + g) * c->page_size + slot) *
               (size_t)c->head_dim;
  return base + off;
}

/* Scores s_t = scale * <q, k_t> for t in [0, T); returns -1 on a bad index. */
static int or_scores(const or_cache *c, const double *qd, int b, int g, long T,
                     double scale, double *s) {
  for (long t = 0; t < T; ++t) {
    const uint16_t *k = or_row(c, c->k_cache, b, g, t);
    if (!k) return -1;
    double acc = 0.0;
    for (int i = 0; i < c->head_dim; ++i) acc += qd[i] * or_dec(k[i], c->dtype);
    s[t] = scale * acc;
  }
  return 0;
}

/* Full softmax of one row of T scores, then the weighted sum of V rows.
 * T == 0 gives a zero vector (the pages are silent; this is our reading). */
static int or_attend_full(const or_cache *c, const double *qd, int b, int g,
                          long T, double scale, double *s, double *o) {
  int D = c->head_dim;
  for (int i = 0; i < D; ++i) o[i] = 0.0;
  if (T == 0) return 0;
  if (or_scores(c, qd, b, g, T, scale, s)) return -1;
  double m = -INFINITY;
  for (long t = 0; t < T; ++t)
    if (s[t] > m) m = s[t];
  double denom = 0.0;
  for (long t = 0; t < T; ++t) {
    double w = exp(s[t] - m);
    denom += w;
    const uint16_t *v = or_row(c, c->v_cache, b, g, t);
    if (!v) return -1;
    for (int i = 0; i < D; ++i) o[i] += w * or_dec(v[i], c->dtype);
  }
  for (int i = 0; i < D; ++i) o[i] /= denom;
  return 0;
}

static int or_check_heads(int n_q_heads, int n_kv_heads) {
  return (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) ? -1 : 0;
}

/* Decode attention, plain definition: per (sequence, query head) gather every
 * cached token through the block table and apply full softmax.
 * out: double [batch, n_q_heads, head_dim]. */
int oracle_decode(const uint16_t *q, const uint16_t *k_cache,
                  const uint16_t *v_cache, const int32_t *block_table,
                  const int32_t *ctx_lens, double *out, double scale,
                  int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                  int batch, int max_blocks, int num_pages, int dtype,
                  int n_threads) {
  if (or_check_heads(n_q_heads, n_kv_heads)) return -1;
  for (int b = 0; b < batch; ++b)
    if (ctx_lens[b] < 0 || (long)ctx_lens[b] > (long)max_blocks * page_size)
      return -1;
  or_cache c = {k_cache, v_cache, block_table, n_kv_heads, head_dim,
                page_size, max_blocks, num_pages, dtype};
  int G = n_q_heads / n_kv_heads;
  int bad = 0;
  or_set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long bh = 0; bh < (long)batch * n_q_heads; ++bh) {
    int b = (int)(bh / n_q_heads), h = (int)(bh % n_q_heads), g = h / G;
    long T = ctx_lens[b];
    double *s = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
    double *qd = (double *)malloc(sizeof(double) * head_dim);
    const uint16_t *qr = q + ((size_t)b * n_q_heads + h) * head_dim;
    for (int i = 0; i < head_dim; ++i) qd[i] = or_dec(qr[i], dtype);
    if (or_attend_full(&c, qd, b, g, T, scale, s, out + bh * head_dim)) bad = 1;
    free(s);
    free(qd);
  }
  return bad ? -1 : 0;
}

/* Decode attention over the attention-sink + sliding-window key set ("推理系统
 * 与性能工程", KV-cache eviction: keep the first tokens of the sequence and a
 * window of the most recent ones).  Key t of a T-token sequence is kept iff
 * t < sink or t >= T - window; the softmax runs over the kept keys only (a
 * row with none gives zeros).  out: double [batch, n_q_heads, head_dim]. */
static int or_attend_kept(const or_cache *c, const double *qd, int b, int g, long T,
                          long sink, long window, double scale, double *s,
                          double *o) {
  int D = c->head_dim;
  for (int i = 0; i < D; ++i) o[i] = 0.0;
  if (T == 0) return 0;
  if (or_scores(c, qd, b, g, T, scale, s)) return -1;
  double m = -INFINITY;
  long kept = 0;
  for (long t = 0; t < T; ++t)
    if (t < sink || t >= T - window) {
      if (s[t] > m) m = s[t];
      ++kept;
    }
  if (kept == 0) return 0;
  double denom = 0.0;
  for (long t = 0; t < T; ++t) {
    if (!(t < sink || t >= T - window)) continue;
    double w = exp(s[t] - m);
    denom += w;
    const uint16_t *v = or_row(c, c->v_cache, b, g, t);
    if (!v) return -1;
    for (int i = 0; i < D; ++i) o[i] += w * or_dec(v[i], c->dtype);
  }
  for (int i = 0; i < D; ++i) o[i] /= denom;
  return 0;
}

int oracle_decode_window(const uint16_t *q, const uint16_t *k_cache,
                         const uint16_t *v_cache, const int32_t *block_table,
                         const int32_t *ctx_lens, double *out, double scale,
                         int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                         int batch, int max_blocks, int num_pages, int dtype, int sink,
                         int window, int n_threads) {
  if (or_check_heads(n_q_heads, n_kv_heads) || sink < 0 || window < 0) return -1;
  for (int b = 0; b < batch; ++b)
    if (ctx_lens[b] < 0 || (long)ctx_lens[b] > (long)max_blocks * page_size)
      return -1;
  or_cache c = {k_cache, v_cache, block_table, n_kv_heads, head_dim,
                page_size, max_blocks, num_pages, dtype};
  int G = n_q_heads / n_kv_heads;
  int bad = 0;
  or_set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long bh = 0; bh < (long)batch * n_q_heads; ++bh) {
    int b = (int)(bh / n_q_heads), h = (int)(bh % n_q_heads), g = h / G;
    long T = ctx_lens[b];
    double *s = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
    double *qd = (double *)malloc(sizeof(double) * head_dim);
    const uint16_t *qr = q + ((size_t)b * n_q_heads + h) * head_dim;
    for (int i = 0; i < head_dim; ++i) qd[i] = or_dec(qr[i], dtype);
    if (or_attend_kept(&c, qd, b, g, T, sink, window, scale, s, out + bh * head_dim))
      bad = 1;
    free(s);
    free(qd);
  }
  return bad ? -1 : 0;
}

/* The same result reached the way the pages' recurrence reaches it: the row
 * is cut into blocks at the given positions (cuts[] ascending, in tokens) and
 * the blocks are folded in order with
 *   m_{k+1} = max(m_k, max of the block),  c = e^(m_k - m_{k+1}),
 *   l_{k+1} = c l_k + sum e^(x_j - m_{k+1}),
 *   O_{k+1} = c O_k + sum e^(x_j - m_{k+1}) v_j,
 * and the answer is O / l after the last block. */
int oracle_decode_online(const uint16_t *q, const uint16_t *k_cache,
                         const uint16_t *v_cache, const int32_t *block_table,
                         const int32_t *ctx_lens, double *out, double scale,
                         int n_q_heads, int n_kv_heads, int head_dim,
                         int page_size, int batch, int max_blocks,
                         int num_pages, int dtype, const int32_t *cuts,
                         int n_cuts) {
  if (or_check_heads(n_q_heads, n_kv_heads)) return -1;
  or_cache c = {k_cache, v_cache, block_table, n_kv_heads, head_dim,
                page_size, max_blocks, num_pages, dtype};
  int G = n_q_heads / n_kv_heads;
  for (long bh = 0; bh < (long)batch * n_q_heads; ++bh) {
    int b = (int)(bh / n_q_heads), h = (int)(bh % n_q_heads), g = h / G;
    long T = ctx_lens[b];
    if (T < 0 || T > (long)max_blocks * page_size) return -1;
    double *o = out + bh * head_dim;
    double *qd = (double *)malloc(sizeof(double) * head_dim);
    double *s = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
    const uint16_t *qr = q + ((size_t)b * n_q_heads + h) * head_dim;
    for (int i = 0; i < head_dim; ++i) qd[i] = or_dec(qr[i], dtype);
    int rc = or_scores(&c, qd, b, g, T, scale, s);
    double m = -INFINITY, l = 0.0;
    for (int i = 0; i < head_dim; ++i) o[i] = 0.0;
    long start = 0;
    for (int k = 0; k <= n_cuts && rc == 0; ++k) {
      long end = (k < n_cuts) ? cuts[k] : T;
      if (end > T) end = T;
      if (end <= start) continue;
      double mt = -INFINITY;
      for (long t = start; t < end; ++t)
        if (s[t] > mt) mt = s[t];
      double m_new = m > mt ? m : mt;
      double cf = exp(m - m_new); /* m = -inf on the first block: c = 0 */
      l *= cf;
      for (int i = 0; i < head_dim; ++i) o[i] *= cf;
      for (long t = start; t < end; ++t) {
        double w = exp(s[t] - m_new);
        const uint16_t *v = or_row(&c, c.v_cache, b, g, t);
        if (!v) { rc = -1; break; }
        l += w;
        for (int i = 0; i < head_dim; ++i) o[i] += w * or_dec(v[i], dtype);
      }
      m = m_new;
      start = end;
    }
    if (rc == 0 && l > 0.0)
      for (int i = 0; i < head_dim; ++i) o[i] /= l;
    free(qd);
    free(s);
    if (rc) return -1;
  }
  return 0;
}

/* Partial states of fixed-size chunks of the row: chunk p covers tokens
 * [p*part_tokens, min((p+1)*part_tokens, T)).  For each (b, h, p) it writes
 * head_dim + 2 doubles: O_p (unnormalised, based on m_p), then m_p, then l_p.
 * An empty chunk has m_p = -inf, l_p = 0, O_p = 0.
 * parts: double [batch, n_q_heads, n_parts, head_dim + 2]. */
int oracle_partials(const uint16_t *q, const uint16_t *k_cache,
                    const uint16_t *v_cache, const int32_t *block_table,
                    const int32_t *ctx_lens, double *parts, double scale,
                    int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                    int batch, int max_blocks, int num_pages, int dtype,
                    int part_tokens, int n_parts, int n_threads) {
  if (or_check_heads(n_q_heads, n_kv_heads) || part_tokens <= 0) return -1;
  for (int b = 0; b < batch; ++b)
    if (ctx_lens[b] < 0 || (long)ctx_lens[b] > (long)max_blocks * page_size)
      return -1;
  or_cache c = {k_cache, v_cache, block_table, n_kv_heads, head_dim,
                page_size, max_blocks, num_pages, dtype};
  int G = n_q_heads / n_kv_heads;
  int W = head_dim + 2;
  int bad = 0;
  or_set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long bh = 0; bh < (long)batch * n_q_heads; ++bh) {
    int b = (int)(bh / n_q_heads), h = (int)(bh % n_q_heads), g = h / G;
    long T = ctx_lens[b];
    double *qd = (double *)malloc(sizeof(double) * head_dim);
    double *s = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
    const uint16_t *qr = q + ((size_t)b * n_q_heads + h) * head_dim;
    for (int i = 0; i < head_dim; ++i) qd[i] = or_dec(qr[i], dtype);
    if (or_scores(&c, qd, b, g, T, scale, s)) bad = 1;
    for (int p = 0; p < n_parts && !bad; ++p) {
      double *dst = parts + (bh * n_parts + p) * W;
      long lo = (long)p * part_tokens, hi = lo + part_tokens;
      if (hi > T) hi = T;
      double m = -INFINITY, l = 0.0;
      for (int i = 0; i < head_dim; ++i) dst[i] = 0.0;
      for (long t = lo; t < hi; ++t)
        if (s[t] > m) m = s[t];
      for (long t = lo; t < hi; ++t) {
        double w = exp(s[t] - m);
        const uint16_t *v = or_row(&c, c.v_cache, b, g, t);
        if (!v) { bad = 1; break; }
        l += w;
        for (int i = 0; i < head_dim; ++i) dst[i] += w * or_dec(v[i], dtype);
      }
      dst[head_dim] = m;
      dst[head_dim + 1] = l;
    }
    free(qd);
    free(s);
  }
  return bad ? -1 : 0;
}

/* Exact merge of n_parts partial states per row (rows = n_rows):
 *   M = max_p m_p,  l = sum_p e^(m_p - M) l_p,  o = sum_p e^(m_p - M) O_p / l.
 * A part with l_p = 0 (an empty chunk, m_p = -inf) contributes nothing; a row
 * with no non-empty part gives zeros.  Input rows as written by
 * oracle_partials: head_dim + 2 doubles per part. */
int oracle_merge(const double *parts, double *out, int n_rows, int n_parts,
                 int head_dim) {
  int W = head_dim + 2;
  for (long r = 0; r < n_rows; ++r) {
    const double *src = parts + (size_t)r * n_parts * W;
    double *o = out + (size_t)r * head_dim;
    double M = -INFINITY;
    for (int p = 0; p < n_parts; ++p)
      if (src[p * W + head_dim + 1] > 0.0 && src[p * W + head_dim] > M)
        M = src[p * W + head_dim];
    for (int i = 0; i < head_dim; ++i) o[i] = 0.0;
    if (M == -INFINITY) continue;
    double l = 0.0;
    for (int p = 0; p < n_parts; ++p) {
      const double *sp = src + (size_t)p * W;
      if (!(sp[head_dim + 1] > 0.0)) continue;
      double f = exp(sp[head_dim] - M);
      l += f * sp[head_dim + 1];
      for (int i = 0; i < head_dim; ++i) o[i] += f * sp[i];
    }
    for (int i = 0; i < head_dim; ++i) o[i] /= l;
  }
  return 0;
}

/* KV append: token j of the new batch belongs to sequence seq_idx[j] at
 * logical position pos[j]; its K and V rows for every kv head are stored at
 * (block_table[seq][pos / P], pos % P).  Plain element copies. */
int oracle_append_kv(const uint16_t *k_new, const uint16_t *v_new,
                     uint16_t *k_cache, uint16_t *v_cache,
                     const int32_t *block_table, const int32_t *seq_idx,
                     const int32_t *pos, int n_tok, int n_kv_heads,
                     int head_dim, int page_size, int batch, int max_blocks,
                     int num_pages) {
  for (int j = 0; j < n_tok; ++j) {
    int b = seq_idx[j];
    long p = pos[j];
    if (b < 0 || b >= batch || p < 0 || p >= (long)max_blocks * page_size)
      return -1;
    int32_t page = block_table[(long)b * max_blocks + p / page_size];
    if (page < 0 || page >= num_pages) return -1;
    for (int g = 0; g < n_kv_heads; ++g) {
      size_t dst = (((size_t)page * n_kv_heads + g) * page_size + p % page_size) *
                   (size_t)head_dim;
      size_t src = ((size_t)j * n_kv_heads + g) * head_dim;
      for (int i = 0; i < head_dim; ++i) {
        k_cache[dst + i] = k_new[src + i];
        v_cache[dst + i] = v_new[src + i];
      }
    }
  }
  return 0;
}

/* Chunked prefill over the paged cache.  ctx_lens[b] counts the tokens that
 * were cached before the chunk; the chunk's own n_new K/V rows are already
 * stored at positions ctx_lens[b] .. ctx_lens[b] + n_new - 1.  Query i of
 * sequence b attends keys 0 .. ctx_lens[b] + i (causal), full softmax.
 * q: [batch, n_new, n_q_heads, head_dim]; out: double, same shape. */
int oracle_prefill(const uint16_t *q, const uint16_t *k_cache,
                   const uint16_t *v_cache, const int32_t *block_table,
                   const int32_t *ctx_lens, int n_new, double *out,
                   double scale, int n_q_heads, int n_kv_heads, int head_dim,
                   int page_size, int batch, int max_blocks, int num_pages,
                   int dtype, int n_threads) {
  if (or_check_heads(n_q_heads, n_kv_heads) || n_new < 0) return -1;
  for (int b = 0; b < batch; ++b)
    if (ctx_lens[b] < 0 ||
        (long)ctx_lens[b] + n_new > (long)max_blocks * page_size)
      return -1;
  or_cache c = {k_cache, v_cache, block_table, n_kv_heads, head_dim,
                page_size, max_blocks, num_pages, dtype};
  int G = n_q_heads / n_kv_heads;
  int bad = 0;
  or_set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long r = 0; r < (long)batch * n_new * n_q_heads; ++r) {
    int h = (int)(r % n_q_heads);
    long bi = r / n_q_heads;
    int i = (int)(bi % n_new), b = (int)(bi / n_new), g = h / G;
    long T = (long)ctx_lens[b] + i + 1;
    double *s = (double *)malloc(sizeof(double) * T);
    double *qd = (double *)malloc(sizeof(double) * head_dim);
    const uint16_t *qr = q + (size_t)r * head_dim;
    for (int d = 0; d < head_dim; ++d) qd[d] = or_dec(qr[d], dtype);
    if (or_attend_full(&c, qd, b, g, T, scale, s, out + (size_t)r * head_dim))
      bad = 1;
    free(s);
    free(qd);
  }
  return bad ? -1 : 0;
}
