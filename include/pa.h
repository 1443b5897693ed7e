/*
 * pa.h -- C ABI of libpa, paged GQA attention for GB300 (sm_103a).
 *
 * Every entry point takes plain pointers and sizes.  Device pointers are
 * marked "device"; they must point into memory of the current CUDA device.
 * The caller owns every buffer.  The library allocates no device memory,
 * never synchronises a stream (except pa_last_device_error, which says so),
 * and queues its kernels on `stream` (NULL = the legacy default stream).
 *
 * Return value of every int entry point: PA_OK (0), or a negative PA_ERR_*
 * code when an argument is invalid -- in that case nothing was launched --
 * or PA_ERR_CUDA when a launch failed.  Data-dependent errors that only the
 * GPU can see (a block-table entry outside the pool, a context length out of
 * range, a wait that ran out) do not fault: the kernel skips the bad access,
 * records the first such error in a device status word, and carries on;
 * pa_last_device_error() reads and clears it.
 *
 * Cache layout (the pages do not fix one; this is the library's choice):
 *   k_cache, v_cache: [num_pages][n_kv_heads][page_size][head_dim] elements,
 *   so one (page, kv head) tile of page_size rows is one contiguous block.
 * Logical token t of sequence b lives in physical page
 *   block_table[b * max_blocks_per_seq + t / page_size], slot t % page_size
 * (PagedAttention's block table: ch. 19 "推理系统与性能工程", 19.7.3).
 * Query head h reads KV head h / (n_q_heads / n_kv_heads): contiguous GQA
 * groups ("吞吐与延迟的系统模型", sections 4-5: several query heads share one
 * KV head; the grouping order is our reading).
 *
 * Supported: head_dim 64 or 128, page_size 16 (the block size whose internal
 * fragmentation is at most 15 token slots, 19.7.3), n_q_heads a multiple of
 * n_kv_heads, bf16 or fp16 Q/K/V, fp32 output and accumulation.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so this header needs no CUDA
 * include. */
typedef struct CUstream_st *pa_stream_t;

typedef enum { PA_BF16 = 0, PA_F16 = 1 } pa_dtype;

enum {
  PA_OK = 0,
  PA_ERR_NULL = -1,        /* a required pointer is NULL */
  PA_ERR_HEADS = -2,       /* heads <= 0 or n_q_heads % n_kv_heads != 0 */
  PA_ERR_HEAD_DIM = -3,    /* head_dim not 64 or 128 */
  PA_ERR_PAGE_SIZE = -4,   /* page_size not 16 */
  PA_ERR_SHAPE = -5,       /* batch, max_blocks_per_seq, num_pages, n_tok or
                              n_new negative/zero where not allowed, or too big */
  PA_ERR_DTYPE = -6,       /* dtype not PA_BF16 / PA_F16 */
  PA_ERR_WORKSPACE = -7,   /* workspace NULL or smaller than required */
  PA_ERR_ALIGN = -8,       /* a pointer not 16-byte aligned */
  PA_ERR_PARTITION = -9,   /* partition_tokens not 0 and not a positive
                              multiple of page_size (decode) or of 128
                              (pa_prefill_paged_split) */
  PA_ERR_CUDA = -10,       /* a CUDA runtime call or launch failed */
  PA_ERR_BAD_BLOCK = -11,  /* device: block-table entry outside [0, num_pages) */
  PA_ERR_BAD_CTX = -12,    /* device: context length < 0 or beyond the table */
  PA_ERR_TIMEOUT = -13,    /* device: a bounded wait for a copy ran out */
  PA_ERR_BAD_INDEX = -14,  /* device: append seq_idx / pos outside the table */
  PA_ERR_SCRATCH_LIMIT = -15, /* pa_decode_static_workspace: the call needs more
                                 split-K scratch than its fixed 16 MiB array */
  PA_ERR_POOL_EMPTY = -16,   /* pa_pool_*: not enough free pages (nothing taken) */
  PA_ERR_POOL_STATE = -17    /* pa_pool_*: a page that is not in use (a double
                                release, a share of a free page) */
};

/* Human-readable name of a status code.  Never NULL. */
const char *pa_strerror(int status);

/*
 * pa_decode -- decode-step attention over the paged cache.
 *
 * For every sequence b and query head h, with g = h / G, G = n_q_heads /
 * n_kv_heads and T = ctx_lens[b]:
 *   s_t = scale * <q[b][h], k_t>            t = 0 .. T-1, k_t = K row of token t
 *   out[b][h] = sum_t e^(s_t - m) v_t / sum_t e^(s_t - m),   m = max_t s_t
 * i.e. o = softmax(q K^T * scale) V (ch. 19 "推理系统与性能工程", 19.4.1 and the
 * stable softmax of 19.6.2).  It is evaluated page by page with the online
 * recurrence of 19.6.2 (running max m, running sum l, unnormalised O); one
 * K/V page read serves all G query heads of its group.  Long contexts are
 * cut into partitions of `partition_tokens` tokens whose partial states
 * (m_p, l_p, O_p) are merged exactly (the exponent law of 19.6.2) by the
 * last CTA of the sequence's head group to finish.  T = 0 writes zeros.
 *
 *   q            device, [batch][n_q_heads][head_dim], dtype
 *   k_cache      device, [num_pages][n_kv_heads][page_size][head_dim], dtype
 *   v_cache      device, same shape
 *   block_table  device int32 [batch][max_blocks_per_seq]; only the first
 *                ceil(T/page_size) entries of row b are read
 *   ctx_lens     device int32 [batch], 0 <= T <= max_blocks_per_seq*page_size
 *   out          device float [batch][n_q_heads][head_dim]
 *   scale        softmax scale, applied before the max (1/sqrt(head_dim) in
 *                the pages' formula)
 *   partition_tokens  0 = choose automatically; otherwise a multiple of
 *                page_size: every sequence is processed in chunks of that
 *                many tokens and merged
 *   workspace    device, >= pa_decode_workspace_size(...) bytes, 16-byte
 *                aligned; may be NULL when that size is 0.  Holds the
 *                partial states and arrival counters; contents on entry do
 *                not matter (the call clears its counters on the stream
 *                first).  Two calls that overlap on the GPU must not share a
 *                workspace.
 * q, k_cache, v_cache, out and workspace must be 16-byte aligned.
 */
int pa_decode(const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_table, const int32_t *ctx_lens, float *out,
              float scale, int n_q_heads, int n_kv_heads, int head_dim,
              int page_size, int batch, int max_blocks_per_seq, int num_pages,
              pa_dtype dtype, int partition_tokens, void *workspace,
              size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_append -- one decode step of the pages' serving loop in one
 * call: the step's new K/V rows go into the cache and every query attends
 * the whole context, new token included.
 *
 * For every sequence b with T = ctx_lens[b] >= 1 (T counts the new token):
 *   1. the rows k_new[b][g], v_new[b][g] of every kv head g are stored at
 *      position T - 1, page block_table[b][(T-1) / page_size], slot
 *      (T-1) % page_size -- the per-step KV write of "吞吐与延迟的系统模型",
 *      section 4 (2 L B d_kv b_kv bytes per step over all layers);
 *   2. out[b] is what pa_decode computes over the T tokens.
 * The result equals pa_append_kv (seq_idx = b, pos = T - 1) followed by
 * pa_decode with the same arguments; one kernel does both: the CTA that
 * reads the last page puts the new rows into its copy of that page, and one
 * CTA per (sequence, kv head) writes them to the cache.  T = 0 writes zeros
 * and stores nothing.
 *   k_new, v_new  device, [batch][n_kv_heads][head_dim], dtype, 16-byte
 *                 aligned
 *   k_cache, v_cache  written in place (position T - 1 of every sequence)
 * Every other argument, the workspace (pa_decode_workspace_size) and the
 * plan are pa_decode's.  The page holding position T - 1 must be mapped in
 * the table; a bad page id stores nothing and records PA_ERR_BAD_BLOCK.  As
 * with pa_append_kv, no two sequences may place their token at the same
 * (page, slot): a page that forks of a shared prefix still share is copied
 * first (pa_pool_prepare_append, pa_copy_pages).
 */
int pa_decode_append(const void *q, const void *k_new, const void *v_new, void *k_cache,
                     void *v_cache, const int32_t *block_table, const int32_t *ctx_lens,
                     float *out, float scale, int n_q_heads, int n_kv_heads, int head_dim,
                     int page_size, int batch, int max_blocks_per_seq, int num_pages,
                     pa_dtype dtype, int partition_tokens, void *workspace,
                     size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_window -- decode attention over an attention sink plus a sliding
 * window of recent keys (ch. 19 "推理系统与性能工程", KV-cache eviction: keep
 * the first tokens and the most recent window).
 *
 * Same arguments and result layout as pa_decode, plus sink_tokens and
 * window_tokens (both >= 0, PA_ERR_SHAPE otherwise).  Key t of a sequence of
 * T = ctx_lens[b] tokens is attended iff t < sink_tokens or
 * t >= T - window_tokens; when sink_tokens + window_tokens >= T every key is
 * (plain decode), and a row with no attended key gives zeros.  Only the
 * attended keys' pages are read, so the HBM traffic is that of
 * sink + window tokens whatever T is.  Partitions (partition_tokens, as in
 * pa_decode) cut the attended keys; the workspace is sized by
 * pa_decode_window_workspace_size.  The block table still maps every
 * position below T (the pages in the gap are simply not read).
 */
int pa_decode_window(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, const int32_t *ctx_lens, float *out,
                     float scale, int n_q_heads, int n_kv_heads, int head_dim,
                     int page_size, int batch, int max_blocks_per_seq, int num_pages,
                     pa_dtype dtype, int sink_tokens, int window_tokens,
                     int partition_tokens, void *workspace, size_t workspace_bytes,
                     pa_stream_t stream);

/* Workspace bytes pa_decode_window needs (0 when it runs in a single pass). */
size_t pa_decode_window_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                       int head_dim, int page_size, int max_blocks_per_seq,
                                       int sink_tokens, int window_tokens,
                                       int partition_tokens);

/* The partition size pa_decode would use (0 = a single pass, no workspace)
 * for these arguments and partition_tokens (0 = automatic), on the current
 * device.  Returns a negative PA_ERR_* on invalid arguments. */
int pa_decode_partition_tokens(int batch, int n_q_heads, int n_kv_heads,
                               int head_dim, int page_size,
                               int max_blocks_per_seq, int partition_tokens);

/* Workspace bytes pa_decode needs for the same arguments (0 when it runs in a
 * single pass).  Layout: float [batch][n_q_heads][n_parts][head_dim + 4] of
 * rows (O[0..head_dim-1], m, l, 2 unused) with m in natural-log units --
 * partial states of one partition or of the consecutive partitions one CTA
 * holds -- then, at the next 16-byte boundary, one int32 arrival counter per
 * (sequence, head group). */
size_t pa_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                int head_dim, int page_size,
                                int max_blocks_per_seq, int partition_tokens);

/*
 * pa_merge_partials -- the exact merge of partition states on its own (the
 * same arithmetic pa_decode runs in the last CTA of each head group).
 *
 * For row (b, h) with n = ceil(ctx_lens[b] / partition_tokens) valid parts
 * p < n (parts at p >= n are not read):
 *   M = max_p m_p,  l = sum_p e^(m_p - M) l_p,  out = sum_p e^(m_p - M) O_p / l
 * (the exponent law e^(a+b) = e^a e^b of ch. 19 19.6.2, applied to two
 * summarised chunks).  A part with l_p = 0 contributes nothing; a row with
 * none writes zeros.
 *   partials  device float [batch][n_q_heads][n_parts][head_dim + 4], rows
 *             (O_p[0..head_dim-1], m_p, l_p, 2 unused), 16-byte aligned
 *   out       device float [batch][n_q_heads][head_dim]
 */
int pa_merge_partials(const float *partials, const int32_t *ctx_lens,
                      float *out, int batch, int n_q_heads, int head_dim,
                      int n_parts, int partition_tokens, pa_stream_t stream);

/*
 * pa_append_kv -- write the K and V rows of new tokens into their pages.
 *
 * Token j (0 <= j < n_tok) belongs to sequence seq_idx[j] at logical position
 * pos[j]; for every kv head its rows k_new[j][g], v_new[j][g] are stored at
 * page block_table[seq_idx[j]][pos[j] / page_size], slot pos[j] % page_size.
 * This is the new-KV write of a decode step ("吞吐与延迟的系统模型", section 4:
 * 2LBd_kv b_kv bytes written per step).  The block table must already map
 * the position's block (allocating pages is the caller's business).
 *   k_new, v_new  device, [n_tok][n_kv_heads][head_dim], dtype, 16-B aligned
 *   k_cache, v_cache  device, written in place
 *   seq_idx, pos  device int32 [n_tok]
 * Two tokens must not target the same (page, slot): the order of such writes
 * is unspecified.  A bad seq_idx/pos/page skips that token and records
 * PA_ERR_BAD_INDEX / PA_ERR_BAD_BLOCK.
 */
int pa_append_kv(const void *k_new, const void *v_new, void *k_cache,
                 void *v_cache, const int32_t *block_table,
                 const int32_t *seq_idx, const int32_t *pos, int n_tok,
                 int n_kv_heads, int head_dim, int page_size, int batch,
                 int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                 pa_stream_t stream);

/*
 * pa_prefill_paged -- chunked-prefill attention of n_new new query tokens per
 * sequence over the paged cache, causal.
 *
 * ctx_lens[b] counts tokens cached before the chunk; the chunk's own K/V rows
 * must already be stored (e.g. by pa_append_kv) at positions ctx_lens[b] ..
 * ctx_lens[b] + n_new - 1.  Query i of sequence b attends keys
 * 0 .. ctx_lens[b] + i (prefill over the cache, ch. 19 19.3.1; tiled as the
 * FlashAttention forward of 19.6.3 with the online recurrence of 19.6.2).
 *   q    device, [batch][n_new][n_q_heads][head_dim], dtype
 *   out  device float [batch][n_new][n_q_heads][head_dim]
 * Same cache, table and head arguments as pa_decode.
 */
int pa_prefill_paged(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, const int32_t *ctx_lens,
                     int n_new, float *out, float scale, int n_q_heads,
                     int n_kv_heads, int head_dim, int page_size, int batch,
                     int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                     pa_stream_t stream);

/*
 * pa_prefill_paged_split -- pa_prefill_paged with each sequence's keys cut
 * into partitions whose partial states (O, m, l) are merged exactly.
 *
 * Computes what pa_prefill_paged computes (same arguments, same result up to
 * rounding order).  When there are few (query, head) row tiles -- a short
 * chunk over a long context, and in particular the verify step of
 * speculative decoding, where the gamma drafted tokens are attended in one
 * pass with causal masking among themselves (ch. 19 "推理系统与性能工程",
 * speculative sampling) -- a CTA per row tile leaves most SMs idle.  Here
 * each CTA also takes one key range of partition_tokens keys, writes its
 * rows' partial states, and a merge applies the exponent law of 19.6.2.
 *   partition_tokens  0 = choose (see pa_prefill_partition_tokens), else a
 *                     multiple of 128 (PA_ERR_PARTITION otherwise)
 *   workspace         device float [batch][n_new][n_q_heads][n_parts]
 *                     [head_dim + 4], 16-byte aligned, at least
 *                     pa_prefill_workspace_size(...) bytes; owned by the
 *                     caller, overwritten; may be NULL when that size is 0.
 * Returns PA_ERR_WORKSPACE if the workspace is missing or too small.
 */
int pa_prefill_paged_split(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *ctx_lens,
                           int n_new, float *out, float scale, int n_q_heads,
                           int n_kv_heads, int head_dim, int page_size, int batch,
                           int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                           int partition_tokens, void *workspace,
                           size_t workspace_bytes, pa_stream_t stream);

/*
 * The key-range size pa_prefill_paged_split uses for these shapes (0 = no
 * split), or a negative PA_ERR_* for invalid arguments.  The automatic
 * choice splits only when there are fewer row-tile CTAs than SMs, into
 * ranges of at least 512 keys: as many as fit one wave of one CTA per SM,
 * or, when that wave would leave more than 30% of the SMs idle, as fill two.
 */
int pa_prefill_partition_tokens(int batch, int n_new, int n_q_heads, int n_kv_heads,
                                int head_dim, int page_size, int max_blocks_per_seq,
                                int partition_tokens);

/* Workspace bytes pa_prefill_paged_split needs (0 when it does not split). */
size_t pa_prefill_workspace_size(int batch, int n_new, int n_q_heads, int n_kv_heads,
                                 int head_dim, int page_size, int max_blocks_per_seq,
                                 int partition_tokens);

/*
 * Page pool with reference counts, and copy-on-write (prefix sharing).
 *
 * PagedAttention lets the block tables of several requests point to the same
 * physical block; a block shared that way is reference-counted and copied
 * before one of its users writes into it (ch. 19 "推理系统与性能工程", 19.7.3).
 * The pool is a host-side allocator of the pages [0, num_pages) of one K/V
 * cache pair: it counts, per page, the block-table entries that point to it.
 * The attention entry points read through the tables and need nothing else:
 * aliased entries are transparent to them.  A pool is an opaque handle owned
 * by the caller; its functions may be called from several host threads.
 * Tables passed to the pool are HOST int32 arrays (the caller uploads them).
 * Every function validates before it changes anything: on an error the pool
 * is as it was.
 */
typedef struct pa_pool pa_pool;

/* A pool of num_pages free pages (NULL if num_pages <= 0 or out of memory). */
pa_pool *pa_pool_create(int num_pages);
void pa_pool_destroy(pa_pool *pool);

/* Number of free pages, or PA_ERR_NULL. */
int pa_pool_free_pages(pa_pool *pool);

/* Block-table entries pointing at `page` (0 = free), or PA_ERR_SHAPE. */
int pa_pool_refcount(pa_pool *pool, int page);

/* Takes n free pages (reference count 1 each) into pages[0..n); returns
 * PA_ERR_POOL_EMPTY and takes nothing if fewer than n are free. */
int pa_pool_alloc(pa_pool *pool, int n, int32_t *pages);

/* One more reference to each page listed (a forked sequence's table now
 * points to them too); negative entries (unmapped blocks) are skipped.
 * PA_ERR_POOL_STATE if a listed page is free. */
int pa_pool_share(pa_pool *pool, const int32_t *pages, int n);

/* One reference fewer to each page listed; a page reaching 0 returns to the
 * free list.  Negative entries are skipped.  PA_ERR_POOL_STATE if a page
 * would drop below 0 (a page listed k times needs k references). */
int pa_pool_release(pa_pool *pool, const int32_t *pages, int n);

/*
 * Prepares the write of token position `pos` of one sequence whose host
 * block-table row is table[0 .. max_blocks):
 *   block pos / page_size unmapped (< 0): a fresh page is mapped; returns 0;
 *   mapped and used by this table only: nothing to do; returns 0;
 *   mapped and shared: copy-on-write -- a fresh page is mapped in its place,
 *     the shared page loses this reference, *copy_src / *copy_dst receive the
 *     (old, new) pair for pa_copy_pages; returns 1.
 * *copy_src = *copy_dst = -1 when no copy is due.  Negative PA_ERR_* on bad
 * arguments, PA_ERR_POOL_EMPTY when no page is free, PA_ERR_POOL_STATE when
 * the table maps a page the pool holds as free.
 */
int pa_pool_prepare_append(pa_pool *pool, int32_t *table, int max_blocks, int page_size,
                           int pos, int32_t *copy_src, int32_t *copy_dst);

/*
 * pa_copy_pages -- on the device, copies page src[i] to page dst[i] of both
 * caches, every kv head (the copy of copy-on-write), for i < n.
 *   k_cache, v_cache  device [num_pages][n_kv_heads][page_size][head_dim],
 *                     16-byte aligned
 *   src, dst          DEVICE int32 [n]; no dst may equal any src (the copies
 *                     run in parallel)
 * An out-of-range page skips that pair and records PA_ERR_BAD_BLOCK in the
 * status word.  Asynchronous on `stream`.
 */
int pa_copy_pages(void *k_cache, void *v_cache, const int32_t *src, const int32_t *dst,
                  int n, int n_kv_heads, int head_dim, int page_size, int num_pages,
                  pa_dtype dtype, pa_stream_t stream);

/*
 * pa_topm_retain -- budgeted global top-M KV retention (ch. 19 "推理系统与
 * 性能工程", 19.4.3, KV-cache compression by eviction).
 *
 * scores[l][h][t] rates the K/V row of token t for layer l, head h (e.g. the
 * attention mass it received).  Position `current` (C, the generation
 * position) of every (layer, head) is kept unconditionally: L*H rows.  Every
 * other (l, h, t) is a candidate, and the candidates compete for the
 * remaining budget - L*H rows in one global order, key (-score, l, h, t)
 * ascending: higher score first, ties by lower layer, then head, then token.
 * The key is a total order, so the kept set is unique.  budget <= L*H keeps
 * only the current positions; a budget above the candidates keeps all.
 * -0.0 ranks as 0.0; a NaN score ranks after every number.
 *   scores         device float [n_layers][n_heads][n_tokens], 16-B aligned
 *   keep           device uint8 [n_layers][n_heads][n_tokens], 16-B aligned;
 *                  written: 1 = kept
 *   kept_per_head  device int32 [n_layers][n_heads] or NULL; written: the
 *                  kept rows of each (layer, head) (they differ: the budget
 *                  is global)
 *   workspace      device, pa_topm_workspace_size bytes, 16-B aligned: about
 *                  8 bytes per element (the select's candidate list, an index
 *                  and a key, can hold every element) plus 21 KiB and 4 bytes
 *                  per 4096 elements
 * PA_ERR_SHAPE for non-positive sizes, more than 2^31 - 2^13 elements, current
 * outside [0, n_tokens) or a negative budget; PA_ERR_WORKSPACE when
 * workspace_bytes is below pa_topm_workspace_size.  Asynchronous on `stream`.
 */
size_t pa_topm_workspace_size(int n_layers, int n_heads, int n_tokens);
int pa_topm_retain(const float *scores, int n_layers, int n_heads, int n_tokens, int current,
                   long long budget, uint8_t *keep, int32_t *kept_per_head, void *workspace,
                   size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_cascade -- decode of `batch` forks of one shared prefix, reading
 * the prefix's K/V once for all of them.
 *
 * Prefix sharing (ch. 19 "推理系统与性能工程", 19.7.3: the block tables of
 * several requests point to the same physical pages): fork b attends the
 * prefix_len tokens of the shared prefix (pages prefix_table[0 ..
 * prefix_blocks - 1], device) followed by its own ctx_lens[b] tokens (pages
 * block_table[b][..], its own table starting at its first own token).  The
 * result is pa_decode's over the concatenated sequence.  Instead of every
 * fork streaming the prefix again, the forks' queries are attended to the
 * prefix together -- one sequence of `batch` queries that all see every
 * prefix key, on the tensor-core prefill kernel, cut into key ranges -- each
 * fork's own tokens by the decode kernel, and the partial states (O, m, l) of
 * both merged exactly (the exponent law of 19.6.2).
 *   q, out            [batch][n_q_heads][head_dim] (q dtype, out float)
 *   prefix_len        1 .. prefix_blocks * page_size
 *   block_table       [batch][max_blocks_per_seq]; ctx_lens[b] >= 0 (0: the
 *                     fork has no tokens of its own yet)
 *   partition_tokens  0 = choose, else a multiple of 128: the prefix's key
 *                     ranges
 *   workspace         device, pa_decode_cascade_workspace_size(...) bytes,
 *                     16-byte aligned, owned by the caller; contents on
 *                     entry do not matter
 * Returns PA_ERR_SHAPE for a prefix_len outside that range, PA_ERR_WORKSPACE
 * for a missing or short workspace; otherwise as pa_decode.  Asynchronous on
 * `stream` (three launches).
 */
int pa_decode_cascade(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *prefix_table, int prefix_len, int prefix_blocks,
                      const int32_t *block_table, const int32_t *ctx_lens, float *out,
                      float scale, int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                      int batch, int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                      int partition_tokens, void *workspace, size_t workspace_bytes,
                      pa_stream_t stream);
/* The workspace pa_decode_cascade needs for these shapes (0 if invalid). */
size_t pa_decode_cascade_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                        int page_size, int prefix_blocks, int prefix_len,
                                        int partition_tokens);

/*
 * pa_decode_static_workspace -- pa_decode for callers that cannot allocate.
 *
 * The pages have no counterpart to this entry point: it is a convenience of
 * this library.  Some callers cannot call cudaMalloc: code embedded in a host
 * framework that owns every device allocation (a private allocation would
 * bypass its allocator and its accounting), code on a latency-critical path
 * where cudaMalloc/cudaFree may synchronise the whole device, or code that
 * only speaks this C ABI and has no allocator.  This entry point computes
 * exactly what pa_decode computes, with the same arguments minus the
 * workspace: the split-K partial states go to a 16 MiB array that lives in
 * the library's device image (every GPU that loads the library holds it until
 * the process exits).  It allocates nothing and frees nothing.
 *
 * Limit: a call whose partition plan needs more than 16 MiB of scratch
 * (pa_decode_workspace_size() > 16 MiB; about batch * n_q_heads * n_parts *
 * (head_dim + 4) * 4 bytes above that) returns PA_ERR_SCRATCH_LIMIT and
 * launches nothing.
 * The first call in a CUDA context looks up the array's device address (with
 * that context's device current) and caches it under the context's unique
 * id, so a device reset or a second context on the same device looks it up
 * again; make that first call before any stream capture.  Every call shares
 * the one array and leaves its contents behind;
 * nothing in it needs to start at zero (each call clears its own arrival
 * counters on the stream first).  Calls that overlap on the GPU (two
 * streams, or two host threads, with split-K plans) race on the array: the
 * caller must order them.
 */
int pa_decode_static_workspace(const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *block_table,
                               const int32_t *ctx_lens, float *out, float scale,
                               int n_q_heads, int n_kv_heads, int head_dim,
                               int page_size, int batch, int max_blocks_per_seq,
                               int num_pages, pa_dtype dtype,
                               int partition_tokens, pa_stream_t stream);

/*
 * pa_last_device_error -- synchronise `stream`, then return and clear the
 * device status word (PA_OK if no kernel recorded an error since the last
 * call).  The word is shared by every stream of the device: it reports the
 * first error any pa kernel recorded.  Returns PA_ERR_CUDA if the stream
 * itself reports a CUDA error.
 */
int pa_last_device_error(pa_stream_t stream);

/*
 * pa_selftest_wait_timeout -- exercise the failure path of the kernels'
 * bounded waits.  The pages have no counterpart: every copy or hand-off a pa
 * kernel waits for is waited on for at most 2 s, after which the kernel
 * records PA_ERR_TIMEOUT in the device status word and leaves without
 * faulting.  This launches one warp that waits on a barrier phase nothing
 * completes, so the next pa_last_device_error() returns PA_ERR_TIMEOUT after
 * about 2 s, and later calls run normally.  Asynchronous on `stream`.
 */
int pa_selftest_wait_timeout(pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
