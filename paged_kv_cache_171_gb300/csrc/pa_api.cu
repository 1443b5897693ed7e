// pa_api.cu -- the C ABI of libpa: argument validation, dispatch, the device
// status word, tensor-map encoding, and the KV-append kernel.
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// One status word per device: the first data-dependent error any kernel saw.
__device__ int g_status_word;

uint64_t current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;  // nothing cached: every lookup is made again
  return id;
}

int *device_status() {
  static ContextCache<int *> cache;
  int *addr = nullptr;
  if (cache.get(current_context_id(), &addr)) return addr;
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  cache.put(current_context_id(), static_cast<int *>(p));  // the lookup made one current
  return static_cast<int *>(p);
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                   void *, const cuuint64_t *, const cuuint64_t *,
                                   const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

int make_rows_map(CUtensorMap *map, const void *base, uint64_t rows,
                  int head_dim, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

namespace {

// ---- KV append: one thread moves 16 bytes of K and 16 bytes of V
__global__ void __launch_bounds__(256)
    append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                  uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                  const int32_t *__restrict__ block_table,
                  const int32_t *__restrict__ seq_idx,
                  const int32_t *__restrict__ pos, int *status, long total,
                  int n_kv_heads, int chunks, int batch, int max_blocks,
                  int num_pages) {
  griddep_release();
  griddep_wait();  // the rows may come from the previous kernel in the stream
  const long idx = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int c = static_cast<int>(idx % chunks);
  const long jg = idx / chunks;
  const int g = static_cast<int>(jg % n_kv_heads);
  const long j = jg / n_kv_heads;
  const bool reporter = (c == 0 && g == 0);
  const int b = seq_idx[j];
  const int t = pos[j];
  if (b < 0 || b >= batch || t < 0 || t >= max_blocks * kPageSize) {
    if (reporter) record_error(status, PA_ERR_BAD_INDEX);
    return;
  }
  const int page = block_table[static_cast<size_t>(b) * max_blocks + t / kPageSize];
  if (page < 0 || page >= num_pages) {
    if (reporter) record_error(status, PA_ERR_BAD_BLOCK);
    return;
  }
  const size_t dst =
      ((static_cast<size_t>(page) * n_kv_heads + g) * kPageSize + t % kPageSize) *
          chunks + c;
  const size_t src = static_cast<size_t>(jg) * chunks + c;
  k_cache[dst] = k_new[src];
  v_cache[dst] = v_new[src];
}

}  // namespace

int launch_append(const void *k_new, const void *v_new, void *k_cache,
                  void *v_cache, const int32_t *block_table,
                  const int32_t *seq_idx, const int32_t *pos, int *status,
                  int n_tok, int n_kv_heads, int head_dim, int batch,
                  int max_blocks, int num_pages, cudaStream_t stream) {
  const int chunks = head_dim / 8;  // 16-byte chunks per row
  const long total = static_cast<long>(n_tok) * n_kv_heads * chunks;
  const int threads = 256;
  const long blocks = (total + threads - 1) / threads;
  const cudaError_t e = launch_pdl(
      append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), block_table, seq_idx,
      pos, status, total, n_kv_heads, chunks, batch, max_blocks, num_pages);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_common(int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                 int batch, int max_blocks, int num_pages, int dtype) {
  if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) return PA_ERR_HEADS;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_HEAD_DIM;
  if (page_size != kPageSize) return PA_ERR_PAGE_SIZE;
  if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_DTYPE;
  if (batch <= 0 || batch > 65535 || max_blocks <= 0 || num_pages <= 0)
    return PA_ERR_SHAPE;
  // Token positions and TMA row coordinates are 32-bit.
  if (static_cast<int64_t>(max_blocks) * page_size > (int64_t(1) << 30)) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(num_pages) * n_kv_heads * page_size >= (int64_t(1) << 31))
    return PA_ERR_SHAPE;
  return PA_OK;
}

int current_status_ptr(int **status) {
  *status = device_status();
  return *status ? PA_OK : PA_ERR_CUDA;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

// Partition plan of pa_decode: pages per partition (0 = single pass) and the
// partition count.  Automatic mode, with R = resident CTAs (2 per SM) and
// I = batch * kv heads * head tiles (CTAs of a single pass):
//   I <  3R/4: cut sequences into about R / I equal partitions, so that one
//              wave of CTAs keeps enough copies in flight, of 16 to 256 pages
//              each; on the CUDA-core path (group tile 1: MHA), whose per-page
//              arithmetic is the slow part of a small call, about R / I CTA
//              slots of single-warp partitions of 2 pages or more instead
//              (a 4 MB call then holds all its pages in flight at once:
//              16 heads x 512 tokens, kernel 7.6 -> 6.2 us; 1 x 32 heads x 4k
//              and 2 x 32 x 2k tokens 25-28% faster; GQA calls were slower
//              with the bigger merge);
//   I <  R   : a single pass (one wave, no merge);
//   I >= R   : cut into 4 partitions of >= 32 pages, so that one long
//              sequence of a ragged batch cannot make a tail of its own.
int decode_plan(int batch, int n_q_heads, int n_kv_heads, int max_blocks,
                int partition_tokens, int *part_pages, int *n_parts,
                int *warp_parts = nullptr) {
  if (partition_tokens < 0 || partition_tokens % kPageSize) return PA_ERR_PARTITION;
  int pp = partition_tokens / kPageSize;
  if (pp == 0) {
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const int64_t resident = static_cast<int64_t>(sms) * 2;
    const int64_t items = static_cast<int64_t>(batch) * n_kv_heads *
                          ((n_q_heads / n_kv_heads) / group_tile(n_q_heads / n_kv_heads));
    if (items * 4 < resident * 3) {
      const int64_t want = resident / items > 1 ? resident / items : 1;
      int64_t per = (max_blocks + want - 1) / want;
      if (group_tile(n_q_heads / n_kv_heads) == 1 && per <= 32) {
        // short partitions go to single warps (below): about `want` CTA
        // slots per item is kDecodeWarps partitions per slot
        per = (max_blocks + want * kDecodeWarps - 1) / (want * kDecodeWarps);
        if (per < 2) per = 2;
      } else if (per < 16) {
        per = 16;
      }
      if (per > 256) per = 256;  // longer ranges leave a slow tail (measured at 32k)
      pp = static_cast<int>(per);
    } else if (items < resident) {
      pp = 0;
    } else {
      int64_t per = (max_blocks + 3) / 4;
      if (per < 32) per = 32;
      pp = static_cast<int>(per);
    }
  }
  if (pp >= max_blocks) pp = 0;
  *part_pages = pp;
  *n_parts = pp ? (max_blocks + pp - 1) / pp : 1;
  // Small partitions: let each warp own whole partitions (no cross-warp merge
  // inside the CTA, prefetch across its partition boundaries), with enough
  // partitions per warp that the grid is about four waves of resident CTAs.
  // Several CTAs per SM over the kernel's life balance its tail: at 32k
  // tokens x 4 sequences x 8 kv heads in 512-token partitions, one partition
  // per warp (512 CTAs) runs 5% faster than two (256 CTAs, one wave).
  int wp = 0;
  if (pp > 0 && pp <= 32 && *n_parts >= kDecodeWarps) {
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const int64_t resident = static_cast<int64_t>(sms) * 2;
    const int64_t items = static_cast<int64_t>(batch) * n_kv_heads *
                          ((n_q_heads / n_kv_heads) / group_tile(n_q_heads / n_kv_heads));
    const int64_t warps = 4 * resident * kDecodeWarps;
    int64_t w = (items * *n_parts + warps - 1) / warps;
    const int64_t wmax = (*n_parts + kDecodeWarps - 1) / kDecodeWarps;
    wp = static_cast<int>(w < 1 ? 1 : (w > wmax ? wmax : w));
  }
  if (warp_parts) *warp_parts = wp;
  return PA_OK;
}

// Key-range partitions of the chunked prefill (multiples of 128 keys, the
// kernel's key tile).  A CTA holds two row tiles of 128 (query, head) rows
// and one CTA fits an SM; with fewer CTAs than SMs, a sequence's keys are cut
// into as many ranges as fit one wave of CTAs (equal ranges finish together,
// and every further wave pays the CTAs' start-up and a bigger merge again:
// at 4 x 32k keys, 64/8 heads, 128 CTAs in one wave ran 96 us, 288 in two
// waves 106 us), or as fill two waves when one wave would leave more than
// 30% of the SMs idle; each range at least 512 keys.
int prefill_plan(int batch, int n_new, int n_q_heads, int n_kv_heads, int max_blocks,
                 int partition_tokens, int *part_tokens, int *n_parts) {
  constexpr int kTile = 128;
  if (partition_tokens < 0 || partition_tokens % kTile) return PA_ERR_PARTITION;
  const int64_t max_tokens = static_cast<int64_t>(max_blocks) * kPageSize;
  int64_t per = partition_tokens;
  if (per == 0) {
    const int gt = group_tile(n_q_heads / n_kv_heads);
    const int64_t rows_per_cta = 2 * (128 / gt);  // queries of two row tiles
    const int64_t items = static_cast<int64_t>(batch) * n_kv_heads *
                          ((n_q_heads / n_kv_heads) / gt) *
                          ((n_new + rows_per_cta - 1) / rows_per_cta);
    const int sms = sm_count() > 0 ? sm_count() : 148;
    if (items < sms) {
      const int64_t one_wave = sms / items;
      const int64_t want = 10 * items * one_wave >= 7 * sms ? one_wave : (2 * sms) / items;
      per = (max_tokens + want - 1) / want;
      per = (per + kTile - 1) / kTile * kTile;
      if (per < 4 * kTile) per = 4 * kTile;
    }
  }
  if (per <= 0 || per >= max_tokens) {
    *part_tokens = 0;
    *n_parts = 1;
  } else {
    *part_tokens = static_cast<int>(per);
    *n_parts = static_cast<int>((max_tokens + per - 1) / per);
  }
  return PA_OK;
}

// Plan of a cascade decode: the shared prefix's key ranges, cut as
// pa_prefill_paged_split would cut one sequence whose n_new queries are the
// forks, but counting only the ranges that hold prefix keys.  Returns the
// range size in tokens (0: one range) and their number.
int cascade_plan(int batch, int n_q_heads, int n_kv_heads, int prefix_blocks, int prefix_len,
                 int partition_tokens, int *part_tokens, int *n_ranges) {
  int pt = 0, np = 1;
  const int rc = prefill_plan(1, batch, n_q_heads, n_kv_heads, prefix_blocks, partition_tokens,
                              &pt, &np);
  if (rc) return rc;
  *part_tokens = pt;
  *n_ranges = pt ? (prefix_len + pt - 1) / pt : 1;
  return PA_OK;
}

int check_cascade(int batch, int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                  int max_blocks, int num_pages, int dtype, int prefix_blocks, int prefix_len) {
  const int rc = check_common(n_q_heads, n_kv_heads, head_dim, page_size, batch, max_blocks,
                              num_pages, dtype);
  if (rc) return rc;
  if (batch > (1 << 20) || prefix_blocks <= 0 || prefix_len < 1 ||
      static_cast<int64_t>(prefix_len) > static_cast<int64_t>(prefix_blocks) * page_size ||
      static_cast<int64_t>(prefix_blocks) * page_size > (int64_t(1) << 30))
    return PA_ERR_SHAPE;
  return PA_OK;
}

size_t cascade_workspace_bytes(int batch, int n_q_heads, int head_dim, int n_ranges) {
  return static_cast<size_t>(batch) * n_q_heads * (n_ranges + 1) * (head_dim + 4) *
         sizeof(float);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

const char *pa_strerror(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_HEADS: return "PA_ERR_HEADS: bad head counts";
    case PA_ERR_HEAD_DIM: return "PA_ERR_HEAD_DIM: head_dim must be 64 or 128";
    case PA_ERR_PAGE_SIZE: return "PA_ERR_PAGE_SIZE: page_size must be 16";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: bad or too large sizes";
    case PA_ERR_DTYPE: return "PA_ERR_DTYPE: dtype must be PA_BF16 or PA_F16";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: pointer not 16-byte aligned";
    case PA_ERR_PARTITION:
      return "PA_ERR_PARTITION: partition_tokens not a multiple of page_size (decode) or 128 "
             "(prefill)";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA call failed";
    case PA_ERR_BAD_BLOCK: return "PA_ERR_BAD_BLOCK: block-table entry outside the page pool";
    case PA_ERR_BAD_CTX: return "PA_ERR_BAD_CTX: context length outside [0, max_blocks*page_size]";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: a bounded wait for a copy ran out";
    case PA_ERR_BAD_INDEX: return "PA_ERR_BAD_INDEX: append seq_idx/pos outside the table";
    case PA_ERR_SCRATCH_LIMIT:
      return "PA_ERR_SCRATCH_LIMIT: needs more split-K scratch than the 16 MiB static array";
    case PA_ERR_POOL_EMPTY: return "PA_ERR_POOL_EMPTY: not enough free pages in the pool";
    case PA_ERR_POOL_STATE: return "PA_ERR_POOL_STATE: a page that is not in use";
    default: return "unknown pa status";
  }
}

int pa_decode_partition_tokens(int batch, int n_q_heads, int n_kv_heads,
                               int head_dim, int page_size,
                               int max_blocks_per_seq, int partition_tokens) {
  int rc = check_common(n_q_heads, n_kv_heads, head_dim, page_size, batch,
                        max_blocks_per_seq, 1, PA_BF16);
  if (rc) return rc;
  int pp = 0, np = 1;
  rc = decode_plan(batch, n_q_heads, n_kv_heads, max_blocks_per_seq,
                   partition_tokens, &pp, &np);
  return rc ? rc : pp * kPageSize;
}

size_t pa_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                int head_dim, int page_size,
                                int max_blocks_per_seq, int partition_tokens) {
  if (check_common(n_q_heads, n_kv_heads, head_dim, page_size, batch,
                   max_blocks_per_seq, 1, PA_BF16))
    return 0;
  int pp = 0, np = 1;
  if (decode_plan(batch, n_q_heads, n_kv_heads, max_blocks_per_seq,
                  partition_tokens, &pp, &np))
    return 0;
  if (np <= 1) return 0;
  return decode_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim, np);
}

}  // extern "C"

namespace pa {
namespace {
// Pages a sequence's query may attend: every table entry, or with an
// attention sink and a window at most ceil(sink/16) + ceil(window/16) + 1.
int attended_blocks(int max_blocks, int sink, int window) {
  if (window < 0) return max_blocks;
  const int64_t n = (static_cast<int64_t>(sink) + 15) / 16 +
                    (static_cast<int64_t>(window) + 15) / 16 + 1;
  return static_cast<int>(n < max_blocks ? n : max_blocks);
}

int decode_impl(const void *q, const void *k_cache, const void *v_cache,
                const int32_t *block_table, const int32_t *ctx_lens, float *out,
                float scale, int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                int batch, int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                int sink, int window, int partition_tokens, void *workspace,
                size_t workspace_bytes, pa_stream_t stream, const void *k_new = nullptr,
                const void *v_new = nullptr) {
  if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !out)
    return PA_ERR_NULL;
  int rc = check_common(n_q_heads, n_kv_heads, head_dim, page_size, batch,
                        max_blocks_per_seq, num_pages, dtype);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_ALIGN;
  int pp = 0, np = 1, wp = 0;
  rc = decode_plan(batch, n_q_heads, n_kv_heads, attended_blocks(max_blocks_per_seq, sink, window),
                   partition_tokens, &pp, &np, &wp);
  if (rc) return rc;
  if (np > 1) {
    const size_t need = decode_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim, np);
    if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_ALIGN;
  }
  DecodeLaunch a;
  rc = current_status_ptr(&a.status);
  if (rc) return rc;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.out = out;
  a.workspace = np > 1 ? static_cast<float *>(workspace) : nullptr;
  a.scale = scale;
  a.n_q_heads = n_q_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  a.batch = batch;
  a.max_blocks = max_blocks_per_seq;
  a.num_pages = num_pages;
  a.bf16 = dtype == PA_BF16;
  a.part_pages = pp;
  a.n_parts = np;
  a.warp_parts = wp;
  a.sink = sink;
  a.window = window;
  a.k_new = k_new;
  a.v_new = v_new;
  return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace
}  // namespace pa

extern "C" {

int pa_decode(const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_table, const int32_t *ctx_lens, float *out,
              float scale, int n_q_heads, int n_kv_heads, int head_dim,
              int page_size, int batch, int max_blocks_per_seq, int num_pages,
              pa_dtype dtype, int partition_tokens, void *workspace,
              size_t workspace_bytes, pa_stream_t stream) {
  return decode_impl(q, k_cache, v_cache, block_table, ctx_lens, out, scale, n_q_heads,
                     n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq, num_pages,
                     dtype, 0, -1, partition_tokens, workspace, workspace_bytes, stream);
}

int pa_decode_append(const void *q, const void *k_new, const void *v_new, void *k_cache,
                     void *v_cache, const int32_t *block_table, const int32_t *ctx_lens,
                     float *out, float scale, int n_q_heads, int n_kv_heads, int head_dim,
                     int page_size, int batch, int max_blocks_per_seq, int num_pages,
                     pa_dtype dtype, int partition_tokens, void *workspace,
                     size_t workspace_bytes, pa_stream_t stream) {
  if (!k_new || !v_new) return PA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new)) return PA_ERR_ALIGN;
  return decode_impl(q, k_cache, v_cache, block_table, ctx_lens, out, scale, n_q_heads,
                     n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq, num_pages,
                     dtype, 0, -1, partition_tokens, workspace, workspace_bytes, stream, k_new,
                     v_new);
}

int pa_decode_window(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, const int32_t *ctx_lens, float *out,
                     float scale, int n_q_heads, int n_kv_heads, int head_dim,
                     int page_size, int batch, int max_blocks_per_seq, int num_pages,
                     pa_dtype dtype, int sink_tokens, int window_tokens,
                     int partition_tokens, void *workspace, size_t workspace_bytes,
                     pa_stream_t stream) {
  if (sink_tokens < 0 || window_tokens < 0) return PA_ERR_SHAPE;
  return decode_impl(q, k_cache, v_cache, block_table, ctx_lens, out, scale, n_q_heads,
                     n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq, num_pages,
                     dtype, sink_tokens, window_tokens, partition_tokens, workspace,
                     workspace_bytes, stream);
}

size_t pa_decode_window_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                       int head_dim, int page_size, int max_blocks_per_seq,
                                       int sink_tokens, int window_tokens,
                                       int partition_tokens) {
  if (sink_tokens < 0 || window_tokens < 0) return 0;
  return pa_decode_workspace_size(
      batch, n_q_heads, n_kv_heads, head_dim, page_size,
      attended_blocks(max_blocks_per_seq, sink_tokens, window_tokens), partition_tokens);
}

int pa_merge_partials(const float *partials, const int32_t *ctx_lens,
                      float *out, int batch, int n_q_heads, int head_dim,
                      int n_parts, int partition_tokens, pa_stream_t stream) {
  if (!partials || !ctx_lens || !out) return PA_ERR_NULL;
  if (n_q_heads <= 0) return PA_ERR_HEADS;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_HEAD_DIM;
  if (batch <= 0 || batch > 65535 || n_q_heads > 65535 || n_parts <= 0)
    return PA_ERR_SHAPE;
  if (partition_tokens <= 0) return PA_ERR_PARTITION;
  int *status = nullptr;
  int rc = current_status_ptr(&status);
  if (rc) return rc;
  return launch_merge(partials, ctx_lens, out, status, batch, n_q_heads,
                      head_dim, n_parts, partition_tokens,
                      reinterpret_cast<cudaStream_t>(stream));
}

int pa_append_kv(const void *k_new, const void *v_new, void *k_cache,
                 void *v_cache, const int32_t *block_table,
                 const int32_t *seq_idx, const int32_t *pos, int n_tok,
                 int n_kv_heads, int head_dim, int page_size, int batch,
                 int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                 pa_stream_t stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_idx || !pos)
    return PA_ERR_NULL;
  int rc = check_common(n_kv_heads, n_kv_heads, head_dim, page_size, batch,
                        max_blocks_per_seq, num_pages, dtype);
  if (rc) return rc;
  if (n_tok < 0) return PA_ERR_SHAPE;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ALIGN;
  if (n_tok == 0) return PA_OK;
  int *status = nullptr;
  rc = current_status_ptr(&status);
  if (rc) return rc;
  return launch_append(k_new, v_new, k_cache, v_cache, block_table, seq_idx, pos,
                       status, n_tok, n_kv_heads, head_dim, batch,
                       max_blocks_per_seq, num_pages,
                       reinterpret_cast<cudaStream_t>(stream));
}

int pa_prefill_paged(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, const int32_t *ctx_lens,
                     int n_new, float *out, float scale, int n_q_heads,
                     int n_kv_heads, int head_dim, int page_size, int batch,
                     int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                     pa_stream_t stream) {
  if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !out)
    return PA_ERR_NULL;
  int rc = check_common(n_q_heads, n_kv_heads, head_dim, page_size, batch,
                        max_blocks_per_seq, num_pages, dtype);
  if (rc) return rc;
  if (n_new < 0 || n_new > (1 << 20)) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(n_new) > static_cast<int64_t>(max_blocks_per_seq) * page_size)
    return PA_ERR_SHAPE;  // the chunk alone would overflow the table
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_ALIGN;
  if (n_new == 0) return PA_OK;
  PrefillLaunch a;
  rc = current_status_ptr(&a.status);
  if (rc) return rc;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.out = out;
  a.scale = scale;
  a.n_new = n_new;
  a.n_q_heads = n_q_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  a.batch = batch;
  a.max_blocks = max_blocks_per_seq;
  a.num_pages = num_pages;
  a.bf16 = dtype == PA_BF16;
  return launch_prefill(a, reinterpret_cast<cudaStream_t>(stream));
}

int pa_prefill_partition_tokens(int batch, int n_new, int n_q_heads, int n_kv_heads,
                                int head_dim, int page_size, int max_blocks_per_seq,
                                int partition_tokens) {
  int rc = check_common(n_q_heads, n_kv_heads, head_dim, page_size, batch,
                        max_blocks_per_seq, 1, PA_BF16);
  if (rc) return rc;
  if (n_new < 0 || n_new > (1 << 20)) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(n_new) > static_cast<int64_t>(max_blocks_per_seq) * page_size)
    return PA_ERR_SHAPE;  // the chunk alone would overflow the table
  int pt = 0, np = 1;
  rc = prefill_plan(batch, n_new, n_q_heads, n_kv_heads, max_blocks_per_seq,
                    partition_tokens, &pt, &np);
  return rc ? rc : pt;
}

size_t pa_prefill_workspace_size(int batch, int n_new, int n_q_heads, int n_kv_heads,
                                 int head_dim, int page_size, int max_blocks_per_seq,
                                 int partition_tokens) {
  if (check_common(n_q_heads, n_kv_heads, head_dim, page_size, batch,
                   max_blocks_per_seq, 1, PA_BF16))
    return 0;
  if (n_new <= 0 || n_new > (1 << 20)) return 0;
  int pt = 0, np = 1;
  if (prefill_plan(batch, n_new, n_q_heads, n_kv_heads, max_blocks_per_seq,
                   partition_tokens, &pt, &np))
    return 0;
  if (np <= 1) return 0;
  return prefill_partials_bytes(batch, n_new, n_q_heads, np, head_dim);
}

int pa_prefill_paged_split(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *ctx_lens,
                           int n_new, float *out, float scale, int n_q_heads,
                           int n_kv_heads, int head_dim, int page_size, int batch,
                           int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                           int partition_tokens, void *workspace, size_t workspace_bytes,
                           pa_stream_t stream) {
  if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !out)
    return PA_ERR_NULL;
  int rc = check_common(n_q_heads, n_kv_heads, head_dim, page_size, batch,
                        max_blocks_per_seq, num_pages, dtype);
  if (rc) return rc;
  if (n_new < 0 || n_new > (1 << 20)) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(n_new) > static_cast<int64_t>(max_blocks_per_seq) * page_size)
    return PA_ERR_SHAPE;  // the chunk alone would overflow the table
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_ALIGN;
  int pt = 0, np = 1;
  rc = prefill_plan(batch, n_new, n_q_heads, n_kv_heads, max_blocks_per_seq,
                    partition_tokens, &pt, &np);
  if (rc) return rc;
  if (np > 1 && n_new > 0) {
    const size_t need = prefill_partials_bytes(batch, n_new, n_q_heads, np, head_dim);
    if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_ALIGN;
  }
  if (n_new == 0) return PA_OK;
  PrefillLaunch a;
  rc = current_status_ptr(&a.status);
  if (rc) return rc;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.out = out;
  a.scale = scale;
  a.n_new = n_new;
  a.n_q_heads = n_q_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  a.batch = batch;
  a.max_blocks = max_blocks_per_seq;
  a.num_pages = num_pages;
  a.bf16 = dtype == PA_BF16;
  a.n_parts = np;
  a.part_tokens = pt;
  a.workspace = np > 1 ? static_cast<float *>(workspace) : nullptr;
  return launch_prefill(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t pa_decode_cascade_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                        int page_size, int prefix_blocks, int prefix_len,
                                        int partition_tokens) {
  if (check_cascade(batch, n_q_heads, n_kv_heads, head_dim, page_size, 1, 1, PA_BF16,
                    prefix_blocks, prefix_len))
    return 0;
  int pt = 0, nr = 1;
  if (cascade_plan(batch, n_q_heads, n_kv_heads, prefix_blocks, prefix_len, partition_tokens,
                   &pt, &nr))
    return 0;
  return cascade_workspace_bytes(batch, n_q_heads, head_dim, nr);
}

int pa_decode_cascade(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *prefix_table, int prefix_len, int prefix_blocks,
                      const int32_t *block_table, const int32_t *ctx_lens, float *out,
                      float scale, int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                      int batch, int max_blocks_per_seq, int num_pages, pa_dtype dtype,
                      int partition_tokens, void *workspace, size_t workspace_bytes,
                      pa_stream_t stream) {
  if (!q || !k_cache || !v_cache || !prefix_table || !block_table || !ctx_lens || !out ||
      !workspace)
    return PA_ERR_NULL;
  int rc = check_cascade(batch, n_q_heads, n_kv_heads, head_dim, page_size,
                         max_blocks_per_seq, num_pages, dtype, prefix_blocks, prefix_len);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace))
    return PA_ERR_ALIGN;
  int pt = 0, nr = 1;
  rc = cascade_plan(batch, n_q_heads, n_kv_heads, prefix_blocks, prefix_len, partition_tokens,
                    &pt, &nr);
  if (rc) return rc;
  if (workspace_bytes < cascade_workspace_bytes(batch, n_q_heads, head_dim, nr))
    return PA_ERR_WORKSPACE;
  int *status = nullptr;
  rc = current_status_ptr(&status);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float *ws = static_cast<float *>(workspace);
  // 1. every fork's queries over the shared prefix at once: one sequence
  //    whose n_new = batch queries all see keys 0 .. prefix_len - 1; partial
  //    states in slots 0 .. nr - 1 of each (fork, head) row
  PrefillLaunch a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = prefix_table;
  a.ctx_lens = ctx_lens;  // not read with shared keys
  a.out = out;            // not written while partial states go to the workspace
  a.status = status;
  a.scale = scale;
  a.n_new = batch;
  a.n_q_heads = n_q_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  a.batch = 1;
  a.max_blocks = prefix_blocks;
  a.num_pages = num_pages;
  a.bf16 = dtype == PA_BF16;
  a.n_parts = nr;
  a.part_tokens = pt;
  a.workspace = ws;
  a.shared_ctx = prefix_len;
  a.ws_slots = nr + 1;
  a.merge = false;
  rc = launch_prefill(a, s);
  if (rc) return rc;
  // 2. each fork's own tokens: a single-pass decode whose state goes to slot
  //    nr (a separate merge folds all rows in parallel: folding the prefix's
  //    states in the decode's epilogue, one element after another, was slower)
  DecodeLaunch d;
  d.q = q;
  d.k_cache = k_cache;
  d.v_cache = v_cache;
  d.block_table = block_table;
  d.ctx_lens = ctx_lens;
  d.out = out;
  d.workspace = nullptr;
  d.status = status;
  d.scale = scale;
  d.n_q_heads = n_q_heads;
  d.n_kv_heads = n_kv_heads;
  d.head_dim = head_dim;
  d.batch = batch;
  d.max_blocks = max_blocks_per_seq;
  d.num_pages = num_pages;
  d.bf16 = dtype == PA_BF16;
  d.part_pages = 0;
  d.n_parts = 1;
  d.warp_parts = 0;
  d.part = ws;
  d.part_stride = nr + 1;
  d.part_slot = nr;
  rc = launch_decode(d, s);
  if (rc) return rc;
  // 3. the exponent law over the nr + 1 states of every row (19.6.2)
  return launch_merge_all(ws, out, status, batch, n_q_heads, head_dim, nr + 1, s);
}

int pa_last_device_error(pa_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  int *status = nullptr;
  if (current_status_ptr(&status)) return PA_ERR_CUDA;
  int value = 0;
  const int zero = 0;
  if (cudaMemcpyAsync(&value, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemcpyAsync(status, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  return value;
}

}  // extern "C"
