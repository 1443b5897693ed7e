// pa_decode_static.cu -- pa_decode for callers that cannot allocate device
// memory: the split-K partial states go to a fixed array that lives in the
// library's own device image instead of a caller-supplied workspace.
//
// Who needs this: a caller embedded in a host framework that owns every
// device allocation (a private cudaMalloc would bypass its allocator and its
// memory accounting), a caller on a latency-critical path where cudaMalloc and
// cudaFree may synchronise the whole device, or a caller that only speaks the
// C ABI and has no allocator at hand.  Such callers still pass q, the caches,
// the tables and the output; only the scratch comes from here.
#include "pa_internal.h"

namespace {

// Largest split-K workspace this entry point can serve.  Every GPU that loads
// this part of the library holds the array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of the array in the current context (the symbol's name in
// host code is only a stand-in).  Looked up once per CUDA context and cached
// under the context's unique id, so a device reset or another context on
// the same device never sees a stale address.
void *scratch_address() {
  static pa::ContextCache<void *> cache;
  void *addr = nullptr;
  if (cache.get(pa::current_context_id(), &addr)) return addr;
  if (cudaGetSymbolAddress(&addr, g_decode_scratch) != cudaSuccess) return nullptr;
  cache.put(pa::current_context_id(), addr);  // the lookup made a context current
  return addr;
}

}  // namespace

extern "C" int pa_decode_static_workspace(
    const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, const int32_t *ctx_lens, float *out, float scale,
    int n_q_heads, int n_kv_heads, int head_dim, int page_size, int batch,
    int max_blocks_per_seq, int num_pages, pa_dtype dtype, int partition_tokens,
    pa_stream_t stream) {
  // Same argument checks and partition plan as pa_decode; the plan decides
  // how much scratch the call needs.
  const int part = pa_decode_partition_tokens(batch, n_q_heads, n_kv_heads, head_dim,
                                              page_size, max_blocks_per_seq,
                                              partition_tokens);
  if (part < 0) return part;
  const size_t need = pa_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
                                               page_size, max_blocks_per_seq,
                                               partition_tokens);
  if (need > kStaticScratchBytes) return PA_ERR_SCRATCH_LIMIT;
  void *scratch = nullptr;
  if (need > 0) {
    scratch = scratch_address();
    if (!scratch) return PA_ERR_CUDA;
  }
  // Every partial state the merge reads is written by the same call first,
  // and pa_decode clears the arrival counters before its kernel runs, so the
  // array never needs clearing by the caller.
  return pa_decode(q, k_cache, v_cache, block_table, ctx_lens, out, scale, n_q_heads,
                   n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq,
                   num_pages, dtype, partition_tokens, scratch,
                   need > 0 ? kStaticScratchBytes : 0, stream);
}
