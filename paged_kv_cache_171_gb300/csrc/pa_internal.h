// pa_internal.h -- host-side interfaces between the C-ABI layer (pa_api.cu)
// and the translation units that hold the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

#include "pa.h"

namespace pa {

// Unique id of the calling thread's current CUDA context, or 0 while none is
// current.  CUDA never gives two contexts of one process the same id, so
// values cached under it go stale neither after cudaDeviceReset (the next
// primary context has a new id) nor when a second context is made current on
// the same device.
uint64_t current_context_id();

// Values computed once per CUDA context (a symbol's device address, whether a
// kernel attribute is set), keyed by current_context_id().  Thread-safe.
template <class T>
class ContextCache {
 public:
  bool get(uint64_t ctx, T *out) {
    if (ctx == 0) return false;
    std::lock_guard<std::mutex> lock(mu_);
    for (const auto &e : entries_)
      if (e.first == ctx) {
        *out = e.second;
        return true;
      }
    return false;
  }
  void put(uint64_t ctx, T value) {
    if (ctx == 0) return;
    std::lock_guard<std::mutex> lock(mu_);
    for (auto &e : entries_)
      if (e.first == ctx) {
        e.second = value;
        return;
      }
    entries_.emplace_back(ctx, value);
  }

 private:
  std::mutex mu_;
  std::vector<std::pair<uint64_t, T>> entries_;
};

// Raises `kern`'s dynamic shared-memory limit to `bytes`, once per context.
template <class K>
int set_smem_limit(K *kern, int bytes, ContextCache<bool> &done) {
  bool set = false;
  if (done.get(current_context_id(), &set)) return PA_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  done.put(current_context_id(), true);  // the call above made a context current
  return PA_OK;
}

constexpr int kPageSize = 16;  // tokens per page (the only one supported)

// Everything the decode kernels need, already validated by pa_api.cu.
struct DecodeLaunch {
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_table;
  const int32_t *ctx_lens;
  float *out;
  float *workspace;  // partial states, or nullptr for a single pass
  int *status;
  float scale;
  int n_q_heads, n_kv_heads, head_dim, batch, max_blocks, num_pages;
  bool bf16;
  int part_pages;  // pages per partition; 0 = a single pass over the sequence
  int n_parts;     // partitions per sequence (1 for a single pass)
  int warp_parts;  // > 0: each warp owns this many whole partitions
  // Attention sink + sliding window: window >= 0 attends only keys t < sink
  // and t >= T - window (window < 0: every key).  Partitions then cut the
  // attended keys' pages.
  int sink = 0, window = -1;
  // Single pass only (part_pages 0): each row's partial state goes to slot
  // part_slot of part [row][part_stride][head_dim + 4] instead of O / l to
  // out (the own keys of a cascade decode).
  float *part = nullptr;
  int part_stride = 0, part_slot = 0;
  // Fused append (plain decode only): the rows of each sequence's step token
  // (position ctx_lens[b] - 1), [B][Hkv][head_dim], written into the cache
  // (k_cache / v_cache are then written) and attended.
  const void *k_new = nullptr, *v_new = nullptr;
};

constexpr int kDecodeWarps = 4;  // warps per decode CTA

// Largest group tile (heads handled by one CTA) that divides the group size.
inline int group_tile(int group) {
  return (group % 8 == 0) ? 8 : (group % 4 == 0) ? 4 : (group % 2 == 0) ? 2 : 1;
}

int launch_decode(const DecodeLaunch &a, cudaStream_t stream);

// Workspace of a split pa_decode: float partial states [B][Hq][n_parts][D + 4]
// (O_p, m_p, l_p, two unused floats: rows stay 16-byte aligned), then one int
// arrival counter per (sequence, head tile) at the next 16-byte boundary (the
// last CTA of a (sequence, head tile) to arrive merges its partitions).
inline size_t decode_partials_bytes(int batch, int n_q_heads, int n_parts, int head_dim) {
  return static_cast<size_t>(batch) * n_q_heads * n_parts * (head_dim + 4) * sizeof(float);
}
inline size_t decode_counters_offset(int batch, int n_q_heads, int n_parts, int head_dim) {
  return (decode_partials_bytes(batch, n_q_heads, n_parts, head_dim) + 15) & ~size_t(15);
}
inline size_t decode_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                     int n_parts) {
  const int group = n_q_heads / n_kv_heads;
  const size_t groups = static_cast<size_t>(batch) * n_kv_heads * (group / group_tile(group));
  return decode_counters_offset(batch, n_q_heads, n_parts, head_dim) + groups * sizeof(int);
}

int launch_merge(const float *partials, const int32_t *ctx_lens, float *out,
                 int *status, int batch, int n_q_heads, int head_dim,
                 int n_parts, int partition_tokens, cudaStream_t stream);

// Merge of every slot of each row: rows n_rows x n_q_heads, partials
// [row][n_slots][head_dim + 4] (empty slots carry l = 0).
int launch_merge_all(const float *partials, float *out, int *status, int n_rows, int n_q_heads,
                     int head_dim, int n_slots, cudaStream_t stream);


int launch_append(const void *k_new, const void *v_new, void *k_cache,
                  void *v_cache, const int32_t *block_table,
                  const int32_t *seq_idx, const int32_t *pos, int *status,
                  int n_tok, int n_kv_heads, int head_dim, int batch,
                  int max_blocks, int num_pages, cudaStream_t stream);

struct PrefillLaunch {
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_table;
  const int32_t *ctx_lens;
  float *out;
  int *status;
  float scale;
  int n_new, n_q_heads, n_kv_heads, head_dim, batch, max_blocks, num_pages;
  bool bf16;
  // Key-range partitions (n_parts > 1): part_tokens keys each (a multiple of
  // 128); partial states go to workspace, then a merge writes out.
  int n_parts = 1, part_tokens = 0;
  float *workspace = nullptr;
  // Shared keys (cascade decode): shared_ctx >= 0 makes every query attend
  // keys 0 .. shared_ctx - 1 of its sequence's table, no causal mask; with a
  // workspace, ws_slots (0: n_parts) partial-state slots per row, and merge =
  // false leaves the partial states for the caller to fold.
  int shared_ctx = -1, ws_slots = 0;
  bool merge = true;
};

// Workspace of a split prefill: float [B][n_new][Hq][n_parts][D + 4].
inline size_t prefill_partials_bytes(int batch, int n_new, int n_q_heads, int n_parts,
                                     int head_dim) {
  return static_cast<size_t>(batch) * n_new * n_q_heads * n_parts * (head_dim + 4) *
         sizeof(float);
}

// Clears n arrival counters of a split pa_decode after every earlier kernel in
// the stream (one CTA per 256 counters, programmatic dependent launch).
int launch_clear_counters(int *ctr, int n, cudaStream_t stream);

// Merge of prefill rows: row (b, i, h) of q_len = n_new queries saw
// ctx_lens[b] + i + 1 keys.
int launch_merge_rows(const float *partials, const int32_t *ctx_lens, float *out, int *status,
                      int batch, int n_q_heads, int head_dim, int n_parts,
                      int partition_tokens, int n_new, cudaStream_t stream);

int launch_prefill(const PrefillLaunch &a, cudaStream_t stream);

// Device address of the current context's status word (looked up once per
// context), or nullptr if the lookup fails.
int *device_status();

// Tiled tensor map over a [rows][head_dim] 16-bit matrix, box {64, box_rows},
// 128-byte swizzle.  Returns PA_OK or PA_ERR_CUDA.
int make_rows_map(CUtensorMap *map, const void *base, uint64_t rows,
                  int head_dim, int box_rows);


// Launch with programmatic stream serialisation (the kernel must call
// griddep_wait() before it reads anything a predecessor may write).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

}  // namespace pa
