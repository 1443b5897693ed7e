// pa_pool.cu -- reference-counted page pool (host) and the page copy of
// copy-on-write (device).
//
// Prefix sharing ("推理系统与性能工程" 19.7.3, PagedAttention: the block tables
// of several requests may point to the same physical block, which is then
// reference-counted and copied before a write): the pool hands out physical
// pages of the K/V caches, counts the block-table entries that point to each,
// and, when a sequence is about to write into a page other tables also
// reference, maps a fresh page for it and reports the copy to make.  The
// attention kernels need nothing new: they read through the block tables, so
// aliased entries are transparent to them.
#include <mutex>
#include <vector>

#include "pa_device.cuh"
#include "pa_internal.h"

struct pa_pool {
  std::mutex mu;               // the pool may be shared between host threads
  std::vector<int32_t> refs;   // block-table entries pointing at each page
  std::vector<int32_t> free_;  // pages with refs == 0 (a stack: last freed, first reused)
};

namespace pa {
namespace {

// Copy whole pages src[i] -> dst[i] of both caches, every kv head: one CTA per
// (pair, tensor), 16-byte vectors.
__global__ void __launch_bounds__(256)
    copy_pages_kernel(uint4 *k_cache, uint4 *v_cache, const int32_t *src, const int32_t *dst,
                      int n, int num_pages, size_t page_vecs, int *status) {
  griddep_wait();
  const int i = blockIdx.x >> 1;
  uint4 *cache = (blockIdx.x & 1) ? v_cache : k_cache;
  const int s = src[i], d = dst[i];
  if (static_cast<unsigned>(s) >= static_cast<unsigned>(num_pages) ||
      static_cast<unsigned>(d) >= static_cast<unsigned>(num_pages)) {
    if (threadIdx.x == 0) record_error(status, PA_ERR_BAD_BLOCK);
    return;
  }
  const uint4 *from = cache + static_cast<size_t>(s) * page_vecs;
  uint4 *to = cache + static_cast<size_t>(d) * page_vecs;
  for (size_t e = threadIdx.x; e < page_vecs; e += blockDim.x) to[e] = from[e];
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

pa_pool *pa_pool_create(int num_pages) {
  if (num_pages <= 0) return nullptr;
  pa_pool *p = new (std::nothrow) pa_pool;
  if (!p) return nullptr;
  p->refs.assign(num_pages, 0);
  p->free_.reserve(num_pages);
  for (int i = num_pages - 1; i >= 0; --i) p->free_.push_back(i);  // page 0 first
  return p;
}

void pa_pool_destroy(pa_pool *pool) { delete pool; }

int pa_pool_free_pages(pa_pool *pool) {
  if (!pool) return PA_ERR_NULL;
  std::lock_guard<std::mutex> g(pool->mu);
  return static_cast<int>(pool->free_.size());
}

int pa_pool_refcount(pa_pool *pool, int page) {
  if (!pool) return PA_ERR_NULL;
  std::lock_guard<std::mutex> g(pool->mu);
  if (page < 0 || page >= static_cast<int>(pool->refs.size())) return PA_ERR_SHAPE;
  return pool->refs[page];
}

int pa_pool_alloc(pa_pool *pool, int n, int32_t *pages) {
  if (!pool || (n > 0 && !pages)) return PA_ERR_NULL;
  if (n < 0) return PA_ERR_SHAPE;
  std::lock_guard<std::mutex> g(pool->mu);
  if (static_cast<size_t>(n) > pool->free_.size()) return PA_ERR_POOL_EMPTY;
  for (int i = 0; i < n; ++i) {
    const int32_t page = pool->free_.back();
    pool->free_.pop_back();
    pool->refs[page] = 1;
    pages[i] = page;
  }
  return PA_OK;
}

int pa_pool_share(pa_pool *pool, const int32_t *pages, int n) {
  if (!pool || (n > 0 && !pages)) return PA_ERR_NULL;
  if (n < 0) return PA_ERR_SHAPE;
  std::lock_guard<std::mutex> g(pool->mu);
  const int np = static_cast<int>(pool->refs.size());
  for (int i = 0; i < n; ++i)  // validate first: all or nothing
    if (pages[i] >= np || (pages[i] >= 0 && pool->refs[pages[i]] == 0))
      return PA_ERR_POOL_STATE;
  for (int i = 0; i < n; ++i)
    if (pages[i] >= 0) ++pool->refs[pages[i]];
  return PA_OK;
}

int pa_pool_release(pa_pool *pool, const int32_t *pages, int n) {
  if (!pool || (n > 0 && !pages)) return PA_ERR_NULL;
  if (n < 0) return PA_ERR_SHAPE;
  std::lock_guard<std::mutex> g(pool->mu);
  const int np = static_cast<int>(pool->refs.size());
  // validate first (a page listed k times needs k references): all or nothing
  std::vector<int32_t> want;
  for (int i = 0; i < n; ++i) {
    if (pages[i] < 0) continue;
    if (pages[i] >= np) return PA_ERR_POOL_STATE;
    want.push_back(pages[i]);
  }
  for (size_t i = 0; i < want.size(); ++i) {
    int c = 0;
    for (size_t j = 0; j <= i; ++j) c += want[j] == want[i];
    if (c > pool->refs[want[i]]) return PA_ERR_POOL_STATE;
  }
  for (int32_t page : want)
    if (--pool->refs[page] == 0) pool->free_.push_back(page);
  return PA_OK;
}

int pa_pool_prepare_append(pa_pool *pool, int32_t *table, int max_blocks, int page_size,
                           int pos, int32_t *copy_src, int32_t *copy_dst) {
  if (!pool || !table || !copy_src || !copy_dst) return PA_ERR_NULL;
  if (page_size != kPageSize) return PA_ERR_PAGE_SIZE;
  if (pos < 0 || max_blocks <= 0 || pos / page_size >= max_blocks) return PA_ERR_SHAPE;
  std::lock_guard<std::mutex> g(pool->mu);
  const int np = static_cast<int>(pool->refs.size());
  int32_t &slot = table[pos / page_size];
  *copy_src = *copy_dst = -1;
  if (slot < 0) {  // the block is not mapped yet: a fresh page
    if (pool->free_.empty()) return PA_ERR_POOL_EMPTY;
    slot = pool->free_.back();
    pool->free_.pop_back();
    pool->refs[slot] = 1;
    return 0;
  }
  if (slot >= np || pool->refs[slot] == 0) return PA_ERR_POOL_STATE;
  if (pool->refs[slot] == 1) return 0;  // this table is the only user: write in place
  // shared: copy on write
  if (pool->free_.empty()) return PA_ERR_POOL_EMPTY;
  const int32_t fresh = pool->free_.back();
  pool->free_.pop_back();
  pool->refs[fresh] = 1;
  --pool->refs[slot];
  *copy_src = slot;
  *copy_dst = fresh;
  slot = fresh;
  return 1;
}

int pa_copy_pages(void *k_cache, void *v_cache, const int32_t *src, const int32_t *dst,
                  int n, int n_kv_heads, int head_dim, int page_size, int num_pages,
                  pa_dtype dtype, pa_stream_t stream) {
  if (!k_cache || !v_cache || (n > 0 && (!src || !dst))) return PA_ERR_NULL;
  if (n_kv_heads <= 0) return PA_ERR_HEADS;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_HEAD_DIM;
  if (page_size != kPageSize) return PA_ERR_PAGE_SIZE;
  if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_DTYPE;
  if (n < 0 || n > (1 << 29) || num_pages <= 0) return PA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return PA_ERR_ALIGN;
  if (n == 0) return PA_OK;
  int *status = device_status();
  if (!status) return PA_ERR_CUDA;
  const size_t page_vecs = static_cast<size_t>(n_kv_heads) * page_size * head_dim * 2 / 16;
  if (launch_pdl(copy_pages_kernel, dim3(2 * n), dim3(256), 0,
                 reinterpret_cast<cudaStream_t>(stream), static_cast<uint4 *>(k_cache),
                 static_cast<uint4 *>(v_cache), src, dst, n, num_pages, page_vecs,
                 status) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // extern "C"
