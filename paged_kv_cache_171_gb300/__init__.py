"""paged_kv_cache_171_gb300 -- paged GQA attention for GB300 (sm_103a).

A thin ctypes binding over libpa.so, whose C ABI is include/pa.h.  The
functions named like the C entry points (``pa_decode``, ``pa_append_kv``,
``pa_prefill_paged``, ``pa_merge_partials``, ...) only marshal arguments:
torch tensors become device pointers, the stream becomes a cudaStream_t,
and a nonzero status raises :class:`PAError`.  Every step of the attention
runs in libpa's CUDA kernels; there is no CPU or PyTorch fallback, and using
any of these functions without a built libpa.so raises.

Build the library with ``python -m paged_kv_cache_171_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "PAError", "BF16", "F16", "lib", "dtype_code", "pa_decode", "pa_decode_append",
    "decode_append",
    "pa_decode_partition_tokens", "pa_decode_workspace_size",
    "pa_decode_static_workspace",
    "pa_merge_partials", "pa_append_kv", "pa_prefill_paged",
    "pa_prefill_paged_split", "pa_prefill_partition_tokens", "pa_prefill_workspace_size",
    "pa_decode_window", "pa_decode_window_workspace_size", "decode_window",
    "pa_pool_create", "pa_pool_destroy", "pa_pool_free_pages", "pa_pool_refcount",
    "pa_pool_alloc", "pa_pool_share", "pa_pool_release", "pa_pool_prepare_append",
    "pa_copy_pages", "pa_topm_retain", "pa_topm_workspace_size", "topm_retain",
    "pa_last_device_error", "pa_selftest_wait_timeout", "pa_strerror", "decode", "prefill",
    "prefill_split", "pa_decode_cascade", "pa_decode_cascade_workspace_size",
    "decode_cascade",
    "append_kv",
]

BF16 = 0
F16 = 1

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpa.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "pa.h")

_lib = None


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pa_strerror(status)} ({status})")


def lib():
    """The loaded libpa.so (ctypes.CDLL); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"libpa.so not built ({LIB_PATH}); run "
                "`python -m paged_kv_cache_171_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.pa_strerror.argtypes = [I]
        L.pa_strerror.restype = ctypes.c_char_p
        L.pa_decode.argtypes = [P, P, P, P, P, P, F] + [I] * 8 + [I, P, Z, P]
        L.pa_decode.restype = I
        L.pa_decode_append.argtypes = [P] * 8 + [F] + [I] * 8 + [I, P, Z, P]
        L.pa_decode_append.restype = I
        L.pa_decode_partition_tokens.argtypes = [I] * 7
        L.pa_decode_partition_tokens.restype = I
        L.pa_decode_workspace_size.argtypes = [I] * 7
        L.pa_decode_workspace_size.restype = Z
        L.pa_merge_partials.argtypes = [P, P, P, I, I, I, I, I, P]
        L.pa_merge_partials.restype = I
        L.pa_append_kv.argtypes = [P] * 7 + [I] * 8 + [P]
        L.pa_append_kv.restype = I
        L.pa_prefill_paged.argtypes = [P, P, P, P, P, I, P, F] + [I] * 8 + [P]
        L.pa_prefill_paged.restype = I
        L.pa_prefill_paged_split.argtypes = [P, P, P, P, P, I, P, F] + [I] * 9 + [P, Z, P]
        L.pa_prefill_paged_split.restype = I
        L.pa_prefill_partition_tokens.argtypes = [I] * 8
        L.pa_prefill_partition_tokens.restype = I
        L.pa_prefill_workspace_size.argtypes = [I] * 8
        L.pa_prefill_workspace_size.restype = Z
        L.pa_decode_window.argtypes = [P, P, P, P, P, P, F] + [I] * 11 + [P, Z, P]
        L.pa_decode_window.restype = I
        L.pa_decode_window_workspace_size.argtypes = [I] * 9
        L.pa_decode_window_workspace_size.restype = Z
        L.pa_pool_create.argtypes = [I]
        L.pa_pool_create.restype = P
        L.pa_pool_destroy.argtypes = [P]
        L.pa_pool_destroy.restype = None
        L.pa_pool_free_pages.argtypes = [P]
        L.pa_pool_free_pages.restype = I
        L.pa_pool_refcount.argtypes = [P, I]
        L.pa_pool_refcount.restype = I
        for f in ("pa_pool_alloc", "pa_pool_share", "pa_pool_release"):
            getattr(L, f).argtypes = [P, I, P] if f == "pa_pool_alloc" else [P, P, I]
            getattr(L, f).restype = I
        L.pa_pool_prepare_append.argtypes = [P, P, I, I, I, P, P]
        L.pa_pool_prepare_append.restype = I
        L.pa_copy_pages.argtypes = [P, P, P, P] + [I] * 6 + [P]
        L.pa_copy_pages.restype = I
        L.pa_topm_workspace_size.argtypes = [I, I, I]
        L.pa_topm_workspace_size.restype = Z
        L.pa_topm_retain.argtypes = [P, I, I, I, I, ctypes.c_longlong, P, P, P, Z, P]
        L.pa_topm_retain.restype = I
        L.pa_decode_cascade.argtypes = [P, P, P, P, I, I, P, P, P, F] + [I] * 9 + [P, Z, P]
        L.pa_decode_cascade.restype = I
        L.pa_decode_cascade_workspace_size.argtypes = [I] * 8
        L.pa_decode_cascade_workspace_size.restype = Z
        L.pa_decode_static_workspace.argtypes = [P, P, P, P, P, P, F] + [I] * 9 + [P]
        L.pa_decode_static_workspace.restype = I
        L.pa_last_device_error.argtypes = [P]
        L.pa_last_device_error.restype = I
        L.pa_selftest_wait_timeout.argtypes = [P]
        L.pa_selftest_wait_timeout.restype = I
        _lib = L
    return _lib


def pa_strerror(status: int) -> str:
    try:
        return lib().pa_strerror(int(status)).decode()
    except ImportError:
        return f"status {status}"


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return F16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != 0:
        raise PAError(rc, where)
    return rc


# --- the C entry points, same names and argument order ------------------------

def pa_decode(q, k_cache, v_cache, block_table, ctx_lens, out, scale, n_q_heads,
              n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq,
              num_pages, dtype, partition_tokens=0, workspace=None,
              workspace_bytes=0, stream=None) -> int:
    rc = lib().pa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                         _ptr(ctx_lens), _ptr(out), float(scale), n_q_heads,
                         n_kv_heads, head_dim, page_size, batch,
                         max_blocks_per_seq, num_pages, dtype, partition_tokens,
                         _ptr(workspace), workspace_bytes, _stream(stream))
    return _check(rc, "pa_decode")


def pa_decode_append(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, out, scale,
                     n_q_heads, n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq,
                     num_pages, dtype, partition_tokens=0, workspace=None, workspace_bytes=0,
                     stream=None) -> int:
    rc = lib().pa_decode_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), _ptr(out),
                                float(scale), n_q_heads, n_kv_heads, head_dim, page_size,
                                batch, max_blocks_per_seq, num_pages, dtype, partition_tokens,
                                _ptr(workspace), workspace_bytes, _stream(stream))
    return _check(rc, "pa_decode_append")


def pa_decode_static_workspace(q, k_cache, v_cache, block_table, ctx_lens, out,
                               scale, n_q_heads, n_kv_heads, head_dim, page_size,
                               batch, max_blocks_per_seq, num_pages, dtype,
                               partition_tokens=0, stream=None) -> int:
    """pa_decode with its split-K scratch in the library's fixed 16 MiB
    device array: for callers that cannot allocate device memory."""
    rc = lib().pa_decode_static_workspace(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens),
        _ptr(out), float(scale), n_q_heads, n_kv_heads, head_dim, page_size, batch,
        max_blocks_per_seq, num_pages, dtype, partition_tokens, _stream(stream))
    return _check(rc, "pa_decode_static_workspace")


def pa_decode_partition_tokens(batch, n_q_heads, n_kv_heads, head_dim, page_size,
                               max_blocks_per_seq, partition_tokens=0) -> int:
    rc = lib().pa_decode_partition_tokens(batch, n_q_heads, n_kv_heads, head_dim,
                                          page_size, max_blocks_per_seq,
                                          partition_tokens)
    if rc < 0:
        raise PAError(rc, "pa_decode_partition_tokens")
    return rc


def pa_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, page_size,
                             max_blocks_per_seq, partition_tokens=0) -> int:
    return lib().pa_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
                                          page_size, max_blocks_per_seq,
                                          partition_tokens)


def pa_merge_partials(partials, ctx_lens, out, batch, n_q_heads, head_dim,
                      n_parts, partition_tokens, stream=None) -> int:
    rc = lib().pa_merge_partials(_ptr(partials), _ptr(ctx_lens), _ptr(out), batch,
                                 n_q_heads, head_dim, n_parts, partition_tokens,
                                 _stream(stream))
    return _check(rc, "pa_merge_partials")


def pa_append_kv(k_new, v_new, k_cache, v_cache, block_table, seq_idx, pos, n_tok,
                 n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq,
                 num_pages, dtype, stream=None) -> int:
    rc = lib().pa_append_kv(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                            _ptr(block_table), _ptr(seq_idx), _ptr(pos), n_tok,
                            n_kv_heads, head_dim, page_size, batch,
                            max_blocks_per_seq, num_pages, dtype, _stream(stream))
    return _check(rc, "pa_append_kv")


def pa_prefill_paged(q, k_cache, v_cache, block_table, ctx_lens, n_new, out, scale,
                     n_q_heads, n_kv_heads, head_dim, page_size, batch,
                     max_blocks_per_seq, num_pages, dtype, stream=None) -> int:
    rc = lib().pa_prefill_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_table), _ptr(ctx_lens), n_new, _ptr(out),
                                float(scale), n_q_heads, n_kv_heads, head_dim,
                                page_size, batch, max_blocks_per_seq, num_pages,
                                dtype, _stream(stream))
    return _check(rc, "pa_prefill_paged")


def pa_prefill_paged_split(q, k_cache, v_cache, block_table, ctx_lens, n_new, out,
                           scale, n_q_heads, n_kv_heads, head_dim, page_size, batch,
                           max_blocks_per_seq, num_pages, dtype, partition_tokens=0,
                           workspace=None, workspace_bytes=0, stream=None) -> int:
    rc = lib().pa_prefill_paged_split(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), n_new,
        _ptr(out), float(scale), n_q_heads, n_kv_heads, head_dim, page_size, batch,
        max_blocks_per_seq, num_pages, dtype, partition_tokens, _ptr(workspace),
        workspace_bytes, _stream(stream))
    return _check(rc, "pa_prefill_paged_split")


def pa_prefill_partition_tokens(batch, n_new, n_q_heads, n_kv_heads, head_dim, page_size,
                                max_blocks_per_seq, partition_tokens=0) -> int:
    rc = lib().pa_prefill_partition_tokens(batch, n_new, n_q_heads, n_kv_heads, head_dim,
                                           page_size, max_blocks_per_seq, partition_tokens)
    if rc < 0:
        raise PAError(rc, "pa_prefill_partition_tokens")
    return rc


def pa_prefill_workspace_size(batch, n_new, n_q_heads, n_kv_heads, head_dim, page_size,
                              max_blocks_per_seq, partition_tokens=0) -> int:
    return lib().pa_prefill_workspace_size(batch, n_new, n_q_heads, n_kv_heads, head_dim,
                                           page_size, max_blocks_per_seq, partition_tokens)


def pa_decode_cascade(q, k_cache, v_cache, prefix_table, prefix_len, prefix_blocks,
                      block_table, ctx_lens, out, scale, n_q_heads, n_kv_heads, head_dim,
                      page_size, batch, max_blocks_per_seq, num_pages, dtype, partition_tokens,
                      workspace, workspace_bytes, stream=None):
    rc = lib().pa_decode_cascade(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(prefix_table), prefix_len, prefix_blocks,
        _ptr(block_table), _ptr(ctx_lens), _ptr(out), float(scale), n_q_heads, n_kv_heads,
        head_dim, page_size, batch, max_blocks_per_seq, num_pages, dtype, partition_tokens,
        _ptr(workspace), workspace_bytes, _stream(stream))
    return _check(rc, "pa_decode_cascade")


def pa_decode_cascade_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, page_size,
                                     prefix_blocks, prefix_len, partition_tokens=0) -> int:
    return lib().pa_decode_cascade_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
                                                  page_size, prefix_blocks, prefix_len,
                                                  partition_tokens)


def pa_decode_window(q, k_cache, v_cache, block_table, ctx_lens, out, scale, n_q_heads,
                     n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq, num_pages,
                     dtype, sink_tokens, window_tokens, partition_tokens=0, workspace=None,
                     workspace_bytes=0, stream=None) -> int:
    rc = lib().pa_decode_window(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), _ptr(out),
        float(scale), n_q_heads, n_kv_heads, head_dim, page_size, batch, max_blocks_per_seq,
        num_pages, dtype, sink_tokens, window_tokens, partition_tokens, _ptr(workspace),
        workspace_bytes, _stream(stream))
    return _check(rc, "pa_decode_window")


def pa_decode_window_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, page_size,
                                    max_blocks_per_seq, sink_tokens, window_tokens,
                                    partition_tokens=0) -> int:
    return lib().pa_decode_window_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
                                                 page_size, max_blocks_per_seq, sink_tokens,
                                                 window_tokens, partition_tokens)


def _i32_host(a):
    """A C-contiguous host int32 numpy array (tables and page lists)."""
    import numpy as np
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data


def pa_pool_create(num_pages) -> int:
    """A page pool handle (an opaque pointer as int); raises on failure."""
    h = lib().pa_pool_create(int(num_pages))
    if not h:
        raise PAError(-5, "pa_pool_create")
    return h


def pa_pool_destroy(pool) -> None:
    lib().pa_pool_destroy(pool)


def pa_pool_free_pages(pool) -> int:
    return lib().pa_pool_free_pages(pool)


def pa_pool_refcount(pool, page) -> int:
    rc = lib().pa_pool_refcount(pool, int(page))
    if rc < 0:
        raise PAError(rc, "pa_pool_refcount")
    return rc


def pa_pool_alloc(pool, n):
    """n fresh pages as an int32 numpy array."""
    import numpy as np
    out = np.empty(int(n), dtype=np.int32)
    _check(lib().pa_pool_alloc(pool, int(n), out.ctypes.data if n else None), "pa_pool_alloc")
    return out


def pa_pool_share(pool, pages) -> int:
    a, ptr = _i32_host(pages)
    return _check(lib().pa_pool_share(pool, ptr if a.size else None, a.size), "pa_pool_share")


def pa_pool_release(pool, pages) -> int:
    a, ptr = _i32_host(pages)
    return _check(lib().pa_pool_release(pool, ptr if a.size else None, a.size),
                  "pa_pool_release")


def pa_pool_prepare_append(pool, table_row, page_size, pos):
    """table_row: host int32 numpy array, updated in place.  Returns
    (copy_src, copy_dst): a page pair for pa_copy_pages, or (-1, -1)."""
    import numpy as np
    assert isinstance(table_row, np.ndarray) and table_row.dtype == np.int32 \
        and table_row.flags.c_contiguous
    src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
    rc = lib().pa_pool_prepare_append(pool, table_row.ctypes.data, table_row.size,
                                      int(page_size), int(pos), ctypes.addressof(src),
                                      ctypes.addressof(dst))
    if rc < 0:
        raise PAError(rc, "pa_pool_prepare_append")
    return src.value, dst.value


def pa_copy_pages(k_cache, v_cache, src, dst, n, n_kv_heads, head_dim, page_size, num_pages,
                  dtype, stream=None) -> int:
    rc = lib().pa_copy_pages(_ptr(k_cache), _ptr(v_cache), _ptr(src), _ptr(dst), n,
                             n_kv_heads, head_dim, page_size, num_pages, dtype,
                             _stream(stream))
    return _check(rc, "pa_copy_pages")


def pa_topm_workspace_size(n_layers, n_heads, n_tokens) -> int:
    return lib().pa_topm_workspace_size(n_layers, n_heads, n_tokens)


def pa_topm_retain(scores, n_layers, n_heads, n_tokens, current, budget, keep,
                   kept_per_head=None, workspace=None, workspace_bytes=0, stream=None) -> int:
    rc = lib().pa_topm_retain(_ptr(scores), n_layers, n_heads, n_tokens, current, int(budget),
                              _ptr(keep), _ptr(kept_per_head), _ptr(workspace),
                              workspace_bytes, _stream(stream))
    return _check(rc, "pa_topm_retain")


def pa_last_device_error(stream=None) -> int:
    """Synchronises the stream; returns and clears the device status word."""
    return lib().pa_last_device_error(_stream(stream))


def pa_selftest_wait_timeout(stream=None):
    """One warp waits on a barrier phase nothing completes; the bounded wait
    gives up after 2 s and records PA_ERR_TIMEOUT."""
    return _check(lib().pa_selftest_wait_timeout(_stream(stream)), "pa_selftest_wait_timeout")


# --- tensor-shaped conveniences (allocation by torch, compute by libpa) ------

def decode(q, k_cache, v_cache, block_table, ctx_lens, scale, partition_tokens=0,
           out=None, workspace=None, stream=None):
    """q [B, h_q, D]; caches [pages, h_kv, 16, D]; block_table int32 [B, max_blocks];
    ctx_lens int32 [B].  Returns fp32 [B, h_q, D]."""
    import torch
    B, hq, D = q.shape
    pages, hkv, P, D2 = k_cache.shape
    assert D2 == D and block_table.shape[0] == B
    mb = block_table.shape[1]
    if out is None:
        out = torch.empty((B, hq, D), dtype=torch.float32, device=q.device)
    ws_bytes = pa_decode_workspace_size(B, hq, hkv, D, P, mb, partition_tokens)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=q.device)
    pa_decode(q, k_cache, v_cache, block_table, ctx_lens, out, scale, hq, hkv, D, P,
              B, mb, pages, dtype_code(q), partition_tokens, workspace,
              ws_bytes, stream)
    return out


def decode_append(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, scale,
                  partition_tokens=0, out=None, workspace=None, stream=None):
    """pa_decode_append on tensors: q [B, h_q, D]; k_new, v_new [B, h_kv, D], the
    step's token of each sequence, stored at position ctx_lens[b] - 1 (the
    caches are written in place); ctx_lens counts that token.  Returns fp32
    [B, h_q, D]."""
    import torch
    B, hq, D = q.shape
    pages, hkv, P, D2 = k_cache.shape
    assert D2 == D and block_table.shape[0] == B and tuple(k_new.shape) == (B, hkv, D)
    mb = block_table.shape[1]
    if out is None:
        out = torch.empty((B, hq, D), dtype=torch.float32, device=q.device)
    ws_bytes = pa_decode_workspace_size(B, hq, hkv, D, P, mb, partition_tokens)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=q.device)
    pa_decode_append(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, out, scale, hq,
                     hkv, D, P, B, mb, pages, dtype_code(q), partition_tokens, workspace,
                     ws_bytes, stream)
    return out


def append_kv(k_new, v_new, k_cache, v_cache, block_table, seq_idx, pos, stream=None):
    n_tok, hkv, D = k_new.shape
    pages, _, P, _ = k_cache.shape
    B, mb = block_table.shape
    pa_append_kv(k_new, v_new, k_cache, v_cache, block_table, seq_idx, pos, n_tok,
                 hkv, D, P, B, mb, pages, dtype_code(k_new), stream)


def prefill(q, k_cache, v_cache, block_table, ctx_lens, scale, out=None, stream=None):
    """q [B, n_new, h_q, D]; ctx_lens = cached tokens before the chunk."""
    import torch
    B, n_new, hq, D = q.shape
    pages, hkv, P, _ = k_cache.shape
    mb = block_table.shape[1]
    if out is None:
        out = torch.empty((B, n_new, hq, D), dtype=torch.float32, device=q.device)
    pa_prefill_paged(q, k_cache, v_cache, block_table, ctx_lens, n_new, out, scale,
                     hq, hkv, D, P, B, mb, pages, dtype_code(q), stream)
    return out


def prefill_split(q, k_cache, v_cache, block_table, ctx_lens, scale, partition_tokens=0,
                  out=None, workspace=None, stream=None):
    """pa_prefill_paged_split on tensors: q [B, n_new, h_q, D] (e.g. the gamma
    drafted tokens of a speculative-decoding verify step); ctx_lens = cached
    tokens before the chunk.  Returns fp32 [B, n_new, h_q, D]."""
    import torch
    B, n_new, hq, D = q.shape
    pages, hkv, P, _ = k_cache.shape
    mb = block_table.shape[1]
    if out is None:
        out = torch.empty((B, n_new, hq, D), dtype=torch.float32, device=q.device)
    ws_bytes = pa_prefill_workspace_size(B, n_new, hq, hkv, D, P, mb, partition_tokens)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=q.device)
    pa_prefill_paged_split(q, k_cache, v_cache, block_table, ctx_lens, n_new, out, scale,
                           hq, hkv, D, P, B, mb, pages, dtype_code(q), partition_tokens,
                           workspace, ws_bytes, stream)
    return out


def decode_cascade(q, k_cache, v_cache, prefix_table, prefix_len, block_table, ctx_lens,
                   scale, partition_tokens=0, out=None, workspace=None, stream=None):
    """pa_decode_cascade on tensors: q [B, h_q, D], one query per fork of a
    shared prefix of prefix_len tokens (pages prefix_table, int32 [n]);
    block_table [B, max_blocks] and ctx_lens [B] hold each fork's own tokens
    after the prefix.  Returns fp32 [B, h_q, D]."""
    import torch
    B, hq, D = q.shape
    pages, hkv, P, _ = k_cache.shape
    mb = block_table.shape[1]
    n_pref = prefix_table.shape[0]
    if out is None:
        out = torch.empty((B, hq, D), dtype=torch.float32, device=q.device)
    ws_bytes = pa_decode_cascade_workspace_size(B, hq, hkv, D, P, n_pref, prefix_len,
                                                partition_tokens)
    if workspace is None:
        workspace = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=q.device)
    pa_decode_cascade(q, k_cache, v_cache, prefix_table, prefix_len, n_pref, block_table,
                      ctx_lens, out, scale, hq, hkv, D, P, B, mb, pages, dtype_code(q),
                      partition_tokens, workspace, ws_bytes, stream)
    return out


def decode_window(q, k_cache, v_cache, block_table, ctx_lens, scale, sink_tokens,
                  window_tokens, partition_tokens=0, out=None, workspace=None, stream=None):
    """pa_decode_window on tensors (shapes as decode()): attends keys t < sink_tokens
    and t >= T - window_tokens of each sequence.  Returns fp32 [B, h_q, D]."""
    import torch
    B, hq, D = q.shape
    pages, hkv, P, _ = k_cache.shape
    mb = block_table.shape[1]
    if out is None:
        out = torch.empty((B, hq, D), dtype=torch.float32, device=q.device)
    ws_bytes = pa_decode_window_workspace_size(B, hq, hkv, D, P, mb, sink_tokens,
                                               window_tokens, partition_tokens)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=q.device)
    pa_decode_window(q, k_cache, v_cache, block_table, ctx_lens, out, scale, hq, hkv, D, P,
                     B, mb, pages, dtype_code(q), sink_tokens, window_tokens,
                     partition_tokens, workspace, ws_bytes, stream)
    return out


def topm_retain(scores, current, budget, keep=None, kept_per_head=None, workspace=None,
                stream=None):
    """pa_topm_retain on tensors: scores float32 [L, H, N] on the device.
    Returns (keep uint8 [L, H, N], kept_per_head int32 [L, H])."""
    import torch
    L, H, N = scores.shape
    if keep is None:
        keep = torch.empty((L, H, N), dtype=torch.uint8, device=scores.device)
    if kept_per_head is None:
        kept_per_head = torch.empty((L, H), dtype=torch.int32, device=scores.device)
    ws_bytes = pa_topm_workspace_size(L, H, N)
    if workspace is None:
        workspace = torch.empty(max(1, ws_bytes // 4), dtype=torch.int32, device=scores.device)
    pa_topm_retain(scores, L, H, N, current, budget, keep, kept_per_head, workspace, ws_bytes,
                   stream)
    return keep, kept_per_head
