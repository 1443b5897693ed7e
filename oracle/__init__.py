"""Float64 CPU oracle for paged GQA attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import this package.  The product path
(``paged_kv_cache_171_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``pa_oracle.c`` (compiled by ``oracle/build.py``);
this module only marshals numpy arrays into it.  16-bit inputs are passed as
their bit patterns (``uint16``); outputs are float64.

Functions and the passages they follow (page title, section):
  decode          -- ch. 19 "推理系统与性能工程" 19.4.1 (softmax(Q K^T/sqrt d) V),
                     19.6.2 (stable softmax), 19.7.3 (block table);
                     "吞吐与延迟的系统模型" 4-5 (GQA shares KV heads).
  decode_online   -- 19.6.2, the three-step online-softmax recurrence.
  decode_window   -- decode over the attention-sink + sliding-window key set
                     (ch. 19, KV-cache eviction: the first tokens and the most
                     recent window are kept).
  partials/merge  -- 19.6.2's exponent law applied to chunk summaries.
  append_kv       -- "吞吐与延迟的系统模型" 4 (one new K and V row per step).
  prefill         -- 19.3.1 / 19.6.3, causal attention of a chunk of new
                     queries over the cache.
  kv_bytes_*      -- appendix "推理基础" eq. 3 and ch. 19 19.4.2.
  topm_retain     -- ch. 19 19.4.3 (KV-cache compression, budgeted eviction):
                     the current position of every (layer, head) is kept, the
                     other (l, h, t) compete globally by the key
                     (-score, l, h, t) for the remaining budget.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

BF16 = 0
F16 = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        Dd = ctypes.c_double
        lib.oracle_decode.argtypes = [P, P, P, P, P, P, Dd] + [I] * 9
        lib.oracle_decode_online.argtypes = [P, P, P, P, P, P, Dd] + [I] * 8 + [P, I]
        lib.oracle_decode_window.argtypes = [P, P, P, P, P, P, Dd] + [I] * 11
        lib.oracle_partials.argtypes = [P, P, P, P, P, P, Dd] + [I] * 11
        lib.oracle_merge.argtypes = [P, P, I, I, I]
        lib.oracle_append_kv.argtypes = [P, P, P, P, P, P, P] + [I] * 7
        lib.oracle_prefill.argtypes = [P, P, P, P, P, I, P, Dd] + [I] * 9
        lib.oracle_decode_half.argtypes = [ctypes.c_uint16, I]
        lib.oracle_decode_half.restype = Dd
        lib.oracle_max_threads.restype = I
        for f in ("oracle_decode", "oracle_decode_online", "oracle_partials",
                  "oracle_merge", "oracle_append_kv", "oracle_prefill",
                  "oracle_decode_window"):
            getattr(lib, f).restype = I
        _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle's OpenMP loops use by default."""
    return _load().oracle_max_threads()


def bits(x) -> np.ndarray:
    """16-bit float tensor/array -> contiguous uint16 bit patterns (no rounding)."""
    if hasattr(x, "detach"):  # a torch tensor; view its bytes, never convert values
        import torch
        assert x.element_size() == 2
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(x)
    assert a.dtype.itemsize == 2, a.dtype
    return a.view(np.uint16)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def decode_half(h: int, dtype: int) -> float:
    return _load().oracle_decode_half(int(h) & 0xFFFF, dtype)


def _geom(k_cache: np.ndarray):
    num_pages, n_kv_heads, page_size, head_dim = k_cache.shape
    return num_pages, n_kv_heads, page_size, head_dim


def decode(q, k_cache, v_cache, block_table, ctx_lens, scale, dtype,
           n_threads: int = 0) -> np.ndarray:
    """Decode attention by its plain definition.

    q [batch, n_q_heads, head_dim]; k_cache/v_cache
    [num_pages, n_kv_heads, page_size, head_dim]; block_table int32
    [batch, max_blocks]; ctx_lens int32 [batch].  Returns float64
    [batch, n_q_heads, head_dim].
    """
    q, kc, vc = bits(q), bits(k_cache), bits(v_cache)
    bt, cl = _i32(block_table), _i32(ctx_lens)
    batch, n_q_heads, head_dim = q.shape
    num_pages, n_kv_heads, page_size, hd = _geom(kc)
    assert hd == head_dim and vc.shape == kc.shape and bt.shape[0] == batch
    out = np.zeros((batch, n_q_heads, head_dim), dtype=np.float64)
    rc = _load().oracle_decode(_p(q), _p(kc), _p(vc), _p(bt), _p(cl), _p(out),
                               float(scale), n_q_heads, n_kv_heads, head_dim,
                               page_size, batch, bt.shape[1], num_pages, dtype,
                               n_threads)
    if rc:
        raise ValueError("oracle_decode: index out of range")
    return out


def decode_window(q, k_cache, v_cache, block_table, ctx_lens, scale, dtype, sink,
                  window, n_threads: int = 0) -> np.ndarray:
    """Decode attention over the attention-sink + sliding-window key set:
    key t of a T-token sequence is kept iff t < sink or t >= T - window."""
    q, kc, vc = bits(q), bits(k_cache), bits(v_cache)
    bt, cl = _i32(block_table), _i32(ctx_lens)
    batch, n_q_heads, head_dim = q.shape
    num_pages, n_kv_heads, page_size, hd = _geom(kc)
    assert hd == head_dim and vc.shape == kc.shape and bt.shape[0] == batch
    out = np.zeros((batch, n_q_heads, head_dim), dtype=np.float64)
    rc = _load().oracle_decode_window(_p(q), _p(kc), _p(vc), _p(bt), _p(cl), _p(out),
                                      float(scale), n_q_heads, n_kv_heads, head_dim,
                                      page_size, batch, bt.shape[1], num_pages, dtype,
                                      int(sink), int(window), n_threads)
    if rc:
        raise ValueError("oracle_decode_window: index out of range")
    return out


def decode_online(q, k_cache, v_cache, block_table, ctx_lens, scale, dtype,
                  cuts) -> np.ndarray:
    """Decode attention through the online-softmax recurrence, blocks cut at
    the ascending token positions ``cuts``."""
    q, kc, vc = bits(q), bits(k_cache), bits(v_cache)
    bt, cl = _i32(block_table), _i32(ctx_lens)
    cu = _i32(np.asarray(cuts, dtype=np.int32).reshape(-1))
    batch, n_q_heads, head_dim = q.shape
    num_pages, n_kv_heads, page_size, _ = _geom(kc)
    out = np.zeros((batch, n_q_heads, head_dim), dtype=np.float64)
    rc = _load().oracle_decode_online(
        _p(q), _p(kc), _p(vc), _p(bt), _p(cl), _p(out), float(scale),
        n_q_heads, n_kv_heads, head_dim, page_size, batch, bt.shape[1],
        num_pages, dtype, _p(cu) if cu.size else None, int(cu.size))
    if rc:
        raise ValueError("oracle_decode_online: index out of range")
    return out


def partials(q, k_cache, v_cache, block_table, ctx_lens, scale, dtype,
             part_tokens: int, n_parts: int, n_threads: int = 0) -> np.ndarray:
    """Per-chunk partial states: float64 [batch, n_q_heads, n_parts, head_dim+2]
    holding (O_p..., m_p, l_p)."""
    q, kc, vc = bits(q), bits(k_cache), bits(v_cache)
    bt, cl = _i32(block_table), _i32(ctx_lens)
    batch, n_q_heads, head_dim = q.shape
    num_pages, n_kv_heads, page_size, _ = _geom(kc)
    out = np.zeros((batch, n_q_heads, n_parts, head_dim + 2), dtype=np.float64)
    rc = _load().oracle_partials(
        _p(q), _p(kc), _p(vc), _p(bt), _p(cl), _p(out), float(scale),
        n_q_heads, n_kv_heads, head_dim, page_size, batch, bt.shape[1],
        num_pages, dtype, int(part_tokens), int(n_parts), n_threads)
    if rc:
        raise ValueError("oracle_partials: index out of range")
    return out


def merge(parts: np.ndarray) -> np.ndarray:
    """Exact merge of partial states [..., n_parts, head_dim + 2] -> [..., head_dim]."""
    parts = np.ascontiguousarray(parts, dtype=np.float64)
    n_parts, w = parts.shape[-2], parts.shape[-1]
    lead = parts.shape[:-2]
    n_rows = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (w - 2,), dtype=np.float64)
    _load().oracle_merge(_p(parts), _p(out), n_rows, n_parts, w - 2)
    return out


def append_kv(k_new, v_new, k_cache, v_cache, block_table, seq_idx, pos):
    """Returns new (k_cache, v_cache) uint16 arrays with the rows scattered in."""
    kn, vn = bits(k_new), bits(v_new)
    kc, vc = bits(k_cache).copy(), bits(v_cache).copy()
    bt, si, ps = _i32(block_table), _i32(seq_idx), _i32(pos)
    n_tok, n_kv_heads, head_dim = kn.shape
    num_pages, _, page_size, _ = _geom(kc)
    rc = _load().oracle_append_kv(_p(kn), _p(vn), _p(kc), _p(vc), _p(bt),
                                  _p(si), _p(ps), n_tok, n_kv_heads, head_dim,
                                  page_size, bt.shape[0], bt.shape[1], num_pages)
    if rc:
        raise ValueError("oracle_append_kv: index out of range")
    return kc, vc


def prefill(q, k_cache, v_cache, block_table, ctx_lens, scale, dtype,
            n_threads: int = 0) -> np.ndarray:
    """Causal chunked prefill: q [batch, n_new, n_q_heads, head_dim]; ctx_lens
    counts cached tokens before the chunk.  Returns float64 like q."""
    q, kc, vc = bits(q), bits(k_cache), bits(v_cache)
    bt, cl = _i32(block_table), _i32(ctx_lens)
    batch, n_new, n_q_heads, head_dim = q.shape
    num_pages, n_kv_heads, page_size, _ = _geom(kc)
    out = np.zeros(q.shape, dtype=np.float64)
    rc = _load().oracle_prefill(_p(q), _p(kc), _p(vc), _p(bt), _p(cl), n_new,
                                _p(out), float(scale), n_q_heads, n_kv_heads,
                                head_dim, page_size, batch, bt.shape[1],
                                num_pages, dtype, n_threads)
    if rc:
        raise ValueError("oracle_prefill: index out of range")
    return out


# --- KV-cache size arithmetic ------------------------------------------------

def kv_bytes_eq3(n_layers: int, d_model: int, seq_len: int, batch: int,
                 elem_bytes: int) -> int:
    """Appendix "推理基础", eq. 3: M_KV = 2 * N_L * d * S * B * s_elem."""
    return 2 * n_layers * d_model * seq_len * batch * elem_bytes


def kv_bytes_per_token(n_layers: int, hidden: int, elem_bytes: int) -> int:
    """Ch. 19, 19.4.2: per layer every head caches one K and one V vector of
    d_h = h/H elements; H heads give 2h elements, L layers 2*L*h, times the
    element size."""
    per_head = 2  # one K vector and one V vector per head, each hidden/H long
    return per_head * hidden * n_layers * elem_bytes


def topm_retain(scores, current, budget) -> np.ndarray:
    """Budgeted global KV retention (ch. 19 19.4.3).

    scores float [L, H, N] (attention mass per layer, head and token);
    current = C, the generation position; budget = M.  Position C of every
    (layer, head) is kept unconditionally (L*H slots).  Every other
    (l, h, t) is a candidate; the candidates are ordered by the key
    (-score, l, h, t) ascending -- score descending, ties by layer, then head,
    then token -- and the first M - L*H are kept (none when M <= L*H, all when
    the budget exceeds them).  -0.0 ranks as 0.0; a NaN score ranks after
    every number.  Returns bool [L, H, N].
    """
    s = np.asarray(scores, dtype=np.float32)
    L, H, N = s.shape
    keep = np.zeros((L, H, N), dtype=bool)
    keep[:, :, current] = True
    rest = int(budget) - L * H
    if rest <= 0:
        return keep
    l_idx, h_idx, t_idx = np.meshgrid(np.arange(L), np.arange(H), np.arange(N),
                                      indexing="ij")
    cand = t_idx.reshape(-1) != current
    neg = -s.reshape(-1).astype(np.float64)[cand]    # -0.0 and 0.0 compare equal
    nan_last = np.isnan(neg).astype(np.int8)          # primary key: NaN after every number
    neg = np.where(np.isnan(neg), 0.0, neg)
    li, hi, ti = l_idx.reshape(-1)[cand], h_idx.reshape(-1)[cand], t_idx.reshape(-1)[cand]
    order = np.lexsort((ti, hi, li, neg, nan_last))  # last key is the primary one
    chosen = order[:rest]
    keep[li[chosen], hi[chosen], ti[chosen]] = True
    return keep
