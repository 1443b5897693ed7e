"""Seeded synthetic inputs for paged GQA attention.

This module only draws numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA library's tests/bench and the float64
oracle can take their inputs from it without sharing any of the method.

Recipe (the pages publish no dataset; their workloads are LLaMA-7B-shaped,
32 layers x 4096 hidden, contexts of 1k-32k tokens, batches of 1-64):
  * Q, K, V elements ~ N(0, 1) drawn in float32 by a seeded torch.Generator,
    then rounded once to the KV dtype (bf16 or fp16); a config may multiply Q
    by a constant before rounding (``q_mul``, "peaky" softmax).
  * The physical page pool is dealt out by a seeded random permutation: the
    first ``sum(pages needed)`` entries of ``randperm(pool_pages)`` go, in
    (layer, sequence, logical block) order, to the block tables.  Unused
    block-table entries are -1 so that a kernel that reads past a sequence's
    last block is caught by its own bounds check.
  * Context lengths are given (an int or a list), or drawn uniformly from an
    inclusive (lo, hi) tuple by the same generator.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}
DTYPE_CODE = {"bf16": 0, "fp16": 1}  # matches pa_dtype in include/pa.h

# The five workloads, by what they are.  ``seed`` values are our choice.
CONFIGS = {
    # MHA decode, 1 layer, batch 1, 16/16 heads, context 512, 32 permuted pages.
    "mha_b1_ctx512": dict(kind="decode", layers=1, batch=1, n_q_heads=16,
                          n_kv_heads=16, head_dim=128, page_size=16, ctx=512,
                          dtype="bf16", pool_pages=32, q_mul=1.0, seed=1001),
    # LLaMA-7B-shaped decode: 32 layers x 32 heads, batch 8, context 4096,
    # fp16 KV, one shuffled pool of 65,536 pages shared by all layers.
    "llama7b_b8_ctx4096": dict(kind="decode", layers=32, batch=8, n_q_heads=32,
                               n_kv_heads=32, head_dim=128, page_size=16,
                               ctx=4096, dtype="fp16", pool_pages=65536,
                               q_mul=1.0, seed=1002),
    # GQA continuous-batching decode: 32/8 heads, 32 layers, batch 64,
    # context ~ U[128, 8192], Q scaled by 2.
    "gqa4_b64_ragged": dict(kind="decode", layers=32, batch=64, n_q_heads=32,
                            n_kv_heads=8, head_dim=128, page_size=16,
                            ctx=(128, 8192), dtype="bf16", pool_pages=None,
                            q_mul=2.0, seed=1003),
    # Long-context split-K decode: 64/8 heads, batch 4, context 32768,
    # 512-token partitions.
    "gqa8_b4_ctx32k": dict(kind="decode", layers=1, batch=4, n_q_heads=64,
                           n_kv_heads=8, head_dim=128, page_size=16, ctx=32768,
                           dtype="bf16", pool_pages=None, q_mul=1.0, seed=1004,
                           partition_tokens=512),
    # Chunked prefill: 32/8 heads, batch 4, 512 new tokens over 8192 cached.
    "prefill_b4_512over8192": dict(kind="prefill", layers=1, batch=4,
                                   n_q_heads=32, n_kv_heads=8, head_dim=128,
                                   page_size=16, ctx=8192, n_new=512,
                                   dtype="bf16", pool_pages=None, q_mul=1.0,
                                   seed=1005),
}


@dataclass
class PagedCase:
    """One layer-stack of paged KV state plus the queries that read it."""
    q: torch.Tensor            # decode [L, B, h_q, D]; prefill [L, B, n_new, h_q, D]
    k_cache: torch.Tensor      # [num_pages, h_kv, P, D]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # int32 [L, B, max_blocks]
    ctx_lens: torch.Tensor     # int32 [B] (prefill: tokens cached before the chunk)
    scale: float
    dtype: str
    n_new: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def layers(self) -> int:
        return self.block_table.shape[0]

    @property
    def dtype_code(self) -> int:
        return DTYPE_CODE[self.dtype]


def _fill_normal(dst: torch.Tensor, gen: torch.Generator, mul: float = 1.0,
                 chunk_elems: int = 1 << 26) -> None:
    """dst (bf16/fp16, contiguous) <- round(N(0,1) * mul), drawn in float32
    chunk by chunk so that temporary memory stays bounded."""
    flat = dst.view(-1)
    n = flat.numel()
    for lo in range(0, n, chunk_elems):
        hi = min(n, lo + chunk_elems)
        tmp = torch.randn(hi - lo, generator=gen, device=dst.device,
                          dtype=torch.float32)
        if mul != 1.0:
            tmp.mul_(mul)
        flat[lo:hi].copy_(tmp)


def draw_ctx_lens(batch: int, ctx, gen: torch.Generator) -> torch.Tensor:
    if isinstance(ctx, tuple):  # (lo, hi): uniform, inclusive
        lo, hi = ctx
        return torch.randint(lo, hi + 1, (batch,), generator=gen,
                             dtype=torch.int64).to(torch.int32)
    if isinstance(ctx, int):
        return torch.full((batch,), ctx, dtype=torch.int32)
    t = torch.as_tensor(ctx, dtype=torch.int32).reshape(-1)
    assert t.numel() == batch
    return t


def paged_case(*, layers: int, batch: int, n_q_heads: int, n_kv_heads: int,
               head_dim: int, page_size: int, ctx, dtype: str, seed: int,
               q_mul: float = 1.0, pool_pages=None, n_new: int = 0,
               max_blocks=None, extra_pool_pages: int = 0, device="cpu",
               kind: str = "decode", **_ignored) -> PagedCase:
    """Build a seeded paged KV cache and queries.

    Decode: each sequence b holds ctx_lens[b] tokens.  Prefill: it holds
    ctx_lens[b] cached tokens plus the chunk's n_new tokens (their K/V rows are
    already in the pages; ctx_lens stays the pre-chunk count).
    """
    device = torch.device(device)
    gen_cpu = torch.Generator(device="cpu").manual_seed(seed)
    ctx_lens = draw_ctx_lens(batch, ctx, gen_cpu)
    held = ctx_lens.to(torch.int64) + (n_new if kind == "prefill" else 0)
    blocks = [int(math.ceil(int(t) / page_size)) for t in held]
    needed = layers * sum(blocks)
    if pool_pages is None:
        pool_pages = needed + extra_pool_pages
    assert pool_pages >= needed, (pool_pages, needed)
    if max_blocks is None:
        max_blocks = max(1, max(blocks))
    perm = torch.randperm(pool_pages, generator=gen_cpu).to(torch.int32)
    bt = torch.full((layers, batch, max_blocks), -1, dtype=torch.int32)
    k = 0
    for layer in range(layers):
        for b in range(batch):
            n = blocks[b]
            bt[layer, b, :n] = perm[k:k + n]
            k += n

    tdt = DTYPES[dtype]
    if device.type == "cuda":
        gen = torch.Generator(device=device).manual_seed(seed)
    else:
        gen = gen_cpu
    shape = (pool_pages, n_kv_heads, page_size, head_dim)
    k_cache = torch.empty(shape, dtype=tdt, device=device)
    v_cache = torch.empty(shape, dtype=tdt, device=device)
    if kind == "prefill":
        q = torch.empty((layers, batch, n_new, n_q_heads, head_dim), dtype=tdt,
                        device=device)
    else:
        q = torch.empty((layers, batch, n_q_heads, head_dim), dtype=tdt,
                        device=device)
    _fill_normal(q, gen, q_mul)
    _fill_normal(k_cache, gen)
    _fill_normal(v_cache, gen)
    return PagedCase(q=q, k_cache=k_cache, v_cache=v_cache,
                     block_table=bt.to(device), ctx_lens=ctx_lens.to(device),
                     scale=1.0 / math.sqrt(head_dim), dtype=dtype, n_new=n_new,
                     meta=dict(seed=seed, pool_pages=pool_pages,
                               max_blocks=max_blocks, needed_pages=needed,
                               q_mul=q_mul, kind=kind))


def config_case(name: str, device="cpu", **overrides) -> PagedCase:
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    return paged_case(device=device, **cfg)


def new_tokens(n_tok: int, n_kv_heads: int, head_dim: int, dtype: str,
               seed: int, device="cpu"):
    """Fresh K and V rows [n_tok, h_kv, D] for an append, N(0,1)."""
    device = torch.device(device)
    gen = (torch.Generator(device=device) if device.type == "cuda"
           else torch.Generator(device="cpu")).manual_seed(seed)
    tdt = DTYPES[dtype]
    k = torch.empty((n_tok, n_kv_heads, head_dim), dtype=tdt, device=device)
    v = torch.empty_like(k)
    _fill_normal(k, gen)
    _fill_normal(v, gen)
    return k, v


def compact_host_copy(case, layer, seqs, extra_tokens=0):
    """Host tensors (q, k, v, table, ctx) holding only sequences `seqs` of
    `layer`, with their pages copied in logical order (table = identity per
    sequence).  extra_tokens counts tokens held beyond ctx_lens (prefill)."""
    ctx = case.ctx_lens.detach().cpu().to(torch.int64)
    bt = case.block_table[layer].detach().cpu()
    ids, rows, pos = [], [], 0
    nb = [int((int(ctx[s]) + extra_tokens + 15) // 16) for s in seqs]
    mb = max(1, max(nb))
    table = torch.full((len(seqs), mb), -1, dtype=torch.int32)
    for i, s in enumerate(seqs):
        pages = bt[s, :nb[i]].to(torch.int64)
        ids.append(pages)
        table[i, :nb[i]] = torch.arange(pos, pos + nb[i], dtype=torch.int32)
        pos += nb[i]
    idx = torch.cat(ids) if ids else torch.zeros(0, dtype=torch.int64)
    idx_dev = idx.to(case.k_cache.device)
    k = case.k_cache.index_select(0, idx_dev).cpu()
    v = case.v_cache.index_select(0, idx_dev).cpu()
    sel = torch.as_tensor(seqs, dtype=torch.int64, device=case.q.device)
    q = case.q[layer].index_select(0, sel).cpu()
    c = ctx[list(seqs)].to(torch.int32)
    return q, k, v, table, c
