"""Test-side helpers: scatter a contiguous per-sequence K/V into a paged pool.

The tests decide a contiguous K/V first (the ground truth a library routine
such as torch's scaled_dot_product_attention can read), then lay it out in
pages through a random block table.  Nothing here computes attention.
"""
from __future__ import annotations

import torch


def scatter_to_pages(kc: torch.Tensor, vc: torch.Tensor, lens, page_size: int,
                     gen: torch.Generator, extra_pages: int = 3,
                     max_blocks=None):
    """kc, vc: [B, h_kv, T_max, D] (any float dtype).  Sequence b keeps its
    first lens[b] tokens.  Returns (k_cache, v_cache, block_table) with the
    pool [num_pages, h_kv, P, D] filled with a junk value outside the used
    slots (so a kernel that reads a slot it should mask shows up)."""
    B, H, _, D = kc.shape
    blocks = [-(-int(t) // page_size) for t in lens]
    need = sum(blocks)
    num_pages = need + extra_pages
    perm = torch.randperm(num_pages, generator=gen)
    if max_blocks is None:
        max_blocks = max(1, max(blocks))
    bt = torch.full((B, max_blocks), -1, dtype=torch.int32)
    k_cache = torch.full((num_pages, H, page_size, D), 7.0, dtype=kc.dtype)
    v_cache = torch.full((num_pages, H, page_size, D), -7.0, dtype=vc.dtype)
    i = 0
    for b in range(B):
        for blk in range(blocks[b]):
            page = int(perm[i])
            i += 1
            bt[b, blk] = page
            lo = blk * page_size
            n = min(page_size, int(lens[b]) - lo)
            k_cache[page, :, :n] = kc[b, :, lo:lo + n]
            v_cache[page, :, :n] = vc[b, :, lo:lo + n]
    return k_cache, v_cache, bt


def sdpa_reference(q, kc, vc, lens, scale):
    """Library route: torch SDPA in float64 per sequence, GQA by enable_gqa.

    q [B, h_q, D]; kc/vc [B, h_kv, T_max, D]. Returns float64 [B, h_q, D]."""
    import torch.nn.functional as F
    outs = []
    for b in range(q.shape[0]):
        T = int(lens[b])
        qb = q[b].double().unsqueeze(0).unsqueeze(2)        # [1, h_q, 1, D]
        kb = kc[b, :, :T].double().unsqueeze(0)             # [1, h_kv, T, D]
        vb = vc[b, :, :T].double().unsqueeze(0)
        if T == 0:
            outs.append(torch.zeros(q.shape[1], q.shape[2], dtype=torch.float64))
            continue
        o = F.scaled_dot_product_attention(qb, kb, vb, scale=scale,
                                           enable_gqa=True)
        outs.append(o[0, :, 0])
    return torch.stack(outs)
