"""Shared pieces of the GPU parity tests: tolerance, moving seeded cases to the
device, and cutting a compact host copy of a few sequences of a large device
case for the oracle (re-indexing pages only; no attention arithmetic)."""
from __future__ import annotations

import numpy as np
import torch

# The stated bar: |gpu - ref| <= 2e-3 + 1e-2 |ref| element-wise, fp32 outputs
# from bf16/fp16 inputs against the float64 oracle.
ATOL = 2e-3
RTOL = 1e-2


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (ATOL + RTOL * np.abs(ref))), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst at {i}: "
            f"got {got[i]!r} ref {ref[i]!r}; max abs err {err.max():.3e}")
    return float(err.max())


def to_device(case, device):
    case.q = case.q.to(device)
    case.k_cache = case.k_cache.to(device)
    case.v_cache = case.v_cache.to(device)
    case.block_table = case.block_table.to(device)
    case.ctx_lens = case.ctx_lens.to(device)
    return case


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
