"""GPU parity of pa_decode_cascade (the forks of a shared prefix decoded with
the prefix's K/V read once for all of them) against the float64 oracle.

Prefix sharing (ch. 19 "推理系统与性能工程", 19.7.3): fork b's sequence is the
shared prefix followed by its own tokens.  The oracle decodes that
concatenated sequence directly (its K/V rows gathered token by token on the
host through the two tables and laid out as fresh pages), so it shares
neither the cascade's split of the keys nor its merge."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_171_gb300 as pa
import workloads
from tests.gpu_support import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_171_gb300 import build
    build.build()


def _case(B, hq, hkv, D, dtype, prefix_len, own, seed, extra_pages=3):
    """A page pool, a shared prefix table, per-fork tables of their own
    tokens (-1 past each fork's pages) and the forks' queries, all seeded."""
    gen = torch.Generator().manual_seed(seed)
    n_pref = math.ceil(prefix_len / 16)
    own_pages = [math.ceil(t / 16) for t in own]
    mb = max(1, max(own_pages))
    pool = n_pref + sum(own_pages) + extra_pages
    perm = torch.randperm(pool, generator=gen).to(torch.int32)
    prefix_table = perm[:n_pref].clone()
    table = torch.full((B, mb), -1, dtype=torch.int32)
    k = n_pref
    for b, n in enumerate(own_pages):
        table[b, :n] = perm[k:k + n]
        k += n
    tdt = workloads.DTYPES[dtype]
    kc = torch.empty((pool, hkv, 16, D), dtype=tdt)
    vc = torch.empty_like(kc)
    q = torch.empty((B, hq, D), dtype=tdt)
    for t in (q, kc, vc):
        workloads._fill_normal(t, gen)
    return q, kc, vc, prefix_table, table, torch.tensor(own, dtype=torch.int32)


def _oracle(q, kc, vc, prefix_table, prefix_len, table, own, scale, dtype_code):
    """Each fork's concatenated sequence (prefix tokens, then its own) in
    fresh pages with an identity table, decoded by the oracle."""
    B, hkv, D = q.shape[0], kc.shape[1], kc.shape[3]
    lens = [prefix_len + int(t) for t in own]
    nb = [math.ceil(t / 16) for t in lens]
    mbo = max(nb)
    K = torch.zeros((sum(nb), hkv, 16, D), dtype=kc.dtype)
    V = torch.zeros_like(K)
    tab = torch.full((B, mbo), -1, dtype=torch.int32)
    base = 0
    for b in range(B):
        for j in range(lens[b]):
            if j < prefix_len:
                page, slot = int(prefix_table[j // 16]), j % 16
            else:
                u = j - prefix_len
                page, slot = int(table[b, u // 16]), u % 16
            K[base + j // 16, :, j % 16] = kc[page, :, slot]
            V[base + j // 16, :, j % 16] = vc[page, :, slot]
        tab[b, :nb[b]] = torch.arange(base, base + nb[b], dtype=torch.int32)
        base += nb[b]
    return oracle.decode(q, K, V, tab, torch.tensor(lens, dtype=torch.int32), scale,
                         dtype_code)


@pytest.mark.parametrize("B,hq,hkv,D,dtype,prefix_len,own,part", [
    (3, 16, 4, 128, "bf16", 700, [0, 1, 40], 0),          # a fork with nothing of its own
    (5, 8, 8, 64, "fp16", 33, [15, 16, 17, 200, 0], 0),   # MHA, prefix ends mid-page
    (4, 64, 8, 128, "bf16", 2048, [128, 3, 129, 64], 512),
    (2, 32, 8, 128, "bf16", 5000, [1000, 1], 128),        # many prefix ranges
    (40, 32, 4, 64, "bf16", 300, [7 * (i % 6) for i in range(40)], 0),  # two row tiles
    (1, 12, 4, 128, "fp16", 1, [31], 0),                  # a one-token prefix
])
def test_cascade_matches_oracle(B, hq, hkv, D, dtype, prefix_len, own, part):
    q, kc, vc, ptab, tab, ctx = _case(B, hq, hkv, D, dtype, prefix_len, own, seed=61 + B)
    scale = 1.0 / math.sqrt(D)
    ref = _oracle(q, kc, vc, ptab, prefix_len, tab, own, scale, workloads.DTYPE_CODE[dtype])
    out = pa.decode_cascade(q.cuda(), kc.cuda(), vc.cuda(), ptab.cuda(), prefix_len,
                            tab.cuda(), ctx.cuda(), scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"cascade B={B} {hq}/{hkv} D={D} prefix {prefix_len}")
    assert pa.pa_last_device_error() == 0


def test_cascade_equals_decode_on_the_aliased_tables():
    """The prefix-sharing workload (32 forks of an 8192-token prefix, 128 own
    tokens each, 32/8 heads): cascade and pa_decode over the forks' full
    tables (prefix pages aliased in every one) agree, whatever the
    workspace held before (NaN)."""
    B, hq, hkv, D, prefix_len, own_len = 32, 32, 8, 128, 8192, 128
    q, kc, vc, ptab, tab, ctx = _case(B, hq, hkv, D, "bf16", prefix_len, [own_len] * B,
                                      seed=1008)
    full = torch.cat([ptab.unsqueeze(0).expand(B, -1), tab], dim=1).contiguous()
    dev = [t.cuda() for t in (q, kc, vc, ptab, tab, ctx, full)]
    q_d, kc_d, vc_d, ptab_d, tab_d, ctx_d, full_d = dev
    scale = 1.0 / math.sqrt(D)
    a = pa.decode(q_d, kc_d, vc_d, full_d, ctx_d + prefix_len, scale)
    ws_bytes = pa.pa_decode_cascade_workspace_size(B, hq, hkv, D, 16, ptab.shape[0],
                                                   prefix_len, 0)
    ws = torch.full((ws_bytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    b = pa.decode_cascade(q_d, kc_d, vc_d, ptab_d, prefix_len, tab_d, ctx_d, scale,
                          workspace=ws)
    torch.cuda.synchronize()
    assert_close(b.cpu().numpy(), a.cpu().numpy().astype(np.float64), "cascade vs decode")
    # and two forks against the oracle
    sel = [0, 31]
    ref = _oracle(q[sel], kc, vc, ptab, prefix_len, tab[sel], [own_len] * 2, scale,
                  workloads.DTYPE_CODE["bf16"])
    assert_close(b[sel].cpu().numpy(), ref, "cascade vs oracle")
    assert pa.pa_last_device_error() == 0
