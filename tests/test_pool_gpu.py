"""Prefix sharing on the GPU: the page copy of copy-on-write, and decode
through block tables that alias the pages of a shared prefix."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_171_gb300 as pa
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_171_gb300 import build
    build.build()


def _rand_caches(pages, hkv, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float16
    k = torch.randn(pages, hkv, 16, D, generator=g).to(dt)
    v = torch.randn(pages, hkv, 16, D, generator=g).to(dt)
    return k, v


@pytest.mark.parametrize("D,hkv,dtype", [(128, 8, "bf16"), (64, 2, "fp16")])
def test_copy_pages_is_bit_exact_and_skips_bad_pairs(D, hkv, dtype):
    k, v = _rand_caches(20, hkv, D, dtype, 61)
    src, dst = [3, 7, 11, 25], [0, 15, 19, 1]  # the last pair is out of range
    want_k, want_v = k.clone(), v.clone()
    want_k[dst[:3]] = k[src[:3]]
    want_v[dst[:3]] = v[src[:3]]
    kd, vd = k.cuda(), v.cuda()
    pa.pa_copy_pages(kd, vd, torch.tensor(src, dtype=torch.int32, device="cuda"),
                     torch.tensor(dst, dtype=torch.int32, device="cuda"), 4, hkv, D, 16, 20,
                     pa.BF16 if dtype == "bf16" else pa.F16)
    assert pa.pa_last_device_error() == -11  # PA_ERR_BAD_BLOCK for the bad pair
    assert torch.equal(kd.cpu(), want_k) and torch.equal(vd.cpu(), want_v)


def test_shared_prefix_copy_on_write_then_decode():
    """Sequences A, B, C share a 1000-token prefix (B and C are forks of A);
    each appends its own token at position 1000, inside the prefix's last,
    shared page: A and B copy it first, C (the last user) writes in place.
    Decode of all three through the aliased tables matches the oracle run on
    the same page copies, appends and tables; the prefix pages stay shared."""
    hq, hkv, D, dtype, T, mb, n_pages = 32, 8, 128, "bf16", 1000, 70, 300
    code = pa.BF16
    k_host, v_host = _rand_caches(n_pages, hkv, D, dtype, 62)
    pool = pa.pa_pool_create(n_pages)
    try:
        a = np.full(mb, -1, dtype=np.int32)
        a[: (T + 15) // 16] = pa.pa_pool_alloc(pool, (T + 15) // 16)
        b, c = a.copy(), a.copy()
        pa.pa_pool_share(pool, b[b >= 0])
        pa.pa_pool_share(pool, c[c >= 0])
        last = T // 16
        assert pa.pa_pool_refcount(pool, a[last]) == 3
        pairs = [pa.pa_pool_prepare_append(pool, t, 16, T) for t in (a, b, c)]
        assert pairs[0][0] == pairs[1][0] == c[last] and pairs[2] == (-1, -1)
        assert len({int(a[last]), int(b[last]), int(c[last])}) == 3
        assert (a[:last] == b[:last]).all() and (a[:last] == c[:last]).all()
        copies = [p for p in pairs if p[0] >= 0]
        tables = np.stack([a, b, c])
    finally:
        pa.pa_pool_destroy(pool)

    k_new, v_new = workloads.new_tokens(3, hkv, D, dtype, seed=63)
    seq_idx = np.arange(3, dtype=np.int32)
    pos = np.full(3, T, dtype=np.int32)
    g = torch.Generator().manual_seed(64)
    q = torch.randn(3, hq, D, generator=g).to(torch.bfloat16)
    ctx = np.full(3, T + 1, dtype=np.int32)
    scale = 1.0 / np.sqrt(D)

    # reference: the page copies (their definition), the oracle's append, decode
    k_ref, v_ref = k_host.clone(), v_host.clone()
    for s, d in copies:
        k_ref[d] = k_ref[s]
        v_ref[d] = v_ref[s]
    k_bits, v_bits = oracle.append_kv(k_new, v_new, k_ref, v_ref, tables, seq_idx, pos)
    ref = oracle.decode(q, k_bits.reshape(k_host.shape), v_bits.reshape(v_host.shape),
                        tables, ctx, scale, code)

    kd, vd = k_host.cuda(), v_host.cuda()
    src = torch.tensor([s for s, _ in copies], dtype=torch.int32, device="cuda")
    dst = torch.tensor([d for _, d in copies], dtype=torch.int32, device="cuda")
    pa.pa_copy_pages(kd, vd, src, dst, len(copies), hkv, D, 16, n_pages, code)
    bt = torch.from_numpy(tables).cuda()
    pa.append_kv(k_new.cuda(), v_new.cuda(), kd, vd, bt, torch.from_numpy(seq_idx).cuda(),
                 torch.from_numpy(pos).cuda())
    out = pa.decode(q.cuda(), kd, vd, bt, torch.from_numpy(ctx).cuda(), scale)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    assert np.array_equal(oracle.bits(kd), k_bits) and np.array_equal(oracle.bits(vd), v_bits)
    from tests.gpu_support import assert_close
    assert_close(out.cpu().numpy(), ref, "decode through shared-prefix tables")
