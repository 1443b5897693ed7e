"""Seeded random configurations of every entry point against the oracle:
shapes, group sizes, head dims, dtypes, context mixes (empty, one token,
page and tile edges, long) and partition sizes drawn at random, sized so the
oracle finishes in seconds.  Complements the hand-picked cases: it reaches
combinations of the kernels' modes (single pass / key ranges / warp-owned
partitions; interleaved and split-row prefill tiles; sink + window spans)
that nobody listed."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_171_gb300 as pa
import workloads
from tests.gpu_support import assert_close, to_device

pytestmark = pytest.mark.gpu

HEADS = [(8, 8), (16, 4), (32, 8), (24, 8), (64, 8), (12, 4), (16, 2), (6, 3)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_171_gb300 import build
    build.build()


def _ctx(rng, n, hi):
    edges = [0, 1, 15, 16, 17, 127, 128, 129, 511, 512, 513]
    return [int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(0, hi))
            for _ in range(n)]


def _case(rng, kind, n_new=0, hi=2500):
    hq, hkv = HEADS[rng.integers(len(HEADS))]
    kw = dict(layers=1, batch=int(rng.integers(1, 5)), n_q_heads=hq, n_kv_heads=hkv,
              head_dim=int(rng.choice([64, 128])), page_size=16,
              dtype=str(rng.choice(["bf16", "fp16"])), seed=int(rng.integers(1 << 30)),
              extra_pool_pages=3)
    kw["ctx"] = _ctx(rng, kw["batch"], hi)
    if kind == "prefill":
        kw.update(n_new=n_new, kind="prefill")
    return kw


@pytest.mark.parametrize("seed", range(12))
def test_random_decode(seed):
    rng = np.random.default_rng(7000 + seed)
    kw = _case(rng, "decode")
    cpu = workloads.paged_case(**kw)
    ref = oracle.decode(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0], cpu.ctx_lens,
                        cpu.scale, cpu.dtype_code)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    part = int(rng.choice([0, 16, 32, 64, 256, 512]))
    out = pa.decode(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0], dev.ctx_lens,
                    dev.scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"decode {kw} part {part}")
    assert pa.pa_last_device_error() == 0


@pytest.mark.parametrize("seed", range(12))
def test_random_decode_append(seed):
    """pa_decode_append: each non-empty sequence's step token written at
    position ctx - 1 (caches bit-exact), the decode over ctx tokens."""
    rng = np.random.default_rng(7500 + seed)
    kw = _case(rng, "decode")
    cpu = workloads.paged_case(**kw)
    B, hkv, D = len(kw["ctx"]), kw["n_kv_heads"], kw["head_dim"]
    k_new, v_new = workloads.new_tokens(B, hkv, D, kw["dtype"], seed=int(rng.integers(1 << 30)))
    seqs = [b for b in range(B) if kw["ctx"][b] > 0]
    k_ref, v_ref = oracle.append_kv(k_new[seqs], v_new[seqs], cpu.k_cache, cpu.v_cache,
                                    cpu.block_table[0], np.array(seqs, np.int32),
                                    np.array([kw["ctx"][b] - 1 for b in seqs], np.int32))
    ref = oracle.decode(cpu.q[0], k_ref.reshape(cpu.k_cache.shape),
                        v_ref.reshape(cpu.v_cache.shape), cpu.block_table[0], cpu.ctx_lens,
                        cpu.scale, cpu.dtype_code)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    part = int(rng.choice([0, 16, 32, 64, 256, 512]))
    out = pa.decode_append(dev.q[0], k_new.cuda(), v_new.cuda(), dev.k_cache, dev.v_cache,
                           dev.block_table[0], dev.ctx_lens, dev.scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    assert np.array_equal(oracle.bits(dev.k_cache), k_ref)
    assert np.array_equal(oracle.bits(dev.v_cache), v_ref)
    assert_close(out.cpu().numpy(), ref, f"decode_append {kw} part {part}")


@pytest.mark.parametrize("seed", range(12))
def test_random_prefill_and_split(seed):
    rng = np.random.default_rng(8000 + seed)
    n_new = int(rng.choice([1, 2, 3, 4, 8, int(rng.integers(1, 200))]))
    kw = _case(rng, "prefill", n_new=n_new, hi=1500)
    cpu = workloads.paged_case(**kw)
    ref = oracle.prefill(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0],
                         cpu.ctx_lens, cpu.scale, cpu.dtype_code)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    out = pa.prefill(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0], dev.ctx_lens,
                     dev.scale)
    part = int(rng.choice([0, 128, 256, 512]))
    out_s = pa.prefill_split(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                             dev.ctx_lens, dev.scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"prefill {kw}")
    assert_close(out_s.cpu().numpy(), ref, f"split prefill {kw} part {part}")
    assert pa.pa_last_device_error() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_window(seed):
    rng = np.random.default_rng(9000 + seed)
    kw = _case(rng, "decode")
    sink, window = int(rng.integers(0, 40)), int(rng.choice([0, 1, 16, 100, 500, 2000]))
    cpu = workloads.paged_case(**kw)
    ref = oracle.decode_window(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0],
                               cpu.ctx_lens, cpu.scale, cpu.dtype_code, sink, window)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    part = int(rng.choice([0, 16, 64, 256]))
    out = pa.decode_window(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                           dev.ctx_lens, dev.scale, sink, window, partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"window {kw} sink {sink} window {window} part {part}")
    assert pa.pa_last_device_error() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_topm(seed):
    rng = np.random.default_rng(9500 + seed)
    L, H, N = int(rng.integers(1, 6)), int(rng.integers(1, 9)), int(rng.integers(1, 3000))
    grid = rng.choice([0, 1, 4, 16])
    s = rng.standard_normal((L, H, N)).astype(np.float32)
    if grid:
        s = (np.round(s * grid) / grid).astype(np.float32)
    current = int(rng.integers(0, N))
    n = L * H * N
    dev = torch.from_numpy(s).cuda()
    for budget in (int(rng.integers(0, n + 2)), int(rng.integers(L * H, n + 1))):
        keep, per_head = pa.topm_retain(dev, current, budget)
        torch.cuda.synchronize()
        want = oracle.topm_retain(s, current, budget)
        assert np.array_equal(keep.cpu().numpy().astype(bool), want), (L, H, N, budget)
        assert np.array_equal(per_head.cpu().numpy(), want.sum(axis=2)), (L, H, N, budget)
    assert pa.pa_last_device_error() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_cascade(seed):
    """pa_decode_cascade on random fork counts, prefix and own lengths (page
    and tile edges included), heads, head dims, dtypes and range sizes,
    against the oracle on each fork's concatenated sequence."""
    import math
    from tests.test_cascade_gpu import _case as cascade_case, _oracle as cascade_oracle
    rng = np.random.default_rng(9500 + seed)
    hq, hkv = HEADS[rng.integers(len(HEADS))]
    D, dtype = int(rng.choice([64, 128])), str(rng.choice(["bf16", "fp16"]))
    B = int(rng.integers(1, 13))
    edges = [1, 15, 16, 17, 127, 128, 129, 511, 512, 513]
    prefix_len = int(rng.choice(edges)) if rng.random() < 0.5 else int(rng.integers(1, 1500))
    own = [int(rng.choice([0, 1, 15, 16, 17])) if rng.random() < 0.4
           else int(rng.integers(0, 200)) for _ in range(B)]
    part = int(rng.choice([0, 128, 256, 512]))
    q, kc, vc, ptab, tab, ctx = cascade_case(B, hq, hkv, D, dtype, prefix_len, own,
                                             seed=int(rng.integers(1 << 30)))
    scale = 1.0 / math.sqrt(D)
    ref = cascade_oracle(q, kc, vc, ptab, prefix_len, tab, own, scale,
                         workloads.DTYPE_CODE[dtype])
    out = pa.decode_cascade(q.cuda(), kc.cuda(), vc.cuda(), ptab.cuda(), prefix_len,
                            tab.cuda(), ctx.cuda(), scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref,
                 f"cascade B={B} {hq}/{hkv} D={D} {dtype} prefix {prefix_len} own {own} part {part}")
    assert pa.pa_last_device_error() == 0


@pytest.mark.parametrize("seed", range(10))
def test_random_topm_routes(seed):
    """Budgeted top-M retention on seeded random shapes: row lengths on both
    sides of 4096 (short rows sum per-row counts in shared memory, long rows
    per warp), arrays on both sides of 2M scores (the sampled first digit),
    coarse and fine score grids, any current position and budget; the kept
    set is unique, so masks and per-row counts must equal the oracle's."""
    rng = np.random.default_rng(7400 + seed)
    N = int(rng.choice([int(rng.integers(1, 4096)), int(rng.integers(4096, 70000)),
                        4095, 4096, 4097]))
    if seed % 3 == 0:  # 2.2M-4.5M scores: the sampled first digit
        rows = -(-int(rng.integers(2_200_000, 4_500_000)) // N)
        L = int(rng.integers(1, 9))
        H = -(-rows // L)
    else:
        L = int(rng.integers(1, 9))
        H = int(rng.integers(1, 9))
    n = L * H * N
    s = rng.standard_normal((L, H, N)).astype(np.float32)
    grid = rng.choice([0, 2, 16, 256])
    if grid:
        s = (np.round(s * grid) / grid).astype(np.float32)
    current = int(rng.integers(0, N))
    budgets = {int(rng.integers(0, n + 10)), L * H + int(rng.integers(1, max(2, n // 4))),
               n // 4}
    dev = torch.from_numpy(s).cuda()
    for budget in sorted(budgets):
        keep, per_head = pa.topm_retain(dev, current, budget)
        torch.cuda.synchronize()
        want = oracle.topm_retain(s, current, budget)
        got = keep.cpu().numpy().astype(bool)
        assert np.array_equal(got, want), (L, H, N, current, budget, grid,
                                           int((got != want).sum()))
        assert np.array_equal(per_head.cpu().numpy(), want.sum(axis=2)), (L, H, N, budget)
    assert pa.pa_last_device_error() == 0
