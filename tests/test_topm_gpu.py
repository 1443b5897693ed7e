"""GPU parity of pa_topm_retain (budgeted global top-M KV retention) with the
oracle: the kept set is unique, so the masks must be identical."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_171_gb300 as pa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_171_gb300 import build
    build.build()


def _scores(L, H, N, seed, grid=None):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((L, H, N)).astype(np.float32)
    if grid:  # coarse values: many exact ties across layers, heads and tokens
        s = (np.round(s * grid) / grid).astype(np.float32)
    return s


@pytest.mark.parametrize("L,H,N,current,grid", [
    (2, 3, 9, 4, 2), (4, 8, 1000, 999, 8), (3, 5, 4097, 0, None), (32, 8, 777, 300, 4),
    (1, 1, 1, 0, None), (5, 7, 33, 32, 1),
])
def test_topm_matches_oracle(L, H, N, current, grid):
    s = _scores(L, H, N, 71 + N, grid)
    n = L * H * N
    dev = torch.from_numpy(s).cuda()
    for budget in sorted({0, L * H - 1, L * H, L * H + 1, n // 3, n // 2, n - 1, n, n + 5}):
        if budget < 0:
            continue
        keep, per_head = pa.topm_retain(dev, current, budget)
        torch.cuda.synchronize()
        want = oracle.topm_retain(s, current, budget)
        got = keep.cpu().numpy().astype(bool)
        assert np.array_equal(got, want), (L, H, N, budget, int((got != want).sum()))
        assert np.array_equal(per_head.cpu().numpy(), want.sum(axis=2)), budget
    assert pa.pa_last_device_error() == 0


def test_topm_special_values():
    """-0.0 ties with 0.0 (the lower index wins), NaN ranks last, infinities."""
    s = np.zeros((2, 2, 8), dtype=np.float32)
    s[1, 1, 3] = -0.0
    s[0, 1, 2] = np.nan
    s[1, 0, 6] = np.inf
    s[0, 0, 5] = -np.inf
    s[1, 1, 7] = 1e-45  # smallest subnormal, above the zeros
    dev = torch.from_numpy(s).cuda()
    for budget in range(0, 33):
        keep, _ = pa.topm_retain(dev, 0, budget)
        torch.cuda.synchronize()
        assert np.array_equal(keep.cpu().numpy().astype(bool),
                              oracle.topm_retain(s, 0, budget)), budget


def test_topm_full_size():
    """32 layers x 8 heads x 32768 tokens (8.4M candidates), scores on a
    grid of 1/16 (heavy ties), budget = a quarter of the rows."""
    L, H, N = 32, 8, 32768
    g = torch.Generator(device="cuda").manual_seed(72)
    dev = (torch.randn(L, H, N, generator=g, device="cuda") * 16).round() / 16
    budget = L * H * N // 4
    keep, per_head = pa.topm_retain(dev, N - 1, budget)
    torch.cuda.synchronize()
    s = dev.cpu().numpy()
    want = oracle.topm_retain(s, N - 1, budget)
    got = keep.cpu().numpy().astype(bool)
    assert int(got.sum()) == budget and np.array_equal(got, want)
    assert np.array_equal(per_head.cpu().numpy(), want.sum(axis=2))


def test_topm_all_scores_equal():
    """Every element ties: the whole array is one candidate bucket and the
    index order alone decides (lowest (l, h, t) first)."""
    L, H, N = 3, 4, 5000
    s = np.full((L, H, N), 1.5, dtype=np.float32)
    dev = torch.from_numpy(s).cuda()
    n = L * H * N
    for budget in (L * H + 1, n // 3, n - 2):
        keep, per_head = pa.topm_retain(dev, 7, budget)
        torch.cuda.synchronize()
        want = oracle.topm_retain(s, 7, budget)
        assert np.array_equal(keep.cpu().numpy().astype(bool), want), budget
        assert np.array_equal(per_head.cpu().numpy(), want.sum(axis=2)), budget
    assert pa.pa_last_device_error() == 0
