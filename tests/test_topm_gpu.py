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


def _first_digit_path(ws):
    """(sure, redo) from the select's state in the workspace (after the three
    histograms of 2048, 2048 and 1024 counts): sure = the 1/32 chunk sample
    named the first digit's bucket, redo = the exact first digit ran."""
    w = ws.cpu().numpy().view(np.uint32)
    state = w[(2048 + 2048 + 1024):][:12]
    return int(state[8]), int(state[9])


def _retain_large(s, current, budget):
    L, H, N = s.shape
    dev = torch.from_numpy(s).cuda()
    ws = torch.empty(pa.pa_topm_workspace_size(L, H, N) // 4, dtype=torch.int32, device="cuda")
    keep, per_head = pa.topm_retain(dev, current, budget, workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    want = oracle.topm_retain(s, current, budget)
    got = keep.cpu().numpy().astype(bool)
    assert np.array_equal(got, want), int((got != want).sum())
    assert np.array_equal(per_head.cpu().numpy(), want.sum(axis=2))
    return _first_digit_path(ws)


def test_topm_sample_confirmed():
    """8 x 8 x 65536 normal scores, a quarter kept: the sample names the
    threshold's first-digit bucket and the split pass confirms it."""
    s = _scores(8, 8, 65536, 73)
    assert _retain_large(s, 65535, s.size // 4) == (1, 0)


def test_topm_sample_misled():
    """The sampled chunks (every 32nd run of 4096 scores) hold scores 3 higher
    than the rest: the sample names a bucket far above the true threshold with
    full confidence, the split pass's counts refute it, and the exact first
    digit runs; the kept set is still exact."""
    s = _scores(8, 8, 65536, 74)
    flat = s.reshape(-1, 4096)
    flat[::32] += 3.0
    assert _retain_large(s, 100, s.size // 4) == (1, 1)


def test_topm_sample_unsure():
    """Two values only, 1.0 on a quarter of the elements (at random) and 0.5
    elsewhere, budget = the count of ones + the rows: the threshold sits on
    the edge of the ones' bucket, inside the sample's error, so the sample
    names nothing and the exact first digit runs."""
    rng = np.random.default_rng(75)
    L, H, N = 8, 8, 65536
    s = np.where(rng.random((L, H, N)) < 0.25, 1.0, 0.5).astype(np.float32)
    cur = 9
    ones = int((np.delete(s, cur, axis=2) == 1.0).sum())
    assert _retain_large(s, cur, ones + L * H) == (0, 1)


def test_topm_sample_all_equal():
    """4M equal scores: one bucket holds every candidate; the sample names it,
    the split pass lists the whole array and the index order decides."""
    s = np.full((4, 16, 65536), -2.25, dtype=np.float32)
    assert _retain_large(s, 0, s.size // 3) == (1, 0)
