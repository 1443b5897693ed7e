"""The seeded input recipe (CPU): determinism, the block tables' page
permutation, context-length draws, value distributions and the five workloads'
sizes.  The GPU parity tests and the bench take every input from here."""
import math

import numpy as np
import pytest
import torch

import workloads


def _small(**over):
    kw = dict(layers=3, batch=5, n_q_heads=8, n_kv_heads=2, head_dim=64, page_size=16,
              ctx=(1, 300), dtype="bf16", seed=11)
    kw.update(over)
    return workloads.paged_case(**kw)


def test_same_seed_same_bytes_other_seed_other_bytes():
    a, b, c = _small(), _small(), _small(seed=12)
    for name in ("q", "k_cache", "v_cache", "block_table", "ctx_lens"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert not torch.equal(a.k_cache, c.k_cache)


def test_block_tables_deal_out_a_permutation_of_the_pool():
    case = _small(extra_pool_pages=7)
    bt = case.block_table.numpy()
    ctx = case.ctx_lens.numpy()
    pool = case.k_cache.shape[0]
    used = []
    for layer in range(bt.shape[0]):
        for b in range(bt.shape[1]):
            n = math.ceil(int(ctx[b]) / 16)
            row = bt[layer, b]
            assert np.all(row[n:] == -1)            # unused slots are flagged
            assert np.all((row[:n] >= 0) & (row[:n] < pool))
            used.extend(row[:n].tolist())
    assert len(used) == len(set(used))              # no page serves two blocks
    assert pool == len(used) + 7
    # pages are dealt out by a permutation, not in order
    assert used != sorted(used)


def test_context_lengths_fixed_list_or_uniform_inclusive():
    g = torch.Generator().manual_seed(3)
    t = workloads.draw_ctx_lens(4000, (128, 8192), g)
    assert t.dtype == torch.int32
    assert int(t.min()) >= 128 and int(t.max()) <= 8192
    assert int(t.min()) < 200 and int(t.max()) > 8100  # both ends reachable
    assert torch.equal(workloads.draw_ctx_lens(3, 77, g), torch.full((3,), 77, dtype=torch.int32))
    assert workloads.draw_ctx_lens(2, [5, 9], g).tolist() == [5, 9]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_values_are_rounded_standard_normals(dtype):
    case = _small(dtype=dtype, layers=1, batch=2, ctx=4096, n_kv_heads=4, q_mul=2.0)
    assert case.k_cache.dtype == workloads.DTYPES[dtype]
    k = case.k_cache.float().numpy().ravel()
    assert abs(k.mean()) < 0.01 and abs(k.std() - 1.0) < 0.01
    q = case.q.float().numpy().ravel()      # q_mul = 2: a peakier softmax
    assert abs(q.std() - 2.0) < 0.1
    assert case.scale == pytest.approx(1.0 / math.sqrt(64))


def test_prefill_pages_hold_the_chunk():
    case = _small(kind="prefill", n_new=20, ctx=[50, 3, 0, 16, 100])
    assert tuple(case.q.shape) == (3, 5, 20, 8, 64)
    blocks = case.block_table[0].numpy() >= 0
    assert blocks.sum(axis=1).tolist() == [math.ceil((t + 20) / 16) for t in [50, 3, 0, 16, 100]]
    assert case.ctx_lens.tolist() == [50, 3, 0, 16, 100]     # tokens before the chunk


def test_the_five_workloads():
    c = workloads.CONFIGS
    assert set(c) == {"mha_b1_ctx512", "llama7b_b8_ctx4096", "gqa4_b64_ragged",
                      "gqa8_b4_ctx32k", "prefill_b4_512over8192"}
    llama = c["llama7b_b8_ctx4096"]
    # one pool of 65,536 pages = 32 layers x 8 sequences x 4096 / 16 blocks
    assert llama["pool_pages"] == llama["layers"] * llama["batch"] * llama["ctx"] // 16
    assert (llama["n_q_heads"], llama["n_kv_heads"], llama["dtype"]) == (32, 32, "fp16")
    assert c["gqa4_b64_ragged"]["ctx"] == (128, 8192) and c["gqa4_b64_ragged"]["q_mul"] == 2.0
    assert c["gqa8_b4_ctx32k"]["partition_tokens"] == 512
    pre = c["prefill_b4_512over8192"]
    assert (pre["kind"], pre["ctx"], pre["n_new"]) == ("prefill", 8192, 512)
    assert len({v["seed"] for v in c.values()}) == 5
    small = workloads.config_case("mha_b1_ctx512")
    assert small.k_cache.shape == (32, 16, 16, 128)
    assert sorted(small.block_table[0, 0].tolist()) == list(range(32))
