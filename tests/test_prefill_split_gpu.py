"""GPU parity of pa_prefill_paged_split (chunked prefill with key-range
partitions and an exact merge) against the float64 oracle.

The short-chunk cases are the verify step of speculative decoding: gamma
drafted tokens per sequence attend the cache and, causally, each other, in
one pass ("推理系统与性能工程", speculative sampling); the oracle's prefill is
that computation's definition (query i of a chunk after ctx cached tokens
sees keys 0 .. ctx + i)."""
import pytest
import torch

import oracle
import paged_kv_cache_171_gb300 as pa
import workloads
from tests.gpu_support import assert_close, to_device
from workloads import compact_host_copy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_171_gb300 import build
    build.build()


@pytest.mark.parametrize("head_dim,hq,hkv,dtype,cached,n_new,part", [
    (128, 64, 8, "bf16", [0, 700, 3000], 4, 256),     # verify, gamma 4, GQA-8, ctx 0
    (128, 32, 8, "bf16", [5000], 8, 0),                # automatic partitions
    (64, 16, 16, "fp16", [1000, 129], 2, 128),         # MHA, smallest partition
    (128, 32, 4, "bf16", [2500, 37], 70, 512),         # both row tiles of a CTA
    (64, 12, 4, "fp16", [1, 250], 33, 128),
    (128, 64, 8, "bf16", [300], 1, 128),               # one query: decode
    (128, 16, 2, "bf16", [2047, 2048, 2049], 3, 1024), # ctx at partition edges
    (128, 64, 8, "bf16", [126, 127, 129], 4, 0),       # odd key tile unseen by some rows
    (128, 64, 8, "bf16", [900, 3000], 8, 0),           # 64 rows: head/remainder row halves
    (128, 64, 8, "fp16", [900, 3000], 9, 0),           # 72 rows: interleaved tiles only
    (64, 32, 4, "bf16", [700, 2100], 16, 0),           # 64 rows at D 64
])
def test_split_prefill_small_shapes(head_dim, hq, hkv, dtype, cached, n_new, part):
    kw = dict(layers=1, batch=len(cached), n_q_heads=hq, n_kv_heads=hkv,
              head_dim=head_dim, page_size=16, ctx=cached, dtype=dtype, seed=41,
              n_new=n_new, kind="prefill", extra_pool_pages=5)
    cpu = workloads.paged_case(**kw)
    ref = oracle.prefill(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0],
                         cpu.ctx_lens, cpu.scale, cpu.dtype_code)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    out = pa.prefill_split(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                           dev.ctx_lens, dev.scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"split prefill {hq}/{hkv} D={head_dim} part {part}")
    assert pa.pa_last_device_error() == 0


def test_split_equals_unsplit_on_the_same_inputs():
    """Both paths compute the same attention: they differ by rounding only."""
    kw = dict(layers=1, batch=2, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=16,
              ctx=[4000, 1500], dtype="bf16", seed=43, n_new=16, kind="prefill")
    dev = to_device(workloads.paged_case(**kw), "cuda")
    a = pa.prefill(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0], dev.ctx_lens,
                   dev.scale)
    b = pa.prefill_split(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                         dev.ctx_lens, dev.scale, partition_tokens=512)
    torch.cuda.synchronize()
    assert_close(b.cpu().numpy(), a.cpu().numpy().astype("float64"), "split vs unsplit")
    assert pa.pa_last_device_error() == 0


@pytest.mark.parametrize("part", [0, 512])
def test_verify_gamma4_ctx32k_sampled_sequences(part):
    """Speculative-decoding verify at the 32k GQA-8 decode shape: 4 sequences
    x 32768 cached tokens, 64/8 heads, 4 drafted tokens each; two whole
    sequences against the oracle."""
    n_new = 4
    case = workloads.paged_case(layers=1, batch=4, n_q_heads=64, n_kv_heads=8,
                                head_dim=128, page_size=16, ctx=[32768] * 4, dtype="bf16",
                                seed=1004, n_new=n_new, kind="prefill", device="cuda")
    out = pa.prefill_split(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                           case.ctx_lens, case.scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    seqs = [0, 3]
    q, k, v, table, ctx = compact_host_copy(case, 0, seqs, extra_tokens=n_new)
    ref = oracle.prefill(q, k, v, table, ctx, case.scale, case.dtype_code)
    sel = torch.tensor(seqs, device="cuda")
    assert_close(out.index_select(0, sel).cpu().numpy(), ref, f"verify part {part}")
