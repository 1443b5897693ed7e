"""GPU parity of pa_decode_window (decode over an attention sink plus a
sliding window of recent keys) against the float64 oracle's decode_window."""
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


CASES = [
    # head_dim, hq, hkv, dtype, ctx, sink, window, partition_tokens
    (128, 32, 32, "fp16", [700, 1500, 33], 4, 256, 0),      # MHA, CUDA-core path
    (128, 64, 8, "bf16", [3000, 40, 1025], 4, 500, 0),      # GQA-8, mma path
    (128, 64, 8, "bf16", [3000, 1024], 4, 500, 64),         # small partitions (warp-owned)
    (64, 16, 4, "bf16", [999, 2048], 17, 333, 128),         # unaligned ranges, D 64
    (128, 16, 2, "fp16", [40, 41, 2000], 3, 30, 0),         # sink end and window start share a page
    (128, 32, 8, "bf16", [800, 100], 0, 1, 0),              # the last key only
    (128, 32, 8, "bf16", [800, 100], 1, 0, 0),              # the first key only
    (128, 32, 8, "bf16", [800, 100], 0, 0, 0),              # nothing attended: zeros
    (128, 32, 8, "bf16", [800, 100, 0], 400, 400, 0),       # covers sequence 0: plain decode
    (64, 8, 8, "bf16", [5000, 4097], 16, 4096, 512),        # page-aligned ranges, split
]


@pytest.mark.parametrize("head_dim,hq,hkv,dtype,ctx,sink,window,part", CASES)
def test_decode_window_small_shapes(head_dim, hq, hkv, dtype, ctx, sink, window, part):
    kw = dict(layers=1, batch=len(ctx), n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim,
              page_size=16, ctx=ctx, dtype=dtype, seed=51, extra_pool_pages=4)
    cpu = workloads.paged_case(**kw)
    ref = oracle.decode_window(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0],
                               cpu.ctx_lens, cpu.scale, cpu.dtype_code, sink, window)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    out = pa.decode_window(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                           dev.ctx_lens, dev.scale, sink, window, partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"window s={sink} w={window} part {part}")
    assert pa.pa_last_device_error() == 0


def test_window_covering_everything_equals_pa_decode():
    kw = dict(layers=1, batch=3, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=16,
              ctx=[1000, 17, 4000], dtype="bf16", seed=52)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    a = pa.decode(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0], dev.ctx_lens,
                  dev.scale)
    b = pa.decode_window(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                         dev.ctx_lens, dev.scale, 0, 4000)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_streaming_window_full_size_sampled_sequences():
    """32 sequences x 32768 cached tokens, 64/8 heads, 4 sink tokens + a 4096
    window: two whole sequences against the oracle."""
    sink, window = 4, 4096
    case = workloads.paged_case(layers=1, batch=32, n_q_heads=64, n_kv_heads=8,
                                head_dim=128, page_size=16, ctx=[32768] * 32, dtype="bf16",
                                seed=1007, device="cuda")
    out = pa.decode_window(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                           case.ctx_lens, case.scale, sink, window)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    seqs = [0, 31]
    q, k, v, table, ctx = compact_host_copy(case, 0, seqs)
    ref = oracle.decode_window(q, k, v, table, ctx, case.scale, case.dtype_code, sink, window)
    sel = torch.tensor(seqs, device="cuda")
    assert_close(out.index_select(0, sel).cpu().numpy(), ref, "streaming window")
