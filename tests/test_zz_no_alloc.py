"""pa_decode_static_workspace: the decode entry point for callers that cannot
allocate device memory (a host framework that owns every allocation, a
latency-critical path where cudaMalloc may synchronise the device, a caller
with only the C ABI and no allocator).  Its split-K scratch lives in the
library's fixed 16 MiB device array.  Checked through the C ABI, on two calls
in a row that both use split-K plans (so the second sees the first call's
leftovers in the shared array), against the float64 oracle and against
pa_decode with a caller-allocated workspace.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_171_gb300 as pa
import workloads
from tests.gpu_support import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from paged_kv_cache_171_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return pa.lib()


def _args(case, out):
    hq, D = case.q.shape[2], case.q.shape[3]
    pages, hkv = case.k_cache.shape[0], case.k_cache.shape[1]
    B, mb = case.block_table.shape[1], case.block_table.shape[2]
    return (case.q[0].data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(),
            case.block_table[0].data_ptr(), case.ctx_lens.data_ptr(), out.data_ptr(),
            ctypes.c_float(case.scale), hq, hkv, D, 16, B, mb, pages, case.dtype_code)


def _reference(L, case, part):
    """pa_decode with a workspace torch allocated for it."""
    hq, D = case.q.shape[2], case.q.shape[3]
    hkv = case.k_cache.shape[1]
    B, mb = case.block_table.shape[1], case.block_table.shape[2]
    out = torch.empty((B, hq, D), dtype=torch.float32, device="cuda")
    ws_bytes = L.pa_decode_workspace_size(B, hq, hkv, D, 16, mb, part)
    ws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.pa_decode(*_args(case, out), part, ws.data_ptr(), ws_bytes, stream)
    assert rc == 0, pa.pa_strerror(rc)
    return out


def _static(L, case, part):
    hq, D = case.q.shape[2], case.q.shape[3]
    B = case.block_table.shape[1]
    out = torch.full((B, hq, D), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.pa_decode_static_workspace(*_args(case, out), part, stream)
    assert rc == 0, pa.pa_strerror(rc)
    return out


def test_static_workspace_matches_oracle_and_pa_decode_on_two_calls_in_a_row(L):
    # call 1: long GQA-8 contexts, 512-token partitions (8.5 MB of partials)
    kw1 = dict(layers=1, batch=4, n_q_heads=64, n_kv_heads=8, head_dim=128, page_size=16,
               ctx=[32768, 1, 20000, 777], dtype="bf16", seed=901)
    # call 2: different shapes and a plan of its own (automatic partitions)
    kw2 = dict(layers=1, batch=6, n_q_heads=16, n_kv_heads=4, head_dim=64, page_size=16,
               ctx=[3000, 0, 4096, 17, 999, 2500], dtype="fp16", seed=902, q_mul=2.0)
    c1 = to_device(workloads.paged_case(**kw1), "cuda")
    c2 = to_device(workloads.paged_case(**kw2), "cuda")
    # both plans split, so both calls go through the shared array
    assert L.pa_decode_workspace_size(4, 64, 8, 128, 16, c1.block_table.shape[2], 512) > 0
    assert L.pa_decode_workspace_size(6, 16, 4, 64, 16, c2.block_table.shape[2], 0) > 0
    r1 = _reference(L, c1, 512)
    r2 = _reference(L, c2, 0)
    s1 = _static(L, c1, 512)
    s2 = _static(L, c2, 0)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    for n, (kw, s_out, r_out) in enumerate(((kw1, s1, r1), (kw2, s2, r2)), 1):
        cpu = workloads.paged_case(**kw)  # the same seeded bytes, on the host
        ref = oracle.decode(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0],
                            cpu.ctx_lens, cpu.scale, cpu.dtype_code)
        assert_close(s_out.cpu().numpy(), ref, f"static workspace, call {n}, vs the oracle")
        assert_close(s_out.cpu().numpy(), r_out.cpu().numpy(),
                     f"static workspace, call {n}, vs pa_decode")


def test_static_workspace_rejects_plans_beyond_its_array(L):
    # 64 sequences x 64 heads x 64 partitions x 130 floats = 136 MB > 16 MiB.
    # Real, valid buffers (empty contexts), so nothing could go wrong even if
    # the call were launched; it must be refused before any launch.
    B, hq, hkv, D, mb, pages = 64, 64, 8, 128, 2048, 64
    q = torch.zeros((B, hq, D), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((pages, hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bt = torch.zeros((B, mb), dtype=torch.int32, device="cuda")
    ctx = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.full((B, hq, D), 7.0, dtype=torch.float32, device="cuda")
    assert L.pa_decode_workspace_size(B, hq, hkv, D, 16, mb, 512) > 16 << 20
    rc = L.pa_decode_static_workspace(q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                      bt.data_ptr(), ctx.data_ptr(), out.data_ptr(),
                                      ctypes.c_float(0.1), hq, hkv, D, 16, B, mb,
                                      pages, 0, 512, None)
    assert rc == -15
    assert "16 MiB" in pa.pa_strerror(rc)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing was launched
