"""GPU parity of pa_append_kv (bit-exact against the oracle's scatter) and of
pa_prefill_paged (within tolerance of the float64 oracle), through the C ABI."""
import numpy as np
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
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert pa.pa_last_device_error() == 0


@pytest.mark.parametrize("head_dim,hkv,dtype", [(128, 8, "bf16"), (64, 4, "fp16"),
                                                (128, 32, "fp16")])
def test_append_is_bit_exact(head_dim, hkv, dtype):
    lens = [0, 15, 16, 31, 200, 1023]
    cpu = workloads.paged_case(layers=1, batch=len(lens), n_q_heads=hkv,
                               n_kv_heads=hkv, head_dim=head_dim, page_size=16,
                               ctx=[t + 40 for t in lens], dtype=dtype, seed=21)
    bt = cpu.block_table[0]
    # several new tokens per sequence at consecutive positions (a chunk append)
    seq_idx, pos = [], []
    for b, t in enumerate(lens):
        for j in range(1 + b % 3):
            seq_idx.append(b)
            pos.append(t + j)
    n_tok = len(pos)
    k_new, v_new = workloads.new_tokens(n_tok, hkv, head_dim, dtype, seed=22)
    k_ref, v_ref = oracle.append_kv(k_new, v_new, cpu.k_cache, cpu.v_cache, bt,
                                    np.array(seq_idx, np.int32), np.array(pos, np.int32))
    kc, vc = cpu.k_cache.cuda(), cpu.v_cache.cuda()
    pa.append_kv(k_new.cuda(), v_new.cuda(), kc, vc, bt.cuda(),
                 torch.tensor(seq_idx, dtype=torch.int32, device="cuda"),
                 torch.tensor(pos, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert np.array_equal(oracle.bits(kc), k_ref)
    assert np.array_equal(oracle.bits(vc), v_ref)
    assert pa.pa_last_device_error() == 0


def test_append_reports_bad_index_and_skips_it():
    cpu = workloads.paged_case(layers=1, batch=2, n_q_heads=4, n_kv_heads=4,
                               head_dim=128, page_size=16, ctx=[20, 20], dtype="bf16",
                               seed=23)
    kc, vc = cpu.k_cache.cuda(), cpu.v_cache.cuda()
    before = kc.clone()
    k_new, v_new = workloads.new_tokens(2, 4, 128, "bf16", seed=24, device="cuda")
    bt = cpu.block_table[0].cuda()
    pa.append_kv(k_new, v_new, kc, vc, bt,
                 torch.tensor([0, 5], dtype=torch.int32, device="cuda"),  # seq 5: bad
                 torch.tensor([3, 3], dtype=torch.int32, device="cuda"))
    assert pa.pa_last_device_error() == -14
    page, slot = int(cpu.block_table[0, 0, 0]), 3
    assert torch.equal(kc[page, :, slot], k_new[0])
    kc[page, :, slot] = before[page, :, slot]
    assert torch.equal(kc, before)
    pa.append_kv(k_new, v_new, kc, vc, bt,
                 torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                 torch.tensor([3, 16 * bt.shape[1]], dtype=torch.int32, device="cuda"))
    assert pa.pa_last_device_error() == -14


@pytest.mark.parametrize("head_dim,hq,hkv,dtype,cached,n_new", [
    (128, 32, 8, "bf16", [0, 100, 1000], 70),
    (128, 8, 8, "fp16", [5, 0], 3),
    (64, 16, 2, "bf16", [64, 17], 129),
    (128, 16, 16, "bf16", [300], 1),
    (64, 12, 4, "fp16", [1, 250], 33),
])
def test_prefill_small_shapes(head_dim, hq, hkv, dtype, cached, n_new):
    kw = dict(layers=1, batch=len(cached), n_q_heads=hq, n_kv_heads=hkv,
              head_dim=head_dim, page_size=16, ctx=cached, dtype=dtype, seed=31,
              n_new=n_new, kind="prefill", extra_pool_pages=3)
    cpu = workloads.paged_case(**kw)
    ref = oracle.prefill(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0],
                         cpu.ctx_lens, cpu.scale, cpu.dtype_code)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    out = pa.prefill(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                     dev.ctx_lens, dev.scale)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"prefill {hq}/{hkv} D={head_dim}")
    assert pa.pa_last_device_error() == 0


def test_prefill_full_workload_sampled_sequences():
    """4 x 512 new tokens over 8192 cached, 32/8 heads: two whole sequences."""
    case = workloads.config_case("prefill_b4_512over8192", device="cuda")
    out = pa.prefill(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                     case.ctx_lens, case.scale)
    torch.cuda.synchronize()
    seqs = [0, 3]
    n_new = case.n_new
    ctx = case.ctx_lens.cpu()
    bt = case.block_table[0].cpu()
    for s in seqs:
        nb = (int(ctx[s]) + n_new + 15) // 16
        idx = bt[s, :nb].to(torch.int64).cuda()
        k = case.k_cache.index_select(0, idx).cpu()
        v = case.v_cache.index_select(0, idx).cpu()
        table = torch.arange(nb, dtype=torch.int32).unsqueeze(0)
        ref = oracle.prefill(case.q[0, s:s + 1].cpu(), k, v, table, ctx[s:s + 1],
                             case.scale, case.dtype_code)
        assert_close(out[s:s + 1].cpu().numpy(), ref, f"prefill seq {s}")
    assert pa.pa_last_device_error() == 0


def test_append_then_decode_round_trip():
    """Append a decode step's new K/V with pa_append_kv, then pa_decode over
    ctx + 1 tokens matches the oracle run on the oracle's own append."""
    lens = [31, 64, 100]
    cpu = workloads.paged_case(layers=1, batch=3, n_q_heads=16, n_kv_heads=4,
                               head_dim=128, page_size=16, ctx=[t + 1 for t in lens],
                               dtype="bf16", seed=41)
    bt = cpu.block_table[0]
    k_new, v_new = workloads.new_tokens(3, 4, 128, "bf16", seed=42)
    k_ref, v_ref = oracle.append_kv(k_new, v_new, cpu.k_cache, cpu.v_cache, bt,
                                    np.arange(3, dtype=np.int32),
                                    np.array(lens, np.int32))
    ref = oracle.decode(cpu.q[0], k_ref.reshape(cpu.k_cache.shape),
                        v_ref.reshape(cpu.v_cache.shape), bt, cpu.ctx_lens, cpu.scale,
                        cpu.dtype_code)
    dev = to_device(cpu, "cuda")
    pa.append_kv(k_new.cuda(), v_new.cuda(), dev.k_cache, dev.v_cache, dev.block_table[0],
                 torch.arange(3, dtype=torch.int32, device="cuda"),
                 torch.tensor(lens, dtype=torch.int32, device="cuda"))
    out = pa.decode(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                    dev.ctx_lens, dev.scale)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, "append+decode")
    assert pa.pa_last_device_error() == 0


@pytest.mark.parametrize("scale", [-0.3, 0.0])
def test_prefill_negative_and_zero_scale(scale):
    """The kernel ranks raw scores, so a negative scale is folded into Q's
    sign and a zero scale becomes a tiny positive factor (every weight 1)."""
    kw = dict(layers=1, batch=2, n_q_heads=16, n_kv_heads=4, head_dim=128, page_size=16,
              ctx=[90, 7], dtype="bf16", seed=33, n_new=20, kind="prefill")
    cpu = workloads.paged_case(**kw)
    ref = oracle.prefill(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0],
                         cpu.ctx_lens, scale, cpu.dtype_code)
    dev = to_device(workloads.paged_case(**kw), "cuda")
    out = pa.prefill(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0], dev.ctx_lens,
                     scale)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"prefill scale {scale}")
    assert pa.pa_last_device_error() == 0
