"""GPU parity of pa_decode (and its split-K merge) against the float64 oracle,
through the C ABI, on seeded inputs: small shapes spanning several pages,
ragged tails, every head-group tiling and partition mode, then the five
workloads' decode shapes at full size on sampled rows."""
import zlib

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


def _run_decode(case, layer=0, partition_tokens=0):
    out = pa.decode(case.q[layer], case.k_cache, case.v_cache,
                    case.block_table[layer], case.ctx_lens, case.scale,
                    partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    return out


def _oracle(case_cpu, layer=0):
    return oracle.decode(case_cpu.q[layer], case_cpu.k_cache, case_cpu.v_cache,
                         case_cpu.block_table[layer], case_cpu.ctx_lens,
                         case_cpu.scale, case_cpu.dtype_code)


CTX_EDGES = [1, 15, 16, 17, 100, 511, 512, 513, 0]


@pytest.mark.parametrize("head_dim", [128, 64])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (8, 2), (16, 2), (12, 4),
                                    (12, 2), (64, 4)])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_decode_small_shapes(head_dim, hq, hkv, dtype):
    """Group sizes 1, 2, 4, 8 (one head tile), 3 and 6 (tiles of 1 and 2) and
    16 (two tiles of 8); contexts at and around page and partition edges."""
    seed = zlib.crc32(repr((head_dim, hq, hkv, dtype)).encode()) % 10000
    cpu = workloads.paged_case(layers=1, batch=len(CTX_EDGES), n_q_heads=hq,
                               n_kv_heads=hkv, head_dim=head_dim, page_size=16,
                               ctx=CTX_EDGES, dtype=dtype, seed=seed,
                               extra_pool_pages=5)
    ref = _oracle(cpu)
    dev = to_device(workloads.paged_case(layers=1, batch=len(CTX_EDGES), n_q_heads=hq,
                                         n_kv_heads=hkv, head_dim=head_dim,
                                         page_size=16, ctx=CTX_EDGES, dtype=dtype,
                                         seed=seed, extra_pool_pages=5), "cuda")
    for pt in (0, 16, 48, 512):
        out = _run_decode(dev, partition_tokens=pt).cpu().numpy()
        assert_close(out, ref, f"D={head_dim} {hq}/{hkv} {dtype} part={pt}")
        assert np.all(out[-1] == 0.0)  # ctx = 0
    assert pa.pa_last_device_error() == 0


def test_decode_long_random_lengths_all_partition_modes():
    lens = [4096, 1, 3000, 777, 2048, 16 * 37]
    cpu = workloads.paged_case(layers=1, batch=len(lens), n_q_heads=32, n_kv_heads=8,
                               head_dim=128, page_size=16, ctx=lens, dtype="bf16",
                               seed=77, q_mul=2.0)
    ref = _oracle(cpu)
    dev = to_device(workloads.paged_case(layers=1, batch=len(lens), n_q_heads=32,
                                         n_kv_heads=8, head_dim=128, page_size=16,
                                         ctx=lens, dtype="bf16", seed=77, q_mul=2.0),
                    "cuda")
    outs = []
    for pt in (0, 256, 512, 1024, 4096, 8192):
        out = _run_decode(dev, partition_tokens=pt).cpu().numpy()
        assert_close(out, ref, f"part={pt}")
        outs.append(out)
    # the same partition plan twice gives bit-identical results (no atomics)
    again = _run_decode(dev, partition_tokens=512).cpu().numpy()
    assert np.array_equal(again, outs[2])
    assert pa.pa_last_device_error() == 0


def test_decode_one_cta_holding_every_partition():
    """Four 512-token partitions of 128-page tables: one CTA per (sequence,
    head tile) whose four warps each own a partition and whose partial states
    the CTA folds itself (no cross-CTA merge); ragged lengths leave some warps
    without pages, and an empty sequence gives zeros."""
    lens = [2048, 600, 1, 0, 1500, 1537]
    for hq, hkv in [(32, 8), (16, 16)]:
        kw = dict(layers=1, batch=len(lens), n_q_heads=hq, n_kv_heads=hkv, head_dim=128,
                  page_size=16, ctx=lens, dtype="bf16", seed=41, max_blocks=128)
        cpu = workloads.paged_case(**kw)
        assert cpu.block_table.shape[2] == 128
        assert pa.pa_decode_partition_tokens(len(lens), hq, hkv, 128, 16, 128, 512) == 512
        ref = _oracle(cpu)
        out = _run_decode(to_device(workloads.paged_case(**kw), "cuda"),
                          partition_tokens=512).cpu().numpy()
        assert_close(out, ref, f"{hq}/{hkv} one CTA, four partitions")
        assert np.all(out[3] == 0.0)
    assert pa.pa_last_device_error() == 0


def test_split_decode_ignores_workspace_contents_and_streams_do_not_interfere():
    """The split plan's arrival counters live in the workspace: a workspace
    full of garbage (every counter -1) gives the right result, and two calls
    on two streams with their own workspaces run concurrently without
    affecting each other."""
    lens = [4096, 2500, 17, 1000]
    kw = dict(layers=1, batch=len(lens), n_q_heads=32, n_kv_heads=8, head_dim=128,
              page_size=16, ctx=lens, dtype="bf16", seed=43)
    ref = _oracle(workloads.paged_case(**kw))
    dev = to_device(workloads.paged_case(**kw), "cuda")
    B, hq, hkv, D, mb = len(lens), 32, 8, 128, dev.block_table.shape[2]
    for pt in (512, 256):
        ws_bytes = pa.pa_decode_workspace_size(B, hq, hkv, D, 16, mb, pt)
        assert ws_bytes > 0
        wss = [torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device="cuda") for _ in range(2)]
        outs = [torch.empty((B, hq, D), dtype=torch.float32, device="cuda") for _ in range(2)]
        streams = [torch.cuda.Stream() for _ in range(2)]
        torch.cuda.synchronize()
        for _ in range(3):
            for ws, out, st in zip(wss, outs, streams):
                with torch.cuda.stream(st):
                    pa.decode(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0],
                              dev.ctx_lens, dev.scale, partition_tokens=pt, out=out,
                              workspace=ws, stream=st.cuda_stream)
        torch.cuda.synchronize()
        for out in outs:
            assert_close(out.cpu().numpy(), ref, f"part={pt}, garbage workspace, two streams")
    assert pa.pa_last_device_error() == 0


def test_merge_partials_matches_oracle_merge():
    """pa_merge_partials on its own, fed the oracle's per-chunk states."""
    lens = [1000, 1, 512, 0, 333]
    part = 256
    cpu = workloads.paged_case(layers=1, batch=len(lens), n_q_heads=8, n_kv_heads=2,
                               head_dim=128, page_size=16, ctx=lens, dtype="bf16",
                               seed=5)
    n_parts = 5  # more parts than the longest row needs: the rest are not read
    parts = oracle.partials(cpu.q[0], cpu.k_cache, cpu.v_cache, cpu.block_table[0],
                            cpu.ctx_lens, cpu.scale, cpu.dtype_code, part, n_parts)
    ref = oracle.merge(parts)
    # the library's rows are (O, m, l, 2 unused floats): 16-byte aligned
    dev_parts = torch.zeros(parts.shape[:-1] + (128 + 4,), dtype=torch.float32)
    dev_parts[..., :130] = torch.tensor(parts, dtype=torch.float32)
    for b, T in enumerate(lens):
        nv = -(-T // part)
        dev_parts[b, :, nv:] = float("nan")  # must never be read
    dev_parts = dev_parts.cuda()
    out = torch.empty((len(lens), 8, 128), dtype=torch.float32, device="cuda")
    pa.pa_merge_partials(dev_parts, cpu.ctx_lens.cuda(), out, len(lens), 8, 128,
                         n_parts, part)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, "merge")
    assert pa.pa_last_device_error() == 0


def test_decode_status_reports_bad_block_and_bad_ctx():
    cpu = workloads.paged_case(layers=1, batch=2, n_q_heads=4, n_kv_heads=4,
                               head_dim=128, page_size=16, ctx=[40, 20], dtype="bf16",
                               seed=3)
    dev = to_device(cpu, "cuda")
    bt = dev.block_table.clone()
    bt[0, 0, 1] = dev.k_cache.shape[0] + 5  # outside the pool: skipped, flagged
    pa.decode(dev.q[0], dev.k_cache, dev.v_cache, bt[0], dev.ctx_lens, dev.scale)
    assert pa.pa_last_device_error() == -11
    assert pa.pa_last_device_error() == 0  # cleared by the previous read
    ctx = dev.ctx_lens.clone()
    ctx[1] = 16 * bt.shape[2] + 1  # beyond the table: clamped, flagged
    pa.decode(dev.q[0], dev.k_cache, dev.v_cache, dev.block_table[0], ctx, dev.scale)
    assert pa.pa_last_device_error() == -12
    assert pa.pa_last_device_error() == 0


# ---- the workloads' decode shapes at full size ----------------------------------

def _full_size_check(name, layers_to_check, seqs, partition_tokens=0):
    cfg = workloads.CONFIGS[name]
    case = workloads.config_case(name, device="cuda")
    for layer in layers_to_check:
        out = _run_decode(case, layer, partition_tokens)
        q, k, v, table, ctx = compact_host_copy(case, layer, seqs)
        ref = oracle.decode(q, k, v, table, ctx, case.scale, case.dtype_code)
        got = out.index_select(0, torch.as_tensor(seqs, device="cuda")).cpu().numpy()
        assert_close(got, ref, f"{name} layer {layer}")
    assert pa.pa_last_device_error() == 0
    del case
    torch.cuda.empty_cache()


def test_full_mha_b1_ctx512():
    _full_size_check("mha_b1_ctx512", [0], [0])


def test_full_llama7b_b8_ctx4096_sampled():
    _full_size_check("llama7b_b8_ctx4096", [0, 17, 31], [0, 3, 7])


def test_full_gqa4_b64_ragged_sampled():
    _full_size_check("gqa4_b64_ragged", [0, 31], [0, 1, 13, 42, 63])


def test_full_gqa8_b4_ctx32k_all_rows():
    _full_size_check("gqa8_b4_ctx32k", [0], [0, 1, 2, 3], partition_tokens=512)


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    """A wait on a barrier phase nothing completes (a copy that never lands)
    ends after the 2 s limit with PA_ERR_TIMEOUT in the status word; the next
    call runs normally."""
    import time
    t0 = time.monotonic()
    pa.pa_selftest_wait_timeout()
    status = pa.pa_last_device_error()
    dt = time.monotonic() - t0
    assert status == -13, pa.pa_strerror(status)  # PA_ERR_TIMEOUT
    assert 1.5 < dt < 30.0, dt
    assert pa.pa_last_device_error() == 0  # read and cleared
    kw = dict(layers=1, batch=2, n_q_heads=8, n_kv_heads=8, head_dim=64, page_size=16,
              ctx=[100, 33], dtype="bf16", seed=99)
    ref = _oracle(workloads.paged_case(**kw))
    out = _run_decode(to_device(workloads.paged_case(**kw), "cuda"), partition_tokens=0)
    assert_close(out.cpu().numpy(), ref, "decode after a timed-out wait")
    assert pa.pa_last_device_error() == 0
