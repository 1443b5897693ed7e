"""GPU parity of pa_decode_append (the step's K/V write and the decode over
the whole context, new token included, in one kernel) against the float64
oracle's append_kv followed by its decode ("吞吐与延迟的系统模型", section 4:
each decode step writes one token's K/V per layer and reads every cached one).
The caches must come out bit-exact; the outputs within the decode tolerance,
and bit-identical to pa_append_kv + pa_decode on the same plan."""
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


def _case(head_dim, hq, hkv, dtype, lens, seed):
    """lens[b] = tokens cached before the step; the step's token goes to
    position lens[b], and the decode attends lens[b] + 1 tokens."""
    return workloads.paged_case(layers=1, batch=len(lens), n_q_heads=hq, n_kv_heads=hkv,
                                head_dim=head_dim, page_size=16, ctx=[t + 1 for t in lens],
                                dtype=dtype, seed=seed, extra_pool_pages=3)


@pytest.mark.parametrize("head_dim,hq,hkv,dtype,lens,part", [
    (128, 16, 4, "bf16", [0, 15, 16, 31, 200], 0),   # slot 0 / 15 / 0 of page 1; T = 1
    (128, 32, 32, "fp16", [5, 100, 1000], 0),         # MHA, CUDA cores
    (64, 8, 2, "bf16", [63, 64, 500], 64),            # split, D 64
    (128, 64, 8, "bf16", [4095, 3000], 512),          # GQA-8, warp-owned partitions
    (128, 32, 8, "bf16", [1, 2, 3], 16),              # one-page partitions
    (128, 12, 4, "fp16", [77, 700], 0),               # group 3: three head tiles per kv head
    (64, 16, 2, "fp16", [300, 17], 32),               # GQA-8 at D 64
])
def test_decode_append_matches_oracle(head_dim, hq, hkv, dtype, lens, part):
    cpu = _case(head_dim, hq, hkv, dtype, lens, seed=61)
    bt = cpu.block_table[0]
    B = len(lens)
    k_new, v_new = workloads.new_tokens(B, hkv, head_dim, dtype, seed=62)
    k_ref, v_ref = oracle.append_kv(k_new, v_new, cpu.k_cache, cpu.v_cache, bt,
                                    np.arange(B, dtype=np.int32), np.array(lens, np.int32))
    ref = oracle.decode(cpu.q[0], k_ref.reshape(cpu.k_cache.shape),
                        v_ref.reshape(cpu.v_cache.shape), bt, cpu.ctx_lens, cpu.scale,
                        cpu.dtype_code)
    dev = to_device(cpu, "cuda")
    out = pa.decode_append(dev.q[0], k_new.cuda(), v_new.cuda(), dev.k_cache, dev.v_cache,
                           dev.block_table[0], dev.ctx_lens, dev.scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    assert np.array_equal(oracle.bits(dev.k_cache), k_ref)
    assert np.array_equal(oracle.bits(dev.v_cache), v_ref)
    assert_close(out.cpu().numpy(), ref, f"decode_append {hq}/{hkv} D={head_dim} part {part}")


@pytest.mark.parametrize("part", [0, 64])
def test_decode_append_equals_append_then_decode(part):
    """The fused call reads the new rows from its own copy of the page instead
    of the cache, with the same arithmetic: results are bit-identical."""
    lens = [3000, 17, 64, 1500]
    k_new, v_new = workloads.new_tokens(len(lens), 8, 128, "bf16", seed=64, device="cuda")
    a = to_device(_case(128, 32, 8, "bf16", lens, seed=63), "cuda")
    b = to_device(_case(128, 32, 8, "bf16", lens, seed=63), "cuda")  # an independent copy
    pa.append_kv(k_new, v_new, a.k_cache, a.v_cache, a.block_table[0],
                 torch.arange(len(lens), dtype=torch.int32, device="cuda"),
                 torch.tensor(lens, dtype=torch.int32, device="cuda"))
    two = pa.decode(a.q[0], a.k_cache, a.v_cache, a.block_table[0], a.ctx_lens, a.scale,
                    partition_tokens=part)
    one = pa.decode_append(b.q[0], k_new, v_new, b.k_cache, b.v_cache, b.block_table[0],
                           b.ctx_lens, b.scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    assert torch.equal(one, two)
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)


def test_decode_append_empty_sequence_and_bad_page():
    """T = 0 writes zeros and stores nothing; a bad page id for the new
    token's page stores nothing and records PA_ERR_BAD_BLOCK."""
    cpu = _case(128, 16, 4, "bf16", [40, 40], seed=65)
    dev = to_device(cpu, "cuda")
    dev.ctx_lens[0] = 0
    before_k, before_v = dev.k_cache.clone(), dev.v_cache.clone()
    k_new, v_new = workloads.new_tokens(2, 4, 128, "bf16", seed=66, device="cuda")
    out = pa.decode_append(dev.q[0], k_new, v_new, dev.k_cache, dev.v_cache,
                           dev.block_table[0], dev.ctx_lens, dev.scale)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    assert torch.count_nonzero(out[0]) == 0
    page, slot = int(cpu.block_table[0, 1, 40 // 16]), 40 % 16
    assert torch.equal(dev.k_cache[page, :, slot], k_new[1])
    assert torch.equal(dev.v_cache[page, :, slot], v_new[1])
    dev.k_cache[page, :, slot] = before_k[page, :, slot]
    dev.v_cache[page, :, slot] = before_v[page, :, slot]
    assert torch.equal(dev.k_cache, before_k) and torch.equal(dev.v_cache, before_v)
    dev.ctx_lens[0] = 41
    dev.block_table[0, 0, 40 // 16] = dev.k_cache.shape[0] + 7  # past the pool
    pa.decode_append(dev.q[0], k_new, v_new, dev.k_cache, dev.v_cache, dev.block_table[0],
                     dev.ctx_lens, dev.scale)
    assert pa.pa_last_device_error() == -11  # PA_ERR_BAD_BLOCK
    # sequence 1 stored its rows again; sequence 0 stored nothing
    dev.k_cache[page, :, slot] = before_k[page, :, slot]
    dev.v_cache[page, :, slot] = before_v[page, :, slot]
    assert torch.equal(dev.k_cache, before_k) and torch.equal(dev.v_cache, before_v)


def test_decode_append_context_beyond_the_table():
    """A context length past the table is reported (PA_ERR_BAD_CTX) and stores
    no token; the other sequences store theirs."""
    cpu = _case(128, 16, 4, "bf16", [40, 40], seed=69)
    dev = to_device(cpu, "cuda")
    before_k, before_v = dev.k_cache.clone(), dev.v_cache.clone()
    dev.ctx_lens[0] = dev.block_table.shape[2] * 16 + 5
    k_new, v_new = workloads.new_tokens(2, 4, 128, "bf16", seed=70, device="cuda")
    pa.decode_append(dev.q[0], k_new, v_new, dev.k_cache, dev.v_cache, dev.block_table[0],
                     dev.ctx_lens, dev.scale)
    assert pa.pa_last_device_error() == -12  # PA_ERR_BAD_CTX
    page, slot = int(dev.block_table[0, 1, 40 // 16]), 40 % 16
    assert torch.equal(dev.k_cache[page, :, slot], k_new[1])
    dev.k_cache[page, :, slot] = before_k[page, :, slot]
    dev.v_cache[page, :, slot] = before_v[page, :, slot]
    assert torch.equal(dev.k_cache, before_k) and torch.equal(dev.v_cache, before_v)


def test_decode_append_llama_layer_sampled_sequences():
    """The LLaMA-7B-shaped layer at full size (8 sequences x 4096 tokens, 32
    heads, bf16), the step's token at position 4095: two sequences against
    the oracle, every sequence's cache rows against the inputs."""
    B, H, D, T = 8, 32, 128, 4096
    case = workloads.paged_case(layers=1, batch=B, n_q_heads=H, n_kv_heads=H, head_dim=D,
                                page_size=16, ctx=[T] * B, dtype="bf16", seed=67,
                                device="cuda")
    k_new, v_new = workloads.new_tokens(B, H, D, "bf16", seed=68, device="cuda")
    out = pa.decode_append(case.q[0], k_new, v_new, case.k_cache, case.v_cache,
                           case.block_table[0], case.ctx_lens, case.scale)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    pages = case.block_table[0, :, (T - 1) // 16].long()
    assert torch.equal(case.k_cache[pages, :, (T - 1) % 16], k_new)
    assert torch.equal(case.v_cache[pages, :, (T - 1) % 16], v_new)
    seqs = [0, 5]
    q, k, v, table, ctx = compact_host_copy(case, 0, seqs)
    ref = oracle.decode(q, k, v, table, ctx, case.scale, case.dtype_code)
    sel = torch.tensor(seqs, device="cuda")
    assert_close(out.index_select(0, sel).cpu().numpy(), ref, "decode_append llama layer")


def test_decode_append_ragged_gqa_layer_sampled_sequences():
    """One layer of the ragged GQA-4 batch at full size (64 sequences of
    128-8192 tokens, 32/8 heads, bf16, Q x 2, the automatic split plan): every
    sequence's new rows land at position ctx - 1; the shortest, the longest and
    one more sequence against the oracle over the updated pages."""
    case = workloads.config_case("gqa4_b64_ragged", device="cuda", layers=1, pool_pages=None)
    B = case.q.shape[1]
    k_new, v_new = workloads.new_tokens(B, 8, 128, "bf16", seed=71, device="cuda")
    out = pa.decode_append(case.q[0], k_new, v_new, case.k_cache, case.v_cache,
                           case.block_table[0], case.ctx_lens, case.scale)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0
    pos = (case.ctx_lens - 1).long()
    pages = case.block_table[0].gather(1, (pos // 16).view(B, 1)).view(B).long()
    assert torch.equal(case.k_cache[pages, :, pos % 16], k_new)
    assert torch.equal(case.v_cache[pages, :, pos % 16], v_new)
    lens = case.ctx_lens.cpu()
    seqs = sorted({int(lens.argmin()), int(lens.argmax()), 17})
    q, k, v, table, ctx = compact_host_copy(case, 0, seqs)
    ref = oracle.decode(q, k, v, table, ctx, case.scale, case.dtype_code)
    sel = torch.tensor(seqs, device="cuda")
    assert_close(out.index_select(0, sel).cpu().numpy(), ref, "decode_append ragged GQA layer")
