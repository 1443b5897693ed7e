"""The bench's algorithmic counters against the figures they must reproduce:
the LLaMA-7B KV bytes per token (2 tensors x 32 layers x 4096 channels x 2
bytes), the unique bytes of one decode call of the 4 k and 32 k workloads,
and the chunked-prefill FLOPs (4 FLOP per (query head, visible key, dim))."""
import bench


def test_kv_bytes_per_token_llama7b():
    # one cached token of one sequence, 32 heads x 128, fp16, over 32 layers;
    # the q read and fp32 output written are separate terms
    per_layer = bench.decode_bytes([1], 32, 32, 128) - 32 * 128 * (2 + 4)
    assert 32 * per_layer == 524288


def test_decode_call_bytes():
    # 8 sequences x 4096 tokens, 32/32 heads (the 4 k step's layer call) and
    # 4 sequences x 32768 tokens, 64/8 heads: the same KV bytes, 512 MiB
    kv = 512 * 1024 * 1024
    assert bench.decode_bytes([4096] * 8, 32, 32, 128) == kv + 8 * 32 * 128 * 6 == 537067520
    assert bench.decode_bytes([32768] * 4, 64, 8, 128) == kv + 4 * 64 * 128 * 6 == 537067520


def test_prefill_flops():
    # query i of 512 new tokens after 8192 cached sees 8192 + i + 1 keys
    keys = sum(8192 + i + 1 for i in range(512))
    want = 4 * (4 * 32 * 128 * keys)
    got = bench.prefill_flops([8192] * 4, 512, 32, 128)
    assert got == want == 283484618752
