"""Pins for the float64 oracle: it is checked against what the pages and the
mathematics fix, never against itself or the CUDA library.

Each test names the plausible oracle mistake it would catch.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.paged_helpers import scatter_to_pages, sdpa_reference

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return oracle.bits(t)


# --- 16-bit decoders: checked against torch's own casts (library routine) ---

@pytest.mark.parametrize("dtype,code", [(torch.bfloat16, oracle.BF16),
                                        (torch.float16, oracle.F16)])
def test_half_decoders_match_torch_casts(dtype, code):
    pats = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    vals = pats.view(dtype).to(torch.float64).numpy()
    u = pats.numpy().view(np.uint16)
    sample = np.concatenate([np.arange(0, 1 << 16, 97), [0, 1, 0x3ff, 0x400,
                             0x7bff, 0x7c00, 0x8000, 0x8001, 0xfbff, 0xfc00,
                             0x3f80, 0x7f7f, 0x0080, 0x007f]]).astype(np.int64)
    for i in sample:
        got = oracle.decode_half(int(u[i]), code)
        want = vals[i]
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want, (hex(int(u[i])), got, want)


# --- hand-derived closed forms (tests/golden/tiny_decode.json) ---------------

def test_hand_derived_cases():
    """Catches a dropped or misplaced scale, a wrong gather (page/slot
    transposed), a sign error in the exponent."""
    data = json.load(open(os.path.join(GOLDEN, "tiny_decode.json")))
    e = math.e
    # the fixture's numbers are the closed forms written in its derivation
    assert data["cases"][0]["expected"] == pytest.approx([1 / (1 + e), e / (1 + e)], abs=1e-15)
    for case in data["cases"]:
        D, P = case["head_dim"], case["page_size"]
        T = len(case["k"])
        bt = np.array([case["block_table"]], dtype=np.int32)
        num_pages = max(case["block_table"]) + 1
        kc = torch.zeros((num_pages, 1, P, D), dtype=torch.bfloat16)
        vc = torch.zeros_like(kc)
        for t in range(T):
            page, slot = case["block_table"][t // P], t % P
            kc[page, 0, slot] = torch.tensor(case["k"][t])
            vc[page, 0, slot] = torch.tensor(case["v"][t])
        q = torch.tensor([[case["q"]]], dtype=torch.bfloat16)
        out = oracle.decode(q, kc, vc, bt, np.array([T], np.int32),
                            case["scale"], oracle.BF16)
        np.testing.assert_allclose(out[0, 0], case["expected"], rtol=0, atol=1e-15)


# --- library route: torch SDPA in float64 --------------------------------------

@pytest.mark.parametrize("B,hq,hkv,D,P,lens", [
    (2, 4, 4, 16, 4, [9, 13]),       # MHA
    (3, 8, 2, 32, 16, [1, 17, 40]),  # GQA 4, ragged, one-token context
    (2, 8, 1, 8, 8, [33, 7]),        # MQA
])
def test_decode_matches_sdpa(B, hq, hkv, D, P, lens):
    """Catches transposed q/k, a wrong GQA head mapping (h % h_kv instead of
    h // G), softmax over the wrong axis, a missing 1/ℓ normalisation."""
    g = torch.Generator().manual_seed(11)
    Tm = max(lens)
    q = torch.randn(B, hq, D, generator=g).to(torch.bfloat16)
    kc = torch.randn(B, hkv, Tm, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, hkv, Tm, D, generator=g).to(torch.bfloat16)
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, lens, P, g)
    scale = 1 / math.sqrt(D)
    got = oracle.decode(q, k_cache, v_cache, bt, np.array(lens, np.int32), scale,
                        oracle.BF16)
    want = sdpa_reference(q, kc, vc, lens, scale).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_gqa_equals_mha_on_duplicated_kv_heads():
    """GQA with G-fold duplicated KV heads laid out as MHA gives the same
    answer; and h_kv = h_q reduces to per-head attention."""
    g = torch.Generator().manual_seed(5)
    B, hq, hkv, D, P, lens = 2, 8, 2, 16, 4, [11, 6]
    G = hq // hkv
    q = torch.randn(B, hq, D, generator=g).to(torch.float16)
    kc = torch.randn(B, hkv, 11, D, generator=g).to(torch.float16)
    vc = torch.randn(B, hkv, 11, D, generator=g).to(torch.float16)
    k1, v1, bt1 = scatter_to_pages(kc, vc, lens, P, g)
    gqa = oracle.decode(q, k1, v1, bt1, np.array(lens, np.int32), 0.25, oracle.F16)
    kd, vd = kc.repeat_interleave(G, dim=1), vc.repeat_interleave(G, dim=1)
    k2, v2, bt2 = scatter_to_pages(kd, vd, lens, P, g)
    mha = oracle.decode(q, k2, v2, bt2, np.array(lens, np.int32), 0.25, oracle.F16)
    np.testing.assert_array_equal(gqa, mha)


# --- special cases with closed forms -----------------------------------------

def _rand_paged(seed, B=2, hq=4, hkv=2, D=16, P=4, lens=(7, 12), dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    Tm = max(lens)
    q = torch.randn(B, hq, D, generator=g).to(dtype)
    kc = torch.randn(B, hkv, Tm, D, generator=g).to(dtype)
    vc = torch.randn(B, hkv, Tm, D, generator=g).to(dtype)
    return g, q, kc, vc


def test_one_token_context_returns_v0_exactly():
    g, q, kc, vc = _rand_paged(1, lens=(1, 1))
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [1, 1], 4, g)
    out = oracle.decode(q, k_cache, v_cache, bt, np.array([1, 1], np.int32), 0.3,
                        oracle.BF16)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b, h], vc[b, h // 2, 0].double().numpy())


def test_identical_v_rows_return_that_row():
    """The weights sum to one whatever q is."""
    g, q, kc, vc = _rand_paged(2)
    row = torch.randn(16, generator=g).to(torch.bfloat16)
    vc[:] = row
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [7, 12], 4, g)
    out = oracle.decode(q, k_cache, v_cache, bt, np.array([7, 12], np.int32), 0.25,
                        oracle.BF16)
    np.testing.assert_allclose(out, np.broadcast_to(row.double().numpy(), out.shape),
                               rtol=1e-14, atol=1e-15)


def test_zero_query_gives_mean_of_v_rows():
    g, q, kc, vc = _rand_paged(3)
    q.zero_()
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [7, 12], 4, g)
    out = oracle.decode(q, k_cache, v_cache, bt, np.array([7, 12], np.int32), 0.25,
                        oracle.BF16)
    for b, T in enumerate([7, 12]):
        for h in range(4):
            want = vc[b, h // 2, :T].double().mean(0).numpy()
            np.testing.assert_allclose(out[b, h], want, rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_v_and_does_not_overflow():
    """q = lambda * k_j with scores near 1000: exp without the max shift would
    overflow to inf/NaN; with it the answer is v_j."""
    g, q, kc, vc = _rand_paged(4, B=1, hq=1, hkv=1, lens=(9,))
    j = 5
    k = kc[0, 0, j].double()
    lam = 1000.0 / float((k * k).sum())
    q[0, 0] = (lam * k).to(torch.bfloat16)
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [9], 4, g)
    out = oracle.decode(q, k_cache, v_cache, bt, np.array([9], np.int32), 1.0,
                        oracle.BF16)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], vc[0, 0, j].double().numpy(), atol=1e-10)


def test_zero_context_gives_zeros():
    g, q, kc, vc = _rand_paged(6)
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [7, 12], 4, g)
    out = oracle.decode(q, k_cache, v_cache, bt, np.array([0, 12], np.int32), 0.25,
                        oracle.BF16)
    assert np.all(out[0] == 0.0) and np.any(out[1] != 0.0)


def test_paging_is_transparent():
    """Two different random page layouts of the same logical contents give
    bit-identical results (the gather, not the layout, decides)."""
    g, q, kc, vc = _rand_paged(7, lens=(13, 5))
    a = scatter_to_pages(kc, vc, [13, 5], 4, torch.Generator().manual_seed(100))
    b = scatter_to_pages(kc, vc, [13, 5], 4, torch.Generator().manual_seed(200),
                         extra_pages=9)
    assert not torch.equal(a[2], b[2])
    oa = oracle.decode(q, *a, np.array([13, 5], np.int32), 0.25, oracle.BF16)
    ob = oracle.decode(q, *b, np.array([13, 5], np.int32), 0.25, oracle.BF16)
    np.testing.assert_array_equal(oa, ob)


def test_out_of_range_block_is_an_error():
    g, q, kc, vc = _rand_paged(8)
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [7, 12], 4, g)
    bt = bt.clone()
    bt[1, 2] = k_cache.shape[0]
    with pytest.raises(ValueError):
        oracle.decode(q, k_cache, v_cache, bt, np.array([7, 12], np.int32), 0.25,
                      oracle.BF16)


# --- online recurrence and exact merge (19.6.2) --------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_online_recurrence_equals_full_softmax(seed):
    """Any block partition gives the full-softmax answer (up to rounding):
    the recurrence only uses e^(a+b) = e^a e^b.  A missing rescale factor c
    on l or on O breaks this."""
    lens = [37, 64]
    g, q, kc, vc = _rand_paged(20 + seed, lens=lens, D=8)
    q = (q.float() * 3).to(torch.bfloat16)  # peaky rows make a wrong c visible
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, lens, 4, g)
    full = oracle.decode(q, k_cache, v_cache, bt, np.array(lens, np.int32), 0.5,
                         oracle.BF16)
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, 64), size=rng.integers(1, 12),
                              replace=False))
    onl = oracle.decode_online(q, k_cache, v_cache, bt, np.array(lens, np.int32),
                               0.5, oracle.BF16, cuts)
    np.testing.assert_allclose(onl, full, rtol=1e-12, atol=1e-13)
    one = oracle.decode_online(q, k_cache, v_cache, bt, np.array(lens, np.int32),
                               0.5, oracle.BF16, [])
    np.testing.assert_allclose(one, full, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("part_tokens", [1, 4, 5, 16, 64, 1000])
def test_partials_then_merge_equal_full_softmax(part_tokens):
    lens = [37, 64, 0]
    g, q, kc, vc = _rand_paged(40, B=3, lens=lens, D=8)
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, lens, 4, g)
    full = oracle.decode(q, k_cache, v_cache, bt, np.array(lens, np.int32), 0.5,
                         oracle.BF16)
    n_parts = -(-64 // part_tokens) + 2  # trailing parts are empty
    parts = oracle.partials(q, k_cache, v_cache, bt, np.array(lens, np.int32), 0.5,
                            oracle.BF16, part_tokens, n_parts)
    assert np.all(parts[2, :, :, -1] == 0) and np.all(np.isneginf(parts[2, :, :, -2]))
    merged = oracle.merge(parts)
    np.testing.assert_allclose(merged, full, rtol=1e-12, atol=1e-13)


def test_merge_closed_form_two_parts():
    """Two chunks summarised by hand: part A has one token (score a, value x),
    part B one token (score b, value y).  Merged: (e^a x + e^b y)/(e^a + e^b)."""
    a, b, x, y = 0.7, -1.3, np.array([2.0, -1.0]), np.array([0.5, 4.0])
    parts = np.array([[list(x * 1.0) + [a, 1.0], list(y * 1.0) + [b, 1.0],
                       [0.0, 0.0, -np.inf, 0.0]]])
    want = (math.exp(a) * x + math.exp(b) * y) / (math.exp(a) + math.exp(b))
    np.testing.assert_allclose(oracle.merge(parts)[0], want, rtol=1e-15)
    assert np.all(oracle.merge(parts[:, 2:3])[0] == 0.0)


# --- append and prefill ----------------------------------------------------------

def test_append_then_decode_matches_sdpa_on_extended_sequence():
    """After appending token T at position T, decode over T+1 tokens equals the
    library attention on the contiguous sequence with the new row at the end:
    pins append's (page, slot) addressing through a second route."""
    g = torch.Generator().manual_seed(9)
    B, hq, hkv, D, P = 2, 4, 2, 16, 4
    lens = [6, 8]            # 8 fills two pages exactly: the new token opens a page
    kc = torch.randn(B, hkv, 9, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, hkv, 9, D, generator=g).to(torch.bfloat16)
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [7, 9], P, g)
    # blank the rows that the append must write
    for b, T in enumerate(lens):
        page, slot = int(bt[b, T // P]), T % P
        k_cache[page, :, slot] = 0
        v_cache[page, :, slot] = 0
    k_new = torch.stack([kc[b, :, lens[b]] for b in range(B)])
    v_new = torch.stack([vc[b, :, lens[b]] for b in range(B)])
    k2, v2 = oracle.append_kv(k_new, v_new, k_cache, v_cache, bt,
                              np.arange(B, dtype=np.int32),
                              np.array(lens, np.int32))
    q = torch.randn(B, hq, D, generator=g).to(torch.bfloat16)
    new_lens = [t + 1 for t in lens]
    got = oracle.decode(q, k2.reshape(k_cache.shape), v2.reshape(v_cache.shape),
                        bt, np.array(new_lens, np.int32), 0.25, oracle.BF16)
    want = sdpa_reference(q, kc, vc, new_lens, 0.25).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_prefill_matches_sdpa_with_offset_causal_mask():
    """Query i of the chunk sees cached keys plus new keys 0..i: torch SDPA with
    an explicit boolean mask, float64."""
    import torch.nn.functional as F
    g = torch.Generator().manual_seed(13)
    B, hq, hkv, D, P, n_new = 2, 4, 2, 16, 4, 5
    cached = [7, 0]
    tot = [c + n_new for c in cached]
    Tm = max(tot)
    q = torch.randn(B, n_new, hq, D, generator=g).to(torch.bfloat16)
    kc = torch.randn(B, hkv, Tm, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, hkv, Tm, D, generator=g).to(torch.bfloat16)
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, tot, P, g)
    got = oracle.prefill(q, k_cache, v_cache, bt, np.array(cached, np.int32), 0.25,
                         oracle.BF16)
    for b in range(B):
        T = tot[b]
        mask = torch.zeros(n_new, T, dtype=torch.bool)
        for i in range(n_new):
            mask[i, :cached[b] + i + 1] = True
        o = F.scaled_dot_product_attention(
            q[b].double().transpose(0, 1).unsqueeze(0),
            kc[b, :, :T].double().unsqueeze(0), vc[b, :, :T].double().unsqueeze(0),
            attn_mask=mask, scale=0.25, enable_gqa=True)
        np.testing.assert_allclose(got[b], o[0].transpose(0, 1).numpy(),
                                   rtol=1e-12, atol=1e-12)


# --- KV bytes (tests/golden/kv_bytes.json) ---------------------------------------

def test_kv_byte_counts_match_the_pages():
    items = json.load(open(os.path.join(GOLDEN, "kv_bytes.json")))["items"]
    per_tok = items[0]
    assert oracle.kv_bytes_per_token(per_tok["n_layers"], per_tok["hidden"],
                                     per_tok["elem_bytes"]) == per_tok["bytes"]
    for it in items[1:3]:
        b = oracle.kv_bytes_eq3(it["n_layers"], it["hidden"], it["seq_len"], 1,
                                it["elem_bytes"])
        assert b == it["gib"] * 2 ** 30
    gpt3 = items[3]
    b = oracle.kv_bytes_eq3(gpt3["n_layers"], gpt3["hidden"], gpt3["seq_len"],
                            gpt3["batch"], gpt3["elem_bytes"])
    assert abs(b / 1e9 - gpt3["gb_approx"]) < 0.005
    # eq. 3 with S = B = 1 is the per-token figure of 19.4.2
    assert oracle.kv_bytes_eq3(32, 4096, 1, 1, 2) == oracle.kv_bytes_per_token(32, 4096, 2)


# --- attention sink + sliding window (decode over a kept key set) ----------

def _kept(T, sink, window):
    return [t for t in range(T) if t < sink or t >= T - window]


@pytest.mark.parametrize("sink,window", [(0, 64), (3, 40), (40, 0), (100, 100)])
def test_window_covering_the_sequence_equals_plain_decode(sink, window):
    """Keeping every key is plain decode (catches a window that drops the
    last key or a sink that drops the first)."""
    g, q, kc, vc = _rand_paged(21, lens=(23, 40))
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [23, 40], 4, g)
    lens = np.array([23, 40], np.int32)
    full = oracle.decode(q, k_cache, v_cache, bt, lens, 0.3, oracle.BF16)
    # every key of both sequences is kept: sink + window >= T
    keep_all = all(len(_kept(int(T), sink, window)) == int(T) for T in lens)
    got = oracle.decode_window(q, k_cache, v_cache, bt, lens, 0.3, oracle.BF16, sink, window)
    if keep_all:
        np.testing.assert_allclose(got, full, rtol=0, atol=1e-14)
    else:
        assert not np.allclose(got, full)


def test_window_of_one_returns_the_last_v_and_sink_of_one_the_first():
    """Catches an off-by-one at either end of the kept set."""
    g, q, kc, vc = _rand_paged(22, lens=(9, 17))
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [9, 17], 4, g)
    lens = np.array([9, 17], np.int32)
    last = oracle.decode_window(q, k_cache, v_cache, bt, lens, 0.3, oracle.BF16, 0, 1)
    first = oracle.decode_window(q, k_cache, v_cache, bt, lens, 0.3, oracle.BF16, 1, 0)
    none = oracle.decode_window(q, k_cache, v_cache, bt, lens, 0.3, oracle.BF16, 0, 0)
    for b, T in enumerate(lens):
        for h in range(4):
            assert np.array_equal(last[b, h], vc[b, h // 2, T - 1].double().numpy())
            assert np.array_equal(first[b, h], vc[b, h // 2, 0].double().numpy())
    assert np.array_equal(none, np.zeros_like(none))


@pytest.mark.parametrize("sink,window", [(4, 16), (1, 5), (7, 33), (0, 20), (13, 0)])
def test_window_matches_sdpa_on_the_gathered_keys(sink, window):
    """Library route: torch SDPA (float64) on the kept keys gathered in order
    (catches mixing up the two ranges or a wrong sequence end)."""
    lens = [57, 70]
    g, q, kc, vc = _rand_paged(23, lens=tuple(lens))
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, lens, 4, g)
    got = oracle.decode_window(q, k_cache, v_cache, bt, np.array(lens, np.int32), 0.25,
                               oracle.BF16, sink, window)
    for b, T in enumerate(lens):
        idx = torch.tensor(_kept(T, sink, window), dtype=torch.int64)
        kb = kc[b:b + 1].index_select(2, idx)
        vb = vc[b:b + 1].index_select(2, idx)
        ref = sdpa_reference(q[b:b + 1], kb, vb, [len(idx)], 0.25)
        np.testing.assert_allclose(got[b:b + 1], ref, rtol=0, atol=1e-12)


def test_window_hand_derived_case():
    """T = 3, sink 1, window 1: keys 0 and 2 only; key 1 would dominate if it
    were kept.  q = (1, 0), k = (0, 0), (8, 0), (1, 0), v = e1, (5, 5), e2:
    weights 1 / (1 + e) and e / (1 + e)."""
    kc = torch.tensor([[[[0., 0.], [8., 0.], [1., 0.]]]], dtype=torch.bfloat16)
    vc = torch.tensor([[[[1., 0.], [5., 5.], [0., 1.]]]], dtype=torch.bfloat16)
    q = torch.tensor([[[1., 0.]]], dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(0)
    k_cache, v_cache, bt = scatter_to_pages(kc, vc, [3], 2, g)
    got = oracle.decode_window(q, k_cache, v_cache, bt, np.array([3], np.int32), 1.0,
                               oracle.BF16, 1, 1)
    e = math.e
    np.testing.assert_allclose(got[0, 0], [1 / (1 + e), e / (1 + e)], rtol=0, atol=1e-15)


# --- budgeted global top-M KV retention --------------------------------------

def _naive_topm(scores, current, budget):
    """The pages' naive method: repeat (budget - L*H) times, scan the whole
    table for the best remaining candidate (highest score, then lowest
    layer, head, token)."""
    L, H, N = scores.shape
    keep = np.zeros((L, H, N), dtype=bool)
    keep[:, :, current] = True
    for _ in range(max(0, budget - L * H)):
        best = None
        for l in range(L):
            for h in range(H):
                for t in range(N):
                    if keep[l, h, t]:
                        continue
                    s = float(scores[l, h, t])
                    key = (1 if math.isnan(s) else 0, -s if not math.isnan(s) else 0.0, l, h, t)
                    if best is None or key < best[0]:
                        best = (key, (l, h, t))
        if best is None:
            break
        keep[best[1]] = True
    return keep


def test_topm_hand_derived_case():
    """L=1, H=2, N=4, C=3, M=5: the two current slots, then three of the six
    candidates: 0.9 (h1, t0); the 0.5 tie goes to head 0 (t2) before head 1
    (t1); then the other 0.5.  Catches a descending/ascending mix-up and a
    tie broken the wrong way."""
    scores = np.array([[[0.1, 0.2, 0.5, 9.0], [0.9, 0.5, 0.3, -1.0]]], dtype=np.float32)
    keep = oracle.topm_retain(scores, 3, 5)
    want = np.array([[[False, False, True, True], [True, True, False, True]]])
    assert np.array_equal(keep, want)
    keep4 = oracle.topm_retain(scores, 3, 4)  # the tie: head 0 wins
    assert np.array_equal(keep4, np.array([[[False, False, True, True],
                                            [True, False, False, True]]]))
    assert np.array_equal(oracle.topm_retain(scores, 3, 2), scores == scores[..., 3:4])
    assert oracle.topm_retain(scores, 3, 100).all()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_topm_equals_the_naive_repeated_scan(seed):
    """Ties (scores on a coarse grid), -0.0 and +0.0, a NaN: the one global
    sort equals the pages' naive repeated scan."""
    rng = np.random.default_rng(seed)
    L, H, N = 2, 3, 9
    scores = np.round(rng.normal(size=(L, H, N)) * 2) / 2
    scores[0, 1, 2] = -0.0
    scores[1, 0, 5] = 0.0
    scores[1, 2, 1] = np.nan
    scores = scores.astype(np.float32)
    for budget in (0, 5, 6, 7, 20, 40, 54, 60):
        got = oracle.topm_retain(scores, 4, budget)
        want = _naive_topm(scores, 4, budget)
        assert np.array_equal(got, want), budget
        assert got.sum() == min(max(budget, L * H), L * H * N)


def test_topm_counts_differ_per_head():
    """The budget is global: a head with high scores keeps more tokens."""
    scores = np.zeros((2, 2, 16), dtype=np.float32)
    scores[1, 0] = 10.0
    keep = oracle.topm_retain(scores, 15, 4 + 10)
    per_head = keep.sum(axis=2)
    assert per_head[1, 0] == 11 and per_head[0, 0] == 1 and per_head.sum() == 14
