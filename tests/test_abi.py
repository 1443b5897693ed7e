"""libpa.so loads, exports every entry point include/pa.h declares, and rejects
invalid arguments on the host before touching a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_171_gb300 as pa
from paged_kv_cache_171_gb300 import build as pa_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pa.h")


@pytest.fixture(scope="module")
def L():
    pa_build.build()
    return pa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("pa_decode", "pa_append_kv", "pa_prefill_paged",
                 "pa_merge_partials", "pa_decode_workspace_size",
                 "pa_decode_partition_tokens", "pa_last_device_error",
                 "pa_strerror"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_exposes_same_names():
    for n in declared_functions():
        assert hasattr(pa, n), n


def test_strerror_names_every_status(L):
    for code in range(0, -18, -1):
        s = pa.pa_strerror(code)
        assert s and "unknown" not in s, code
    assert "unknown" in pa.pa_strerror(-999)


# Host validation: every case returns before any CUDA call, so no GPU is needed.
FAKE = 0x1000  # 16-byte aligned, never dereferenced on these paths


def _decode(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, ctx=FAKE, out=FAKE, scale=0.1,
             hq=32, hkv=8, d=128, p=16, b=2, mb=8, pages=16, dtype=0, pt=0,
             ws=None, wsb=0)
    a.update(kw)
    return L.pa_decode(a["q"], a["k"], a["v"], a["bt"], a["ctx"], a["out"],
                       ctypes.c_float(a["scale"]), a["hq"], a["hkv"], a["d"], a["p"],
                       a["b"], a["mb"], a["pages"], a["dtype"], a["pt"], a["ws"],
                       a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(out=None), -1), (dict(bt=None), -1),
    (dict(hq=30, hkv=8), -2), (dict(hkv=0), -2), (dict(hq=-4), -2),
    (dict(d=96), -3), (dict(d=256), -3),
    (dict(p=8), -4), (dict(p=32), -4),
    (dict(b=0), -5), (dict(mb=0), -5), (dict(pages=0), -5), (dict(b=70000), -5),
    (dict(pages=(1 << 31) // (8 * 16)), -5),
    (dict(dtype=2), -6),
    (dict(q=FAKE + 8), -8), (dict(k=FAKE + 2), -8), (dict(out=FAKE + 4), -8),
    (dict(pt=24), -9), (dict(pt=-16), -9),
    (dict(pt=16, ws=None, wsb=0), -7),
])
def test_decode_rejects_bad_arguments(L, kw, code):
    assert _decode(L, **kw) == code


def _decode_append(L, kn=FAKE, vn=FAKE, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, ctx=FAKE, out=FAKE, scale=0.1,
             hq=32, hkv=8, d=128, p=16, b=2, mb=8, pages=16, dtype=0, pt=0,
             ws=None, wsb=0)
    a.update(kw)
    return L.pa_decode_append(a["q"], kn, vn, a["k"], a["v"], a["bt"], a["ctx"], a["out"],
                              ctypes.c_float(a["scale"]), a["hq"], a["hkv"], a["d"], a["p"],
                              a["b"], a["mb"], a["pages"], a["dtype"], a["pt"], a["ws"],
                              a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(kn=None), -1), (dict(vn=None), -1), (dict(q=None), -1), (dict(k=None), -1),
    (dict(kn=FAKE + 8), -8), (dict(vn=FAKE + 2), -8), (dict(v=FAKE + 4), -8),
    (dict(hq=30, hkv=8), -2), (dict(d=96), -3), (dict(p=8), -4), (dict(b=0), -5),
    (dict(dtype=2), -6), (dict(pt=24), -9), (dict(pt=16, ws=None, wsb=0), -7),
])
def test_decode_append_rejects_bad_arguments(L, kw, code):
    """The fused step checks its new-token pointers, then everything pa_decode
    checks, before any CUDA call."""
    assert _decode_append(L, **kw) == code


def _group_tile(group):
    return 8 if group % 8 == 0 else 4 if group % 4 == 0 else 2 if group % 2 == 0 else 1


def _ws_bytes(b, hq, hkv, d, n_parts):
    """batch * heads * parts * (D + 4) floats, then one int32 arrival counter
    per (sequence, head group) at the next 16-byte boundary."""
    part = b * hq * n_parts * (d + 4) * 4
    return -(-part // 16) * 16 + b * hkv * ((hq // hkv) // _group_tile(hq // hkv)) * 4


def test_workspace_size_matches_layout(L):
    for b, hq, hkv, d, mb, pt in [(4, 64, 8, 128, 2048, 512), (3, 8, 8, 64, 5, 32),
                                  (1, 16, 16, 128, 32, 512), (2, 12, 2, 64, 9, 16)]:
        n_parts = -(-mb * 16 // pt) if pt < mb * 16 else 1
        want = _ws_bytes(b, hq, hkv, d, n_parts) if n_parts > 1 else 0
        assert L.pa_decode_workspace_size(b, hq, hkv, d, 16, mb, pt) == want
        got_pt = L.pa_decode_partition_tokens(b, hq, hkv, d, 16, mb, pt)
        assert got_pt == (pt if n_parts > 1 else 0)
    assert L.pa_decode_workspace_size(1, 30, 8, 128, 16, 8, 0) == 0  # invalid -> 0


def test_auto_partition_is_page_aligned_and_bounded(L):
    for b, hq, hkv, mb in [(8, 32, 32, 256), (64, 32, 8, 512), (4, 64, 8, 2048),
                           (1, 16, 16, 32), (1, 1, 1, 1)]:
        pt = L.pa_decode_partition_tokens(b, hq, hkv, 128, 16, mb, 0)
        assert pt >= 0 and pt % 16 == 0 and pt < mb * 16 + 1
        if pt:
            n_parts = -(-mb * 16 // pt)
            assert L.pa_decode_workspace_size(b, hq, hkv, 128, 16, mb, 0) == \
                _ws_bytes(b, hq, hkv, 128, n_parts)


def test_append_and_prefill_reject_bad_arguments(L):
    P = FAKE
    assert L.pa_append_kv(None, P, P, P, P, P, P, 1, 8, 128, 16, 2, 8, 16, 0, None) == -1
    assert L.pa_append_kv(P, P, P, P, P, P, P, 1, 8, 100, 16, 2, 8, 16, 0, None) == -3
    assert L.pa_append_kv(P, P, P, P, P, P, P, -1, 8, 128, 16, 2, 8, 16, 0, None) == -5
    assert L.pa_append_kv(P + 4, P, P, P, P, P, P, 1, 8, 128, 16, 2, 8, 16, 0, None) == -8
    assert L.pa_append_kv(P, P, P, P, P, P, P, 0, 8, 128, 16, 2, 8, 16, 0, None) == 0
    f = ctypes.c_float(0.1)
    assert L.pa_prefill_paged(P, P, P, P, P, 4, None, f, 32, 8, 128, 16, 2, 8, 16, 0, None) == -1
    assert L.pa_prefill_paged(P, P, P, P, P, 4, P, f, 32, 7, 128, 16, 2, 8, 16, 0, None) == -2
    assert L.pa_prefill_paged(P, P, P, P, P, -1, P, f, 32, 8, 128, 16, 2, 8, 16, 0, None) == -5
    assert L.pa_prefill_paged(P, P, P, P, P, 0, P, f, 32, 8, 128, 16, 2, 8, 16, 0, None) == 0
    assert L.pa_merge_partials(P, P, P, 2, 8, 128, 4, 0, None) == -9
    assert L.pa_merge_partials(P, P, P, 2, 8, 80, 4, 16, None) == -3
    assert L.pa_merge_partials(None, P, P, 2, 8, 128, 4, 16, None) == -1


def test_product_package_does_not_reach_the_oracle():
    """The product path never imports, links or runs anything under oracle/."""
    pkg = os.path.dirname(pa.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "pa_oracle" not in text and "liboracle" not in text, f


def test_prefill_split_plan_and_workspace(L):
    """Key-range partitions of the chunked prefill: multiples of 128 keys; the
    workspace holds (O, m, l, 2 pad) per row and partition."""
    for b, n_new, hq, hkv, d, mb, pt in [(4, 4, 64, 8, 128, 2048, 512),
                                         (2, 70, 32, 8, 64, 300, 1024),
                                         (1, 1, 16, 16, 128, 8, 128),
                                         (3, 5, 8, 8, 128, 4, 128)]:
        max_tokens = mb * 16
        n_parts = -(-max_tokens // pt) if pt < max_tokens else 1
        want = b * n_new * hq * n_parts * (d + 4) * 4 if n_parts > 1 else 0
        assert L.pa_prefill_workspace_size(b, n_new, hq, hkv, d, 16, mb, pt) == want
        got = L.pa_prefill_partition_tokens(b, n_new, hq, hkv, d, 16, mb, pt)
        assert got == (pt if n_parts > 1 else 0)
    assert L.pa_prefill_partition_tokens(4, 4, 64, 8, 128, 16, 2048, 100) == -9
    assert L.pa_prefill_partition_tokens(4, 4, 64, 8, 128, 16, 2048, 48) == -9
    # automatic: a multiple of 128 of at least 512 keys when row tiles are few,
    # no split when they already fill the GPU
    pt = L.pa_prefill_partition_tokens(4, 4, 64, 8, 128, 16, 2048, 0)
    assert pt % 128 == 0 and pt >= 512 and pt < 2048 * 16
    assert L.pa_prefill_partition_tokens(4, 512, 32, 8, 128, 16, 545, 0) == 0
    assert L.pa_prefill_workspace_size(4, 512, 32, 8, 128, 16, 545, 0) == 0


def test_prefill_auto_plan_is_one_full_wave(L):
    """The automatic key-range plan: with 32 row-tile CTAs (4 sequences x 8 kv
    heads, a verify-sized chunk of 4 tokens over 32k keys) four ranges of 8320
    keys give 128 CTAs, one wave on a GPU of 148-152 SMs; a chunk whose row
    tiles already fill most SMs is not split."""
    pt = L.pa_prefill_partition_tokens(4, 4, 64, 8, 128, 16, 2049, 0)
    assert pt == 8320 and -(-2049 * 16 // pt) == 4
    assert L.pa_prefill_partition_tokens(4, 8, 64, 8, 128, 16, 2049, 0) == 8320
    # 120 row-tile CTAs (15 sequences x 8 kv heads): one wave as they are
    assert L.pa_prefill_partition_tokens(15, 4, 64, 8, 128, 16, 2049, 0) == 0


def test_prefill_split_rejects_bad_arguments(L):
    P = FAKE
    f = ctypes.c_float(0.1)
    split = L.pa_prefill_paged_split
    # missing or short workspace, before any launch
    assert split(P, P, P, P, P, 4, P, f, 64, 8, 128, 16, 4, 2048, 16, 0, 512, None, 0,
                 None) == -7
    assert split(P, P, P, P, P, 4, P, f, 64, 8, 128, 16, 4, 2048, 16, 0, 512, P, 1024,
                 None) == -7
    assert split(P, P, P, P, P, 4, P, f, 64, 8, 128, 16, 4, 2048, 16, 0, 100, P, 1 << 30,
                 None) == -9
    assert split(None, P, P, P, P, 4, P, f, 64, 8, 128, 16, 4, 2048, 16, 0, 0, None, 0,
                 None) == -1
    assert split(P, P, P, P, P, 4, P, f, 64, 7, 128, 16, 4, 2048, 16, 0, 0, None, 0,
                 None) == -2
    assert split(P, P, P, P, P, 0, P, f, 64, 8, 128, 16, 4, 2048, 16, 0, 512, None, 0,
                 None) == 0


def test_decode_window_arguments_and_workspace(L):
    P = FAKE
    f = ctypes.c_float(0.1)
    win = L.pa_decode_window
    assert win(P, P, P, P, P, P, f, 32, 8, 128, 16, 2, 64, 16, 0, -1, 8, 0, None, 0,
               None) == -5
    assert win(P, P, P, P, P, P, f, 32, 8, 128, 16, 2, 64, 16, 0, 4, -2, 0, None, 0,
               None) == -5
    assert win(None, P, P, P, P, P, f, 32, 8, 128, 16, 2, 64, 16, 0, 4, 8, 0, None, 0,
               None) == -1
    # partitions cut the attended pages: at most ceil(s/16) + ceil(w/16) + 1
    mb = 2048
    for sink, window, pt in [(4, 4096, 512), (0, 100, 16), (16, 0, 16), (40000, 40000, 512)]:
        att = min(mb, -(-sink // 16) + -(-window // 16) + 1)
        n_parts = -(-att * 16 // pt) if pt < att * 16 else 1
        want = _ws_bytes(4, 64, 8, 128, n_parts) if n_parts > 1 else 0
        assert L.pa_decode_window_workspace_size(4, 64, 8, 128, 16, mb, sink, window, pt) == want
    assert L.pa_decode_window_workspace_size(4, 64, 8, 128, 16, mb, -1, 8, 0) == 0


def test_topm_arguments(L):
    P = FAKE
    ws = L.pa_topm_workspace_size(32, 32, 32768)
    n = 32 * 32 * 32768
    head = (2048 + 2048 + 1024) * 4 + 256 + -(-n // 4096) * 4  # histograms, state, tie counts
    assert ws == -(-head // 16) * 16 + 8 * n                   # + a candidate (index, key) per element
    assert L.pa_topm_workspace_size(0, 1, 1) == 0
    r = L.pa_topm_retain
    assert r(None, 2, 2, 8, 0, 5, P, None, P, ws, None) == -1
    assert r(P, 2, 2, 8, 8, 5, P, None, P, ws, None) == -5     # current outside
    assert r(P, 2, 2, 8, 0, -1, P, None, P, ws, None) == -5    # negative budget
    assert r(P, 2, 2, 8, 0, 5, P, None, P, 16, None) == -7     # workspace too small
    assert r(P + 4, 2, 2, 8, 0, 5, P, None, P, 1 << 20, None) == -8
    assert r(P, 1 << 16, 1 << 16, 2, 0, 5, P, None, P, 1 << 40, None) == -5


def test_chunks_longer_than_the_table_are_rejected(L):
    """n_new new tokens need n_new slots in the table even with no cache: a
    longer chunk is refused on the host (the kernels would otherwise clamp
    the context and still walk past the table row)."""
    P = FAKE
    f = ctypes.c_float(0.1)
    # max_blocks 1 = 16 slots: 17 new tokens cannot fit, 16 can
    assert L.pa_prefill_paged(P, P, P, P, P, 17, P, f, 8, 8, 128, 16, 2, 1, 16, 0, None) == -5
    assert L.pa_prefill_paged_split(P, P, P, P, P, 17, P, f, 8, 8, 128, 16, 2, 1, 16, 0, 0,
                                    None, 0, None) == -5
    assert L.pa_prefill_partition_tokens(2, 17, 8, 8, 128, 16, 1, 0) == -5
    assert L.pa_prefill_partition_tokens(2, 16, 8, 8, 128, 16, 1, 0) == 0


def test_cascade_arguments_and_workspace(L):
    P = FAKE
    f = ctypes.c_float(0.1)
    ws = L.pa_decode_cascade_workspace_size(32, 32, 8, 128, 16, 512, 8192, 512)
    # [batch][n_q_heads][prefix ranges + 1][head_dim + 4] floats: 16 ranges of
    # 512 and the forks' own keys
    assert ws == 32 * 32 * (16 + 1) * (128 + 4) * 4
    assert L.pa_decode_cascade_workspace_size(32, 32, 8, 128, 16, 512, 8192, 100) == 0
    assert L.pa_decode_cascade_workspace_size(32, 32, 8, 128, 16, 512, 0, 0) == 0
    assert L.pa_decode_cascade_workspace_size(32, 32, 8, 128, 16, 512, 8193, 0) == 0
    c = L.pa_decode_cascade
    # prefix_len outside [1, prefix_blocks * page_size], null, short workspace,
    # bad partition: all before any launch
    assert c(P, P, P, P, 0, 512, P, P, P, f, 32, 8, 128, 16, 32, 8, 1024, 0, 0, P, ws,
             None) == -5
    assert c(P, P, P, P, 8193, 512, P, P, P, f, 32, 8, 128, 16, 32, 8, 1024, 0, 0, P, ws,
             None) == -5
    assert c(P, P, P, None, 8192, 512, P, P, P, f, 32, 8, 128, 16, 32, 8, 1024, 0, 0, P, ws,
             None) == -1
    assert c(P, P, P, P, 8192, 512, P, P, P, f, 32, 8, 128, 16, 32, 8, 1024, 0, 512, P,
             ws - 4, None) == -7
    assert c(P, P, P, P, 8192, 512, P, P, P, f, 32, 8, 128, 16, 32, 8, 1024, 0, 100, P, ws,
             None) == -9
