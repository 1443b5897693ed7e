"""Shared pieces of the GPU parity tests: the tolerance and moving seeded
cases to the device.  (Cutting a compact host copy of a few sequences of a
large device case for the oracle is `workloads.compact_host_copy`.)"""
from __future__ import annotations

import numpy as np

# The stated bar: |gpu - ref| <= 2e-3 + 1e-2 |ref| element-wise, fp32 outputs
# from bf16/fp16 inputs against the float64 oracle.
ATOL = 2e-3
RTOL = 1e-2


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (ATOL + RTOL * np.abs(ref))), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst at {i}: "
            f"got {got[i]!r} ref {ref[i]!r}; max abs err {err.max():.3e}")
    return float(err.max())


def to_device(case, device):
    case.q = case.q.to(device)
    case.k_cache = case.k_cache.to(device)
    case.v_cache = case.v_cache.to(device)
    case.block_table = case.block_table.to(device)
    case.ctx_lens = case.ctx_lens.to(device)
    return case
