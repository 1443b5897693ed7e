#!/usr/bin/env python3
"""Benchmark of the paged GQA decode step on GB300.

Headline workload (one "step" = one decode step of a 32-layer model): the
GQA continuous-batching batch, the largest decode workload that the pages
describe.  For each of 32 layers, one pa_decode_append call writes the step's
new K/V row of every sequence into its page and attends each query head over
the sequence's cached tokens, the new one included (paged gather, online
softmax, split-K partitions and their exact merge; pa_append_kv + pa_decode
in one kernel).  64 sequences with seeded lengths drawn
uniformly from [128, 8192], 32 query heads sharing 8 KV heads (GQA-4),
head_dim 128, bf16 KV, page_size 16, random block tables, Q drawn N(0,1) x 2
(peaky softmax).  The LLaMA-7B-shaped step (batch 8, 32/32 heads, context
4096, fp16) is measured the same way as a second block of the line.
Synthetic seeded data.

Metric: decode-attention HBM GB/s (algorithmic bytes = unique KV bytes read +
Q + fp32 output, per (sequence, layer)) and sequences*layers per second.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica of the workload (the
path shards by sequence with no data-path collective): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention HBM GB/s and % of GB300 HBM roofline; sequences·layers/sec"
HEADLINE = "gqa4_b64_ragged"
SECOND = "llama7b_b8_ctx4096"
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# byte and flop models (per (sequence, layer) call; "吞吐与延迟的系统模型" 4-5)

def decode_bytes(ctx_lens, n_q_heads, n_kv_heads, head_dim, elem_bytes=2):
    """Unique KV bytes read + Q read + fp32 output written, summed over the
    sequences of one layer call.  Block tables, the split-K workspace and any
    re-read are not counted."""
    kv = sum(2 * int(t) * n_kv_heads * head_dim * elem_bytes for t in ctx_lens)
    qo = len(ctx_lens) * n_q_heads * head_dim * (elem_bytes + 4)
    return kv + qo


def append_bytes(n_tok, n_kv_heads, head_dim, elem_bytes=2):
    """K and V rows read from the new-token buffers and written to the pages."""
    return 2 * 2 * n_tok * n_kv_heads * head_dim * elem_bytes


def decode_flops(ctx_lens, n_q_heads, head_dim):
    """4 * h_q * d * T per sequence: 2 FLOP per multiply-add of q.K^T and P.V."""
    return sum(4 * n_q_heads * head_dim * int(t) for t in ctx_lens)


def prefill_flops(cached, n_new, n_q_heads, head_dim):
    """Query i sees cached + i + 1 keys; 4 * d FLOP per (query head, key)."""
    keys = sum(n_new * int(c) + n_new * (n_new + 1) // 2 for c in cached)
    return 4 * n_q_heads * head_dim * keys


def prefill_bytes(cached, n_new, n_q_heads, n_kv_heads, head_dim, elem_bytes=2):
    kv = sum(2 * (int(c) + n_new) * n_kv_heads * head_dim * elem_bytes for c in cached)
    qo = len(cached) * n_new * n_q_heads * head_dim * (elem_bytes + 4)
    return kv + qo


# ---------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def traffic_record(workload, kernel_file="pa_decode.cu"):
    """DRAM bytes per launch of `workload`'s dominant kernel from the
    committed ncu summary, if it was taken on the current kernel source
    (sha256 of the .cu file), else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "paged_kv_cache_171_gb300", "csrc", kernel_file)
    try:
        with open(path) as f:
            rec = json.load(f)
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        ent = rec.get(workload)
        if ent and ent.get("kernel_file") == kernel_file and ent.get("source_sha256") == sha:
            return ent
    except (OSError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of this GPU's SM clock and throttle reasons."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_uuid(torch):
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------------------
# our arm

def run_decode_step(torch, pa, workloads, name, args, rank, world):
    """The decode step of one 32-layer workload: per layer, the step's token's
    K/V written into the cache and the decode over every cached token, new
    one included -- one pa_decode_append call (pa_append_kv + pa_decode in
    one kernel; the two-call form is timed beside it)."""
    cfg = workloads.CONFIGS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workloads.config_case(name, device=dev)
    L, B = case.layers, case.q.shape[1]
    hq, hkv, D = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    pages = case.k_cache.shape[0]
    mb = case.block_table.shape[2]
    ctx = case.ctx_lens                      # tokens held, the step's included
    pos = (ctx - 1).to(torch.int32)          # the step's token is the last one
    seq_idx = torch.arange(B, dtype=torch.int32, device=dev)
    k_new, v_new = workloads.new_tokens(L * B, hkv, D, cfg["dtype"], seed=cfg["seed"] + 1,
                                        device=dev)
    k_new = k_new.view(L, B, hkv, D)
    v_new = v_new.view(L, B, hkv, D)
    out = torch.empty((L, B, hq, D), dtype=torch.float32, device=dev)
    part = pa.pa_decode_partition_tokens(B, hq, hkv, D, 16, mb, 0)
    ws_bytes = pa.pa_decode_workspace_size(B, hq, hkv, D, 16, mb, 0)
    ws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=dev)
    dcode = case.dtype_code
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    launches_per_layer = 1 + (1 if part else 0)

    def step(ev=None):
        for layer in range(L):
            if ev is not None:
                ev[layer][0].record(stream)
            pa.pa_decode_append(case.q[layer], k_new[layer], v_new[layer], case.k_cache,
                                case.v_cache, case.block_table[layer], ctx, out[layer],
                                case.scale, hq, hkv, D, 16, B, mb, pages, dcode, 0, ws,
                                ws_bytes, sptr)
            if ev is not None:
                ev[layer][1].record(stream)

    def step_two_calls():
        for layer in range(L):
            pa.pa_append_kv(k_new[layer], v_new[layer], case.k_cache, case.v_cache,
                            case.block_table[layer], seq_idx, pos, B, hkv, D, 16, B, mb,
                            pages, dcode, sptr)
            pa.pa_decode(case.q[layer], case.k_cache, case.v_cache, case.block_table[layer],
                         ctx, out[layer], case.scale, hq, hkv, D, 16, B, mb, pages, dcode,
                         0, ws, ws_bytes, sptr)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0

    ctx_list = [int(t) for t in ctx.cpu()]
    per_layer_bytes = decode_bytes(ctx_list, hq, hkv, D)
    step_bytes = L * per_layer_bytes
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_uuid(torch)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(torch, world)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(torch, world)
    clocks = sampler.stop() if sampler else None
    status = pa.pa_last_device_error()
    assert status == 0, pa.pa_strerror(status)
    ms = t0.elapsed_time(t1)
    ms_max = allreduce_max(torch, world, ms)

    # The same steps as pa_append_kv + pa_decode per layer, for comparison
    for _ in range(2):
        step_two_calls()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step_two_calls()
    t1.record(stream)
    torch.cuda.synchronize()
    two_call_ms = t0.elapsed_time(t1)

    # The dominant call (pa_decode_append) timed on its own
    # stream with events around each call, over the same number of steps.
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(L)]
          for _ in range(args.steps)]
    for k in range(args.steps):
        step(ev[k])
    torch.cuda.synchronize()
    call_ms = [ev[k][l][0].elapsed_time(ev[k][l][1]) for k in range(args.steps)
               for l in range(L)]
    call_avg_ms = sum(call_ms) / len(call_ms)

    # ---- end to end through the public API with host buffers
    host_in = {
        "q": case.q.cpu().pin_memory(),
        "k_new": k_new.cpu().pin_memory(), "v_new": v_new.cpu().pin_memory(),
        "block_table": case.block_table.cpu().pin_memory(),
        "ctx_lens": ctx.cpu().pin_memory(),
    }
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h = host_out.numel() * host_out.element_size()

    # Copies run on streams of their own, in groups of 8 layers: a group's
    # inputs travel while earlier groups compute, its outputs return while
    # later ones do (per-layer copies cost more host time than they hide).
    # Two sets of device inputs and outputs alternate between steps, so that
    # step k + 1's inputs travel while step k computes and step k's outputs
    # return while step k + 1 does; a set is refilled only after the step
    # two back is done computing with it and its outputs are on the host.
    NB = 2
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host_in.items()}
              for _ in range(NB)]
    outs = [out] + [torch.empty_like(out) for _ in range(NB - 1)]
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    G = 8
    groups = [(g0, min(L, g0 + G)) for g0 in range(0, L, G)]
    ev_in = [[torch.cuda.Event() for _ in groups] for _ in range(NB)]
    ev_out = [[torch.cuda.Event() for _ in groups] for _ in range(NB)]
    ev_used = [torch.cuda.Event() for _ in range(NB)]  # a set's last step has computed
    ev_read = [torch.cuda.Event() for _ in range(NB)]  # ... and its outputs are read
    for e in ev_used + ev_read:
        e.record(stream)
    per_layer_in = ("q", "k_new", "v_new", "block_table")
    turn = [0]

    def step_e2e():
        k = turn[0] % NB
        turn[0] += 1
        din, o = dev_in[k], outs[k]
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(ev_used[k])
            din["ctx_lens"].copy_(host_in["ctx_lens"], non_blocking=True)
            for gi, (a, b) in enumerate(groups):
                for name_ in per_layer_in:
                    din[name_][a:b].copy_(host_in[name_][a:b], non_blocking=True)
                ev_in[k][gi].record(h2d_stream)
        stream.wait_event(ev_read[k])
        for gi, (a, b) in enumerate(groups):
            stream.wait_event(ev_in[k][gi])
            for layer in range(a, b):
                pa.pa_decode_append(din["q"][layer], din["k_new"][layer],
                                    din["v_new"][layer], case.k_cache, case.v_cache,
                                    din["block_table"][layer], din["ctx_lens"],
                                    o[layer], case.scale, hq, hkv, D, 16, B, mb, pages,
                                    dcode, 0, ws, ws_bytes, sptr)
            ev_out[k][gi].record(stream)
        ev_used[k].record(stream)
        with torch.cuda.stream(d2h_stream):
            for gi, (a, b) in enumerate(groups):
                d2h_stream.wait_event(ev_out[k][gi])
                host_out[a:b].copy_(o[a:b], non_blocking=True)
            ev_read[k].record(d2h_stream)

    for _ in range(2):
        step_e2e()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_stream.wait_stream(stream)  # the first step's inputs travel inside the timed region
    for _ in range(args.steps):
        step_e2e()
    stream.wait_stream(d2h_stream)  # ... and the last step's outputs are on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allreduce_max(torch, world, e0.elapsed_time(e1))
    assert pa.pa_last_device_error() == 0

    res = dict(
        name=name, cfg=cfg,
        case=case, ms=ms_max, step_bytes=step_bytes, per_layer_bytes=per_layer_bytes,
        call_avg_ms=call_avg_ms, clocks=clocks, part=part, L=L, B=B,
        two_call_ms=two_call_ms / args.steps,
        launches=args.steps * L * launches_per_layer,
        e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, ctx_list=ctx_list,
    )
    return res


def run_other_decode(torch, pa, workloads, name, steps, warmup, partition_tokens=0):
    """One more decode workload: per step, every layer's pa_decode call."""
    cfg = workloads.CONFIGS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workloads.config_case(name, device=dev)
    L, B = case.layers, case.q.shape[1]
    hq, hkv, D = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    pages, mb = case.k_cache.shape[0], case.block_table.shape[2]
    out = torch.empty((L, B, hq, D), dtype=torch.float32, device=dev)
    ws_bytes = pa.pa_decode_workspace_size(B, hq, hkv, D, 16, mb, partition_tokens)
    ws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=dev)
    part = pa.pa_decode_partition_tokens(B, hq, hkv, D, 16, mb, partition_tokens)
    stream = torch.cuda.current_stream()
    flush = None
    ctx_list = [int(t) for t in case.ctx_lens.cpu()]
    per_layer = decode_bytes(ctx_list, hq, hkv, D)
    # Working sets below 2x L2 are flushed (a 2x L2 write) before each step;
    # larger ones stream through L2 with no reuse from the previous step.
    if L * per_layer < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        for layer in range(L):
            pa.pa_decode(case.q[layer], case.k_cache, case.v_cache, case.block_table[layer],
                         case.ctx_lens, out[layer], case.scale, hq, hkv, D, 16, B, mb,
                         pages, case.dtype_code, partition_tokens, ws, ws_bytes,
                         stream.cuda_stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if flush is not None:
        # each step after a flush, timed alone (median)
        times = []
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
    else:
        # steps back to back between one pair of events: the device time per
        # step, without the host's per-call latency of a short step
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
    assert pa.pa_last_device_error() == 0
    gbs = L * per_layer / (ms * 1e-3) / 1e9
    res = {"ms_per_step": round(ms, 4), "GB_s": round(gbs, 1),
           "seq_layers_per_s": round(L * B / (ms * 1e-3), 1),
           "partition_tokens": part, "bytes_per_step": L * per_layer,
           "l2": "flushed (2x L2 write) before each step, each step timed alone"
           if flush is not None
           else "inputs larger than 2x L2, no flush; steps timed back to back"}
    del case, out, ws
    torch.cuda.empty_cache()
    return res


def run_prefill(torch, pa, workloads, steps, warmup, peaks):
    name = "prefill_b4_512over8192"
    cfg = workloads.CONFIGS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workloads.config_case(name, device=dev)
    B, n_new = case.q.shape[1], case.n_new
    hq, hkv, D = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    out = torch.empty((B, n_new, hq, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    cached = [int(t) for t in case.ctx_lens.cpu()]
    for _ in range(warmup):
        pa.prefill(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                   case.ctx_lens, case.scale, out=out)
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pa.prefill(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                   case.ctx_lens, case.scale, out=out)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    assert pa.pa_last_device_error() == 0
    ms = statistics.median(times)
    fl = prefill_flops(cached, n_new, hq, D)
    tf = fl / (ms * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", 1900.0)  # burst: the call is timed alone
    sustained = peaks.get("bf16_tflops_sustained", 1700.0)
    res = {"ms": round(ms, 4), "TFLOP_s": round(tf, 1), "flops": fl,
           "frac_of_bf16_peak": round(tf / peak, 4), "peak_tflops": peak,
           "frac_of_bf16_sustained": round(tf / sustained, 4),
           "kernel": "prefill_tc_kernel: tcgen05.mma, two 128-row tiles per CTA, P and O in TMEM",
           "l2": "flushed (2x L2 write) before each call"}
    del case, out
    torch.cuda.empty_cache()
    return res


def run_verify(torch, pa, workloads, steps, warmup, peaks, gamma=4):
    """Speculative-decoding verify at the 32k GQA-8 decode shape: 4 sequences
    x 32768 cached tokens, 64/8 heads, gamma drafted tokens attended in one
    pass (pa_prefill_paged_split, key ranges merged exactly).  HBM-bound like
    decode: algorithmic bytes = unique K/V of ctx + gamma tokens + q + fp32
    out.  The unsplit pa_prefill_paged is timed beside it."""
    dev = torch.device("cuda", torch.cuda.current_device())
    B, hq, hkv, D, ctx = 4, 64, 8, 128, 32768
    case = workloads.paged_case(layers=1, batch=B, n_q_heads=hq, n_kv_heads=hkv,
                                head_dim=D, page_size=16, ctx=[ctx] * B, dtype="bf16",
                                seed=1006, n_new=gamma, kind="prefill", device=dev)
    mb = case.block_table.shape[2]
    part = pa.pa_prefill_partition_tokens(B, gamma, hq, hkv, D, 16, mb, 0)
    ws_bytes = pa.pa_prefill_workspace_size(B, gamma, hq, hkv, D, 16, mb, 0)
    ws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=dev)
    out = torch.empty((B, gamma, hq, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    nbytes = (2 * (ctx + gamma) * hkv * D * 2) * B + B * gamma * hq * D * (2 + 4)

    def time_it(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    def split():
        pa.pa_prefill_paged_split(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                                  case.ctx_lens, gamma, out, case.scale, hq, hkv, D, 16, B,
                                  mb, case.k_cache.shape[0], case.dtype_code, 0, ws,
                                  ws_bytes, stream.cuda_stream)

    def unsplit():
        pa.pa_prefill_paged(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                            case.ctx_lens, gamma, out, case.scale, hq, hkv, D, 16, B, mb,
                            case.k_cache.shape[0], case.dtype_code, stream.cuda_stream)

    ms = time_it(split)
    ms_unsplit = time_it(unsplit)
    assert pa.pa_last_device_error() == 0
    gbs = nbytes / (ms * 1e-3) / 1e9
    res = {"ms_per_step": round(ms, 4), "GB_s": round(gbs, 1),
           "frac_of_hbm_peak": round(gbs / peaks.get("hbm_gbs", 6800.0), 4),
           "gamma": gamma, "partition_tokens": part, "bytes_per_step": nbytes,
           "unsplit_ms": round(ms_unsplit, 4),
           "kernel": "prefill_tc_kernel over key ranges + merge_kernel",
           "l2": "inputs larger than 2x L2, no flush; steps timed back to back"}
    del case, out, ws
    torch.cuda.empty_cache()
    return res


def run_window(torch, pa, workloads, steps, warmup, peaks, sink=4, window=4096):
    """Attention-sink + sliding-window decode (pa_decode_window): 32 sequences
    x 32768 cached tokens, 64/8 heads, bf16, 4 sink tokens and a 4096-token
    window.  Algorithmic bytes = K/V of the sink + window keys + q + fp32
    out; plain decode of the same caches is timed beside it."""
    dev = torch.device("cuda", torch.cuda.current_device())
    B, hq, hkv, D, ctx = 32, 64, 8, 128, 32768
    case = workloads.paged_case(layers=1, batch=B, n_q_heads=hq, n_kv_heads=hkv,
                                head_dim=D, page_size=16, ctx=[ctx] * B, dtype="bf16",
                                seed=1007, device=dev)
    mb = case.block_table.shape[2]
    out = torch.empty((B, hq, D), dtype=torch.float32, device=dev)
    ws_bytes = pa.pa_decode_window_workspace_size(B, hq, hkv, D, 16, mb, sink, window, 0)
    ws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    kept = min(ctx, sink + window)
    nbytes = B * (2 * kept * hkv * D * 2 + hq * D * (2 + 4))

    def time_it(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    ms = time_it(lambda: pa.pa_decode_window(
        case.q[0], case.k_cache, case.v_cache, case.block_table[0], case.ctx_lens, out,
        case.scale, hq, hkv, D, 16, B, mb, case.k_cache.shape[0], case.dtype_code, sink,
        window, 0, ws, ws_bytes, stream.cuda_stream))
    assert pa.pa_last_device_error() == 0
    gbs = nbytes / (ms * 1e-3) / 1e9
    res = {"ms_per_step": round(ms, 4), "GB_s": round(gbs, 1),
           "frac_of_hbm_peak": round(gbs / peaks.get("hbm_gbs", 6800.0), 4),
           "sink": sink, "window": window, "context": ctx, "bytes_per_step": nbytes,
           "kernel": "decode_kernel over the sink + window pages (in-kernel merge when split)",
           "l2": "inputs larger than 2x L2, no flush; steps timed back to back"}
    del case, out, ws
    torch.cuda.empty_cache()
    return res


def run_prefix_sharing(torch, pa, steps, warmup, peaks, B=32, prefix=8192, suffix=128):
    """Prefix sharing through the page pool: B sequences forked from one
    prefix of `prefix` tokens, each with `suffix` tokens of its own (32/8
    heads, D 128, bf16).  pa_decode reads the shared pages once per sequence
    from the block tables (they stay in L2, so logical bytes -- as if every
    sequence held its own copy -- move faster than HBM); pa_decode_cascade
    reads them once for all sequences.  The same lengths on unshared pages are
    timed beside them, and the copy-on-write page copy (pa_copy_pages) on
    4096 pages."""
    import numpy as np
    dev = torch.device("cuda", torch.cuda.current_device())
    hq, hkv, D = 32, 8, 128
    T = prefix + suffix
    mb = (T + 15) // 16
    n_pref = prefix // 16
    n_own = mb - n_pref
    n_pages = n_pref + B * n_own + B * mb  # shared layout, then an unshared one
    g = torch.Generator(device=dev).manual_seed(1008)
    kc = torch.randn(n_pages, hkv, 16, D, generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn(n_pages, hkv, 16, D, generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn(B, hq, D, generator=g, device=dev).to(torch.bfloat16)
    pool = pa.pa_pool_create(n_pages)
    try:
        root = np.full(mb, -1, dtype=np.int32)
        root[:n_pref] = pa.pa_pool_alloc(pool, n_pref)
        shared = []
        for _ in range(B):
            t = root.copy()
            pa.pa_pool_share(pool, t[:n_pref])
            t[n_pref:] = pa.pa_pool_alloc(pool, n_own)
            shared.append(t)
        pa.pa_pool_release(pool, root)  # the forks keep the prefix alive
        unshared = [pa.pa_pool_alloc(pool, mb) for _ in range(B)]
    finally:
        pa.pa_pool_destroy(pool)
    ctx = torch.full((B,), T, dtype=torch.int32, device=dev)
    out = torch.empty((B, hq, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def time_it(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    res = {}
    logical = B * (2 * T * hkv * D * 2 + hq * D * 6)
    for name, tabs in (("shared", shared), ("unshared", unshared)):
        bt = torch.from_numpy(np.stack(tabs)).to(dev)
        ws_bytes = pa.pa_decode_workspace_size(B, hq, hkv, D, 16, mb, 0)
        ws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=dev)
        ms = time_it(lambda: pa.pa_decode(q, kc, vc, bt, ctx, out, 1.0 / D ** 0.5, hq, hkv,
                                          D, 16, B, mb, n_pages, pa.BF16, 0, ws, ws_bytes,
                                          stream.cuda_stream))
        res[name] = {"ms_per_step": round(ms, 4),
                     "logical_GB_s": round(logical / (ms * 1e-3) / 1e9, 1)}
    unique = (n_pref + B * n_own) * hkv * 16 * D * 2 * 2 + B * hq * D * 6
    res["shared"]["unique_bytes"] = unique
    res["shared"]["unique_GB_s"] = round(unique / (res["shared"]["ms_per_step"] * 1e-3) / 1e9, 1)
    # cascade: the forks' queries over the prefix once, then each fork's own
    # tokens, merged (pa_decode_cascade)
    ptab = torch.from_numpy(np.ascontiguousarray(shared[0][:n_pref])).to(dev)
    own_tab = torch.from_numpy(np.stack([t[n_pref:] for t in shared])).to(dev)
    own_ctx = torch.full((B,), suffix, dtype=torch.int32, device=dev)
    cws_bytes = pa.pa_decode_cascade_workspace_size(B, hq, hkv, D, 16, n_pref, prefix, 0)
    cws = torch.empty(max(1, cws_bytes // 4), dtype=torch.float32, device=dev)
    ms = time_it(lambda: pa.pa_decode_cascade(q, kc, vc, ptab, prefix, n_pref, own_tab, own_ctx,
                                              out, 1.0 / D ** 0.5, hq, hkv, D, 16, B, n_own,
                                              n_pages, pa.BF16, 0, cws, cws_bytes,
                                              stream.cuda_stream))
    res["cascade"] = {"ms_per_step": round(ms, 4),
                      "unique_GB_s": round(unique / (ms * 1e-3) / 1e9, 1),
                      "frac_of_hbm_peak": round(unique / (ms * 1e-3) / 1e9 /
                                                peaks.get("hbm_gbs", 6800.0), 4),
                      "speedup_vs_shared_decode": round(res["shared"]["ms_per_step"] / ms, 3),
                      "kernels": "prefill_tc_kernel over the prefix (shared keys, key ranges) + "
                                 "decode_kernel over each fork's own pages + merge_kernel"}
    res["logical_bytes_per_step"] = logical
    res["speedup_vs_unshared"] = round(res["unshared"]["ms_per_step"] /
                                       res["shared"]["ms_per_step"], 3)
    # copy-on-write page copy: 4096 pages (pairs disjoint), K and V
    n_copy = min(4096, n_pages // 2)
    src = torch.arange(n_copy, dtype=torch.int32, device=dev)
    dst = src + n_copy
    ms = time_it(lambda: pa.pa_copy_pages(kc, vc, src, dst, n_copy, hkv, D, 16, n_pages,
                                          pa.BF16, stream.cuda_stream))
    moved = 2 * 2 * n_copy * hkv * 16 * D * 2  # read + write, K and V
    res["copy_pages"] = {"pages": n_copy, "ms": round(ms, 4),
                         "GB_s": round(moved / (ms * 1e-3) / 1e9, 1),
                         "frac_of_hbm_peak": round(moved / (ms * 1e-3) / 1e9 /
                                                   peaks.get("hbm_gbs", 6800.0), 4)}
    assert pa.pa_last_device_error() == 0
    res["config"] = f"B={B}, prefix {prefix} shared + {suffix} own tokens, 32/8 heads, D 128, bf16"
    del kc, vc, q, out
    torch.cuda.empty_cache()
    return res


def run_topm(torch, pa, steps, warmup, peaks, L=32, H=32, N=32768):
    """Budgeted global top-M KV retention at the LLaMA-7B shape (32 layers x
    32 heads x 32768 tokens = 33.5M scores), budget a quarter of the rows,
    scores on a 1/16 grid (heavy ties).  Algorithmic bytes = the scores read
    once + the uint8 mask written; the select streams the scores once in
    full (the pass that writes the mask and lists the threshold bucket's
    candidates, on a first digit taken from every 32nd chunk and confirmed by
    that pass's counts) and reads one chunk again for the tie rank."""
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev).manual_seed(1009)
    scores = (torch.randn(L, H, N, generator=g, device=dev) * 16).round() / 16
    keep = torch.empty((L, H, N), dtype=torch.uint8, device=dev)
    per_head = torch.empty((L, H), dtype=torch.int32, device=dev)
    ws_bytes = pa.pa_topm_workspace_size(L, H, N)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.int32, device=dev)
    budget = L * H * N // 4
    stream = torch.cuda.current_stream()

    def once():
        pa.pa_topm_retain(scores, L, H, N, N - 1, budget, keep, per_head, ws, ws_bytes,
                          stream.cuda_stream)

    for _ in range(warmup):
        once()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        once()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    assert pa.pa_last_device_error() == 0 and int(keep.sum()) == budget
    n = L * H * N
    algo = n * 4 + n
    res = {"ms": round(ms, 4), "elements": n, "Gelem_s": round(n / (ms * 1e-3) / 1e9, 2),
           "algorithmic_GB_s": round(algo / (ms * 1e-3) / 1e9, 1),
           "frac_of_hbm_peak": round(algo / (ms * 1e-3) / 1e9 / peaks.get("hbm_gbs", 6800.0), 4),
           "score_passes": 1 + 1 / 32, "budget": budget,
           "config": f"{L} layers x {H} heads x {N} tokens, budget 1/4, scores on a 1/16 grid",
           "l2": "134 MB of scores (above L2); steps timed back to back"}
    del scores, keep
    torch.cuda.empty_cache()
    return res


def cpu_baseline_sample(torch, case, cfg, layers_budget_s=10.0):
    """The float64 oracle, as it stands, on whole layers of a decode
    workload (every sequence and head of the layer) until ~budget seconds
    pass (at least one layer)."""
    import oracle
    from workloads import compact_host_copy  # re-indexing only
    B = case.q.shape[1]
    hq, hkv, D = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    threads = oracle.max_threads()
    done_layers, bytes_done, t_total = 0, 0, 0.0
    for layer in range(case.layers):
        q, k, v, table, ctx = compact_host_copy(case, layer, list(range(B)))
        t = time.perf_counter()
        oracle.decode(q, k, v, table, ctx, case.scale, case.dtype_code, n_threads=threads)
        t_total += time.perf_counter() - t
        done_layers += 1
        bytes_done += decode_bytes([int(x) for x in ctx], hq, hkv, D)
        if t_total >= layers_budget_s:
            break
    return {"value": round(bytes_done / t_total / 1e9, 3), "unit": "GB/s",
            "cores": threads, "kind": "oracle",
            "sample": f"{done_layers} of {case.layers} layers x {B} sequences "
                      f"(all heads, every cached token), float64, OpenMP",
            "seconds": round(t_total, 2)}


def describe(name, cfg):
    """One line naming a decode workload by what it is."""
    ctx = cfg["ctx"]
    ctx_s = (f"context ~ U[{ctx[0]}, {ctx[1]}] seeded" if isinstance(ctx, tuple)
             else f"context {ctx}")
    pool = (f"shuffled pool of {cfg['pool_pages']} pages" if cfg.get("pool_pages")
            else "random block tables")
    qm = f", Q x {cfg['q_mul']:g}" if cfg.get("q_mul", 1.0) != 1.0 else ""
    return (f"{name}: decode step of {cfg['layers']} layers (per layer the step token's K/V "
            f"write, then attention over every cached token), "
            f"batch {cfg['batch']}, {cfg['n_q_heads']} q heads / {cfg['n_kv_heads']} kv "
            f"heads, head_dim {cfg['head_dim']}, {ctx_s}, {cfg['dtype']} KV, page_size "
            f"{cfg['page_size']}, {pool}{qm}")


def step_block(r, args, world, peaks, peaks_src):
    """value, roofline and e2e of one measured decode step (run_decode_step)."""
    ms_step = r["ms"] / args.steps
    value = whole_job_gbs(world, r["step_bytes"], ms_step)
    seq_layers = world * r["L"] * r["B"] / (ms_step * 1e-3)
    # The timed region is L decode launches per step, back to back (plus, for
    # split plans, one 1-CTA counter clear per launch that overlaps it under
    # programmatic dependent launch): its time over those launches is the
    # kernel's average launch duration.  Events around each call stop that
    # overlap, so that figure is reported apart.
    launch_ms = r["ms"] / (args.steps * r["L"])
    call_gbs = r["per_layer_bytes"] / (launch_ms * 1e-3) / 1e9
    isolated_gbs = r["per_layer_bytes"] / (r["call_avg_ms"] * 1e-3) / 1e9
    e2e_ms_step = r["e2e_ms"] / args.steps
    hbm = peaks.get("hbm_gbs", 6800.0)
    tr = traffic_record(r["name"])
    cfg = r["cfg"]
    return {
        "value": round(value, 1), "unit": "GB/s", "ms_per_step": round(ms_step, 4),
        "dtype": "f32",
        "data": f"synthetic (seeded N(0,1), rounded to {cfg['dtype']})",
        "config": {
            "workload": describe(r["name"], cfg),
            "kv_dtype": cfg["dtype"], "accumulate": "f32", "out_dtype": "f32",
            "partition_tokens": r["part"],
            "l2": f"inputs larger than L2 ({r['step_bytes'] / 1e9:.1f} GB of KV per step "
                  "vs 129 MB); no flush",
            "bytes_per_step": r["step_bytes"],
            "context_tokens_per_layer": sum(r["ctx_list"]),
        },
        "seq_layers_per_s": round(seq_layers, 1),
        "frac_of_hbm_peak": round(value / world / hbm, 4),
        "roofline": {"bound": "hbm", "achieved": round(call_gbs, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(call_gbs / hbm, 4),
                     "traffic": tr["dram_bytes_per_launch"] if tr else None,
                     "peak_source": f"{peaks_src} hbm_gbs (copy)",
                     "kernel": "pa_decode_append call (decode_kernel with the step's K/V "
                               "write; split plans merge in the last CTA of each head group)",
                     "algorithmic_bytes_per_launch": r["per_layer_bytes"],
                     "avg_launch_ms": round(launch_ms, 5),
                     "avg_launch_ms_from": "timed region / decode launches in it",
                     "isolated_call_ms": round(r["call_avg_ms"], 5),
                     "isolated_call_frac": round(isolated_gbs / hbm, 4),
                     "traffic_capture": tr["capture"] if tr else None},
        "e2e": {"value": round(whole_job_gbs(world, r["step_bytes"], e2e_ms_step), 1),
                "unit": "GB/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "ms_per_step": round(e2e_ms_step, 4)},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "append_then_decode": {
            "ms_per_step": round(r["two_call_ms"], 4),
            "value": round(whole_job_gbs(world, r["step_bytes"], r["two_call_ms"]), 1),
            "unit": "GB/s", "calls": "pa_append_kv + pa_decode per layer"},
    }


# ---------------------------------------------------------------------------

def barrier(torch, world):
    if world > 1:
        torch.distributed.barrier()


def allreduce_max(torch, world, x):
    """The maximum of x over the ranks (the slowest rank's time)."""
    if world <= 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, bytes_per_rank_step, ms_step_max):
    """Whole-job throughput of a replicated step: every rank moves the same
    bytes, and the job takes as long as its slowest rank."""
    return world * bytes_per_rank_step / (ms_step_max * 1e-3) / 1e9


def init_dist(torch, args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return rank, world


def main_ours(args):
    import torch
    import paged_kv_cache_171_gb300 as pa
    from paged_kv_cache_171_gb300 import build as pa_build
    import workloads

    pa_build.build()
    rank, world = init_dist(torch, args)
    peaks, peaks_src = measured_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    if args.only_second:  # the LLaMA-7B-shaped step alone (profiling runs)
        r2 = run_decode_step(torch, pa, workloads, SECOND, args, rank, world)
        blk2 = step_block(r2, args, world, peaks, peaks_src)
        if rank == 0:
            print(json.dumps({"workload": SECOND, "block": blk2}), flush=True)
        return
    r = run_decode_step(torch, pa, workloads, HEADLINE, args, rank, world)
    blk = step_block(r, args, world, peaks, peaks_src)
    line = {"metric": METRIC, "value": blk.pop("value"), "unit": blk.pop("unit"),
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": blk.pop("ms_per_step"), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None}
    line.update(blk)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(torch, r["case"], r["cfg"])
    del r
    torch.cuda.empty_cache()
    if not args.only_headline:
        # the LLaMA-7B-shaped step, measured the same way (a block of its own)
        r2 = run_decode_step(torch, pa, workloads, SECOND, args, rank, world)
        blk2 = step_block(r2, args, world, peaks, peaks_src)
        blk2["steps"], blk2["warmup"] = args.steps, args.warmup
        if rank == 0 and not args.no_cpu_baseline:
            blk2["cpu_baseline"] = cpu_baseline_sample(torch, r2["case"], r2["cfg"])
        line["second_workload"] = blk2
        del r2
        torch.cuda.empty_cache()
        other = {}
        other["gqa8_b4_ctx32k"] = run_other_decode(torch, pa, workloads,
                                                   "gqa8_b4_ctx32k", 20, 5, 512)
        other["mha_b1_ctx512"] = run_other_decode(torch, pa, workloads,
                                                  "mha_b1_ctx512", 20, 5)
        other["prefill_b4_512over8192"] = run_prefill(torch, pa, workloads, 10, 3, peaks)
        other["verify_gamma4_b4_ctx32k"] = run_verify(torch, pa, workloads, 20, 3, peaks)
        other["window_sink4_w4096_b32_ctx32k"] = run_window(torch, pa, workloads, 20, 3, peaks)
        other["prefix_shared_b32_8192p128s"] = run_prefix_sharing(torch, pa, 20, 3, peaks)
        other["topm_retain_l32h32n32k"] = run_topm(torch, pa, 10, 3, peaks)
        for k, v in other.items():
            if "GB_s" in v:
                v["frac_of_hbm_peak"] = round(v["GB_s"] / hbm, 4)
        line["other_workloads"] = other
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main_reference(args):
    """The float64 oracle as the reference arm, on the host cores: the
    headline workload, one whole layer (every sequence and head) per step."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import workloads
    cfg = workloads.CONFIGS[HEADLINE]
    B, hq, hkv, D = cfg["batch"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    # the same sequences (same seed, same drawn lengths), one layer, on the host
    case = workloads.paged_case(**{**cfg, "layers": 1, "pool_pages": None})
    threads = oracle.max_threads()
    ctx = [int(t) for t in case.ctx_lens]
    per_layer = decode_bytes(ctx, hq, hkv, D)

    def step():
        oracle.decode(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                      case.ctx_lens, case.scale, case.dtype_code, n_threads=threads)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    sec = time.perf_counter() - t
    ms = sec * 1e3 / args.steps
    gbs = per_layer / (ms * 1e-3) / 1e9
    sample = (f"one of {cfg['layers']} layers per step: {B} sequences x {hq} heads, "
              f"{sum(ctx)} cached tokens (the oracle's decode)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic (seeded N(0,1), {cfg['dtype']})",
        "config": {"workload": describe(HEADLINE, cfg) + "; one layer per step, float64 "
                                                         "oracle"},
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ncu_case(args):
    """A small launch sequence for ncu captures: one layer of a decode
    workload (the ragged GQA batch: 1.1 GB of KV; the LLaMA-shaped one: 537
    MB; both above L2) decoded `--steps` times after `--warmup` calls, or one
    of the other kernels' workloads.  Prints nothing to measure."""
    import torch
    import paged_kv_cache_171_gb300 as pa
    from paged_kv_cache_171_gb300 import build as pa_build
    import workloads
    pa_build.build()
    torch.cuda.set_device(0)
    if args.ncu_case == "prefill":
        case = workloads.config_case("prefill_b4_512over8192", device="cuda")
        for _ in range(args.warmup + args.steps):
            pa.prefill(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                       case.ctx_lens, case.scale)
    elif args.ncu_case == "verify":  # 4 x 32768 cached + 4 drafted, 64/8 heads
        case = workloads.paged_case(layers=1, batch=4, n_q_heads=64, n_kv_heads=8,
                                    head_dim=128, page_size=16, ctx=[32768] * 4, dtype="bf16",
                                    seed=1006, n_new=4, kind="prefill", device="cuda")
        for _ in range(args.warmup + args.steps):
            pa.prefill_split(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                             case.ctx_lens, case.scale)
    elif args.ncu_case == "window":  # 16 x 32768, 64/8 heads, 4 sink + 4096 window
        case = workloads.paged_case(layers=1, batch=16, n_q_heads=64, n_kv_heads=8,
                                    head_dim=128, page_size=16, ctx=[32768] * 16, dtype="bf16",
                                    seed=1007, device="cuda")
        for _ in range(args.warmup + args.steps):
            pa.decode_window(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                             case.ctx_lens, case.scale, 4, 4096)
    elif args.ncu_case == "topm":  # 32 x 32 x 32768 scores on a 1/16 grid, budget 1/4
        g = torch.Generator(device="cuda").manual_seed(1009)
        sc = (torch.randn(32, 32, 32768, generator=g, device="cuda") * 16).round() / 16
        for _ in range(args.warmup + args.steps):
            pa.topm_retain(sc, 32767, 32 * 32 * 32768 // 4)
    elif args.ncu_case == "cascade":  # 32 forks of an 8192-token prefix + 128 own tokens
        B, hq, hkv, D, prefix, suffix = 32, 32, 8, 128, 8192, 128
        n_pref, n_own = prefix // 16, suffix // 16
        g = torch.Generator(device="cuda").manual_seed(1008)
        pages = n_pref + B * n_own
        kc = torch.randn(pages, hkv, 16, D, generator=g, device="cuda").to(torch.bfloat16)
        vc = torch.randn(pages, hkv, 16, D, generator=g, device="cuda").to(torch.bfloat16)
        q = torch.randn(B, hq, D, generator=g, device="cuda").to(torch.bfloat16)
        ptab = torch.arange(n_pref, dtype=torch.int32, device="cuda")
        own = (n_pref + torch.arange(B * n_own, dtype=torch.int32, device="cuda")).view(B, n_own)
        own_ctx = torch.full((B,), suffix, dtype=torch.int32, device="cuda")
        for _ in range(args.warmup + args.steps):
            pa.decode_cascade(q, kc, vc, ptab, prefix, own, own_ctx, 1.0 / math.sqrt(D))
    elif args.ncu_case == "copy_pages":  # 4096 page pairs, 8 kv heads, D 128, bf16
        kc = torch.zeros(8192, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        src = torch.arange(4096, dtype=torch.int32, device="cuda")
        dst = src + 4096
        for _ in range(args.warmup + args.steps):
            pa.pa_copy_pages(kc, vc, src, dst, 4096, 8, 128, 16, 8192, pa.BF16)
    else:
        name = {"decode": "llama7b_b8_ctx4096", "decode_gqa8": "gqa8_b4_ctx32k",
                "decode_gqa4": "gqa4_b64_ragged", "decode_mha_small": "mha_b1_ctx512"}[
                    args.ncu_case]
        over = {"layers": 1, "pool_pages": None}
        case = workloads.config_case(name, device="cuda", **over)
        cfg = workloads.CONFIGS[name]
        part = cfg.get("partition_tokens", 0)
        step = name in (HEADLINE, SECOND)  # the decode steps' call: the fused append
        if step:
            B = case.q.shape[1]
            k_new, v_new = workloads.new_tokens(B, cfg["n_kv_heads"], cfg["head_dim"],
                                                cfg["dtype"], seed=cfg["seed"] + 1,
                                                device="cuda")
        for _ in range(args.warmup + args.steps):
            if step:
                pa.decode_append(case.q[0], k_new, v_new, case.k_cache, case.v_cache,
                                 case.block_table[0], case.ctx_lens, case.scale,
                                 partition_tokens=part)
            else:
                pa.decode(case.q[0], case.k_cache, case.v_cache, case.block_table[0],
                          case.ctx_lens, case.scale, partition_tokens=part)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error() == 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only-second", action="store_true",
                    help="run only the LLaMA-7B-shaped decode step (for profiling)")
    ap.add_argument("--only-headline", action="store_true",
                    help="skip the second decode step and the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-case", choices=["decode", "decode_gqa8", "decode_gqa4",
                                           "decode_mha_small", "verify", "window", "topm",
                                           "copy_pages", "prefill", "cascade"],
                    help="run a small launch sequence for an ncu capture and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.ncu_case:
        ncu_case(args)
    elif args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)


if __name__ == "__main__":
    main()
