#!/usr/bin/env python
"""Throughput of the exact-attention hot path on GB300; prints one JSON line.

One step = the whole hot path over one batch of synthetic input:
  attn_fwd (BF16) -> attn_bwd (D pre-kernel, main kernel, dQ convert)
  -> attn_quantize_fp8 of Q, K (random-sign Hadamard) and V -> attn_fwd_fp8.
FLOPs per step follow the paper's metric (FlashAttention-3, zenmind.me summary
§7.1): forward 4 B H N^2 d (halved when causal), backward 2.5x forward, so a
step counts 4.5x the forward FLOPs (the quantiser adds no FLOPs).

Default workload: the BF16 sweep point d=128, H=16, N=8192, B=2 (B*N = 16384
tokens), non-causal, Q/K/V/dO i.i.d. N(0,1). Every kernel's inputs exceed the
129 MB L2, so no flush is needed between steps.

Sliding-window workloads (name starting "window_") time a step of
attn_fwd_window + attn_bwd_window (BF16) instead; their FLOPs count only the
visible (query, key) pairs: 4 B H d * pairs forward, 2.5x that backward.

Decode workloads (name starting "decode_") time attn_decode_fp8, one new
token per sequence over a resident block-quantised FP8 KV cache; the metric is
cache bytes read per second (HBM-bound), with the measured copy bandwidth as
the roofline peak.

--impl reference times the float64 CPU oracle on a bounded sample of the same
workload (one head per step) in the same units.
Under torchrun every rank runs the same workload on its own GPU (replicas, no
collective on the data path); value = all ranks' FLOPs / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: (B, Hq, Hkv, N, d, causal, window)
    "bf16_sweep_d128_n8192": (2, 16, 16, 8192, 128, False, None),
    "bf16_sweep_d128_n8192_causal": (2, 16, 16, 8192, 128, True, None),
    "gqa_b2_hq32_hkv8_n8192_causal": (2, 32, 8, 8192, 128, True, None),
    # same token count as the default, shorter rows: the size used for ncu --set full captures
    "bf16_b4_h16_n4096": (4, 16, 16, 4096, 128, False, None),
    # other points of the BF16 sweep (B*N = 16384 tokens): the memory-bound short rows and head dim 64
    "bf16_sweep_d128_n512": (32, 16, 16, 512, 128, False, None),
    "bf16_sweep_d64_n8192": (2, 32, 32, 8192, 64, False, None),
    "bf16_sweep_d256_n8192": (2, 8, 8, 8192, 256, False, None),
    # sliding window: each query sees itself and the 1024 keys before it
    "window_b1_h16_n16384_w1024": (1, 16, 16, 16384, 128, False, (1024, 0)),
}
DEFAULT = "bf16_sweep_d128_n8192"
DECODE_WORKLOADS = {
    # name: (B, Hq, Hkv, Nmax, d, splits): an FP8 cache of 2 * B * Hkv * Nmax * d bytes, GQA groups of 4
    "decode_fp8_b16_hq32_hkv8_n32768_d128": (16, 32, 8, 32768, 128, 8),
    # a quarter of it (268 MB of cache, still above L2): the size used for ncu --set full
    "decode_fp8_b4_hq32_hkv8_n32768_d128": (4, 32, 8, 32768, 128, 8),
}
VARLEN_WORKLOADS = {
    # name: (lengths seed, sequences, Hq, Hkv, d): packed causal BF16 forward + backward,
    # 8 sequences of 1k..32k tokens (T = 129511), GQA groups of 4
    "varlen_t129511_hq32_hkv8_d128_causal": (18, 8, 32, 8, 128),
}


def bwd_launches(B, Hq, Hkv, N, d, causal, window, sms):
    """Kernels one dense attn_bwd call launches: D and the dQ clearing, the
    main kernel, the dQ conversion, plus a second main-kernel launch when the
    library splits the last wave (no mask, the units of the last wave at most
    half the SMs and more than one wave's worth of work before them)."""
    if causal or window is not None:
        return 3
    units = -(-N // 128) * (2 if d == 256 else 1) * Hkv * B
    tail = units % sms
    split = sms >= 2 and 0 < tail and 2 * tail <= sms and (Hq // Hkv) * -(-N // 64) >= 2
    return 4 if split and units > tail else 3


def launches_per_step(B, Hq, Hkv, N, d, causal, window, sms):
    """fwd 1, bwd 3 or 4, quantise 3, fp8 fwd 1 (window: fwd 1, bwd 3 or 4)"""
    nb = bwd_launches(B, Hq, Hkv, N, d, causal, window, sms)
    return 1 + nb if window is not None else 1 + nb + 3 + 1


# The FP8 accuracy configuration, timed on its own inputs after the step:
# B=4, H=16, N=8192, d=128, N(0,1) with 0.1 % of entries replaced by
# N(0, 10^2) (seed 3), Q and K rotated with the random signs of seed 4.
FP8_CONFIG = (4, 16, 8192, 128)


def visible_pairs(N, left, right):
    """Number of (query i, key j) pairs with i - left <= j <= i + right (-1: no bound)."""
    total = 0
    for i in range(N):
        lo = 0 if left < 0 else max(0, i - left)
        hi = N - 1 if right < 0 else min(N - 1, i + right)
        total += hi - lo + 1
    return total


def fwd_flops(B, Hq, N, d, causal, window=None):
    if window is not None:
        return 4.0 * B * Hq * d * visible_pairs(N, *window)
    f = 4.0 * B * Hq * N * N * d
    return f / 2 if causal else f


def max_over_ranks(values, world, device="cpu"):
    """Elementwise maximum of a list of floats over all ranks (the job's time)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64)
    if world > 1:
        import torch.distributed as dist
        t = t.to(device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        t = t.cpu()
    return [float(x) for x in t]


def job_tflops(step_flops, steps, world, ms):
    """Whole-job throughput: every rank ran `steps` steps of `step_flops`; the
    job took the slowest rank's `ms`."""
    return world * step_flops * steps / (ms * 1e-3) / 1e12


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return {"bf16_burst": m["bf16_tflops"], "bf16_sustained": m.get("bf16_tflops_sustained"),
                "hbm_gbs": m["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def sm_count():
    import torch
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons. The sampler is
    started before the warm-up (its start-up competes with the first launches
    for the CPU and the driver, which would stretch a short timed region) and
    only the samples taken inside the timed regions (begin/end) are kept."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None
        self.out = None
        self.windows = []
        self._t = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def begin(self):
        self._t = time.time()

    def end(self):
        if self._t is not None:
            self.windows.append((self._t, time.time()))
            self._t = None

    def stop(self):
        if self.proc is None:
            if self.out is not None:
                self.out.close()
                os.unlink(self.path)
            return None
        # a run shorter than the sampler's start-up would leave no row at all:
        # wait (at most 3 s) for the first one
        t_end = time.time() + 3.0
        while time.time() < t_end and self.proc.poll() is None:
            self.out.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)
        return parse_clock_samples(text, self.windows)


def parse_clock_samples(text, windows=None):
    """Median SM clock, the largest max clock and the throttle reasons seen in
    nvidia-smi CSV rows (the fields of Clocks.Q without the leading timestamp,
    or with it). With `windows` (wall-clock (start, end) pairs) and timestamped
    rows, only the rows inside a window count (all rows if none does)."""
    import datetime
    rows = [[f.strip() for f in r.split(",")] for r in text.strip().splitlines() if r.strip()]
    if not rows:
        return None
    stamped = []
    for r in rows:
        t = None
        if "/" in r[0]:
            try:
                t = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = None
            r = r[1:]
        stamped.append((t, r))
    if windows:
        inside = [r for t, r in stamped if t is not None and any(a - 0.05 <= t <= b + 0.05 for a, b in windows)]
        rows = inside or [r for _, r in stamped]
    else:
        rows = [r for _, r in stamped]
    sm = [float(r[1]) for r in rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
    mx = [float(r[2]) for r in rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v and "Not" not in v})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(rows)}


def make_inputs(wl, device):
    import torch
    from exact_attention_73_gb300 import inputs
    B, Hq, Hkv, N, d, causal, window = wl
    q, k, v, do = inputs.normal(1, [(B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, Hq, N, d)])
    signs = inputs.random_signs(4, d)
    return [x.to(device) for x in (q, k, v, do)] + [signs.to(device)]


def bench_ours(args, wl, rank, world):
    import torch
    from exact_attention_73_gb300 import binding as L

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    L.load(build_if_missing=True)
    B, Hq, Hkv, N, d, causal, window = wl
    nb = (N + 127) // 128
    q, k, v, do, signs = make_inputs(wl, dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((L.attn_bwd_workspace_size(B, Hq, Hkv, N, d),), dtype=torch.uint8, device=dev)
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=dev)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    v8 = torch.empty(v.shape, dtype=torch.uint8, device=dev)
    sq = torch.empty((B, Hq, nb), device=dev)
    sk = torch.empty((B, Hkv, nb), device=dev)
    sv = torch.empty((B, Hkv, nb), device=dev)
    o8 = torch.empty_like(q)
    lse8 = torch.empty_like(lse)
    stream = torch.cuda.current_stream(dev)
    ev = None

    # one set of step inputs and results (the e2e loop uses a second set)
    set0 = {"in": [q, k, v, do], "out": [o, lse, dq, dk, dv, o8, lse8]}

    def run(bs, marks=None):
        q_, k_, v_, do_ = bs["in"]
        o_, lse_, dq_, dk_, dv_, o8_, lse8_ = bs["out"]
        if marks is not None:
            marks[0].record(stream)
        if window is not None:
            L.attn_fwd_window(q_, k_, v_, o_, lse_, window)
        else:
            L.attn_fwd(q_, k_, v_, o_, lse_, causal=causal)
        if marks is not None:
            marks[1].record(stream)
        if window is not None:
            L.attn_bwd_window(q_, k_, v_, o_, lse_, do_, dq_, dk_, dv_, ws, window)
        else:
            L.attn_bwd(q_, k_, v_, o_, lse_, do_, dq_, dk_, dv_, ws, causal=causal)
        if marks is not None:
            marks[2].record(stream)
        if window is not None:      # the FP8 path has no window: BF16 forward + backward only
            if marks is not None:
                marks[3].record(stream)
                marks[4].record(stream)
            return
        L.attn_quantize_fp8(q_, q8, sq, signs)
        L.attn_quantize_fp8(k_, k8, sk, signs)
        L.attn_quantize_fp8(v_, v8, sv)
        if marks is not None:
            marks[3].record(stream)
        L.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o8_, lse8_, causal=causal)
        if marks is not None:
            marks[4].record(stream)

    def step(marks=None):
        run(set0, marks)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = Clocks(dev.index)
    clocks.start()
    for _ in range(args.warmup):
        step()
    status = L.attn_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {L.attn_status_string(status)} after warm-up")

    # ---------------------------------------------------------- device-timed
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    barrier()
    clocks.begin()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(args.steps):
        step(marks[s])
    t1.record(stream)
    barrier()
    clocks.end()
    ms_total = t0.elapsed_time(t1)
    stage = {n: sum(m[i].elapsed_time(m[i + 1]) for m in marks) / args.steps
             for i, n in enumerate(("fwd", "bwd", "quant", "fwd_fp8"))}
    if L.attn_get_device_status() != 0:
        raise RuntimeError("device-side wait timed out during the timed region")

    # --------------------------------------------------------------- e2e
    # Through the public API with host memory: every step copies its inputs
    # (Q, K, V, dO) from pinned host memory and reads back all its results.
    # Steps are pipelined over two buffer sets: the H2D copies of step s+1 and
    # the D2H copies of step s-1 run on their own streams while step s computes.
    sets = [set0, {"in": [torch.empty_like(x) for x in set0["in"]],
                   "out": [torch.empty_like(x) for x in set0["out"]]}]
    pin = [x.cpu().pin_memory() for x in set0["in"]]
    n_out = 5 if window is not None else 7            # a window step produces no FP8 results
    host_out = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in bs["out"][:n_out]] for bs in sets]
    h2d = sum(x.numel() * x.element_size() for x in pin)
    d2h = sum(x.numel() * x.element_size() for x in host_out[0])
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e(nsteps, start_event):
        s_h2d.wait_event(start_event)
        for n in range(nsteps):
            b = n % 2
            bs = sets[b]
            with torch.cuda.stream(s_h2d):
                if n >= 2:
                    s_h2d.wait_event(ev_done[b])          # step n-2 has finished with set b
                for dst, src in zip(bs["in"], pin):
                    dst.copy_(src, non_blocking=True)
                ev_in[b].record(s_h2d)
            stream.wait_event(ev_in[b])
            if n >= 2:
                stream.wait_event(ev_out[b])              # results of step n-2 are on the host
            run(bs)
            ev_done[b].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[b])
                for dst, src in zip(host_out[b], bs["out"]):
                    dst.copy_(src, non_blocking=True)
                ev_out[b].record(s_d2h)
        for n in range(max(0, nsteps - 2), nsteps):
            stream.wait_event(ev_out[n % 2])

    w0 = torch.cuda.Event()
    w0.record(stream)
    e2e(2, w0)                                            # warm the copy path
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.begin()
    e0.record(stream)
    e2e(args.steps, e0)
    e1.record(stream)
    barrier()
    clocks.end()
    ms_e2e = e0.elapsed_time(e1)
    if L.attn_get_device_status() != 0:
        raise RuntimeError("device-side wait timed out during the end-to-end run")

    fp8cfg = None
    if window is None:
        fp8cfg = time_fp8_config(L, dev, stream, args.steps, barrier, clocks)
    clk = clocks.stop()
    ms_total, ms_e2e = max_over_ranks([ms_total, ms_e2e], world, dev)
    return {"ms_total": ms_total, "ms_e2e": ms_e2e, "stage_ms": stage, "clocks": clk,
            "h2d": h2d, "d2h": d2h, "fp8_config": fp8cfg}


def time_fp8_config(L, dev, stream, steps, barrier, clocks):
    """attn_fwd_fp8 on the FP8 accuracy configuration's own inputs (FP8_CONFIG:
    outliers, Q and K rotated; the GPU quantiser runs first, untimed), non-causal
    and causal, `steps` launches each after 3 warm-up launches. Each launch
    reads 201 MB of codes and writes 134 MB of O (above L2, no flush).
    Returns {causal flag: ms per launch}."""
    import torch
    from exact_attention_73_gb300 import inputs
    B, H, N, d = FP8_CONFIG
    nb = (N + 127) // 128
    q, k, v = (x.to(dev) for x in inputs.outliers(3, [(B, H, N, d)] * 3))
    signs = inputs.random_signs(4, d).to(dev)
    codes = []
    for x, sg in ((q, signs), (k, signs), (v, None)):
        x8 = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        sc = torch.empty((B, H, nb), device=dev)
        L.attn_quantize_fp8(x, x8, sc, sg)
        codes += [x8, sc]
    del q, k, v
    q8, sq, k8, sk, v8, sv = codes
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), device=dev)
    out = {}
    for causal in (False, True):
        for _ in range(3):
            L.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, causal=causal)
        barrier()
        clocks.begin()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            L.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, causal=causal)
        e1.record(stream)
        barrier()
        clocks.end()
        out[causal] = e0.elapsed_time(e1) / steps
    if L.attn_get_device_status() != 0:
        raise RuntimeError("device-side wait timed out during the FP8 configuration run")
    return out


def cpu_sample(wl, steps=1):
    """The oracle, as it stands, on one head of the workload: forward, backward
    and the FP8 emulation (block quantisation with the rotation). Returns
    (FLOPs processed, seconds)."""
    import numpy as np
    from oracle import attention as A
    from oracle import fp8 as F
    from exact_attention_73_gb300 import inputs
    B, Hq, Hkv, N, d, causal, window = wl
    q, k, v, do = inputs.normal(1, [(1, 1, N, d)] * 4)
    signs = inputs.random_signs(4, d).numpy()
    sc = d ** -0.5
    t = time.perf_counter()
    for _ in range(steps):
        A.forward(q, k, v, sc, causal, window)
        A.backward(q, k, v, do, sc, causal, window)
        if window is not None:
            continue
        q8, sq = F.quantize_blocks(q, signs)
        k8, sk = F.quantize_blocks(k, signs)
        v8, sv = F.quantize_blocks(v)
        F.attention_fp8(q8, k8, v8, sq, sk, sv, sc, causal)
    dt = time.perf_counter() - t
    per_step = (3.5 if window is not None else 4.5) * fwd_flops(1, 1, N, d, causal, window)
    return per_step * steps, dt


def bench_decode(args, wl, rank, world):
    """Time attn_decode_fp8 on a resident cache; returns the JSON line's fields."""
    import numpy as np
    import torch
    from exact_attention_73_gb300 import binding as L
    from exact_attention_73_gb300 import inputs
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    L.load(build_if_missing=True)
    B, Hq, Hkv, N, d, splits = wl
    g = Hq // Hkv
    gen = torch.Generator(device=dev).manual_seed(7)   # the cache is drawn on the device
    q = torch.randn((B, Hq, d), generator=gen, device=dev).to(torch.bfloat16)
    k = torch.randn((B, Hkv, N, d), generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn((B, Hkv, N, d), generator=gen, device=dev).to(torch.bfloat16)
    signs = inputs.random_signs(4, d).to(dev)
    nb = (N + 127) // 128
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    v8 = torch.empty(v.shape, dtype=torch.uint8, device=dev)
    sk = torch.empty((B, Hkv, nb), device=dev)
    sv = torch.empty((B, Hkv, nb), device=dev)
    L.attn_quantize_fp8(k, k8, sk, signs)
    L.attn_quantize_fp8(v, v8, sv)
    q8 = torch.empty((B, Hq, d), dtype=torch.uint8, device=dev)
    sq3 = torch.empty((B, Hkv, 1), device=dev)
    L.attn_quantize_fp8(q.view(B, Hkv, g, d), q8.view(B, Hkv, g, d), sq3, signs)
    sq = sq3[:, :, 0].contiguous()
    del k, v
    o = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq), device=dev)
    ws = torch.empty((L.attn_decode_fp8_workspace_size(B, Hq, d, splits),), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        L.attn_decode_fp8(q8, sq, k8, v8, sk, sv, o, lse, ws, splits)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = Clocks(dev.index)
    clocks.start()
    for _ in range(args.warmup):
        step()
    barrier()
    clocks.begin()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    barrier()
    clocks.end()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    # end to end: the new token's codes and factors in, O and LSE out, every step
    hq8, hsq = q8.cpu().pin_memory(), sq.cpu().pin_memory()
    ho, hl = torch.empty(o.shape, dtype=o.dtype, pin_memory=True), torch.empty(lse.shape, pin_memory=True)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        q8.copy_(hq8, non_blocking=True)
        sq.copy_(hsq, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)
    e1.record(stream)
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    if L.attn_get_device_status() != 0:
        raise RuntimeError("device-side wait timed out during the decode run")
    ms, ms_e2e = max_over_ranks([ms, ms_e2e], world, dev)
    h2d = hq8.numel() + hsq.numel() * 4
    d2h = ho.numel() * 2 + hl.numel() * 4
    cache_bytes = 2 * B * Hkv * N * d + 2 * B * Hkv * nb * 4
    line = {"ms_total": ms, "ms_e2e": ms_e2e, "clocks": clk, "h2d": h2d, "d2h": d2h,
            "bytes": cache_bytes, "flops": 4.0 * B * Hq * N * d}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle is timed on seeded codes of one sequence's cache (its own inputs, same sizes)
        import numpy as np
        rng = np.random.default_rng(7)
        qn = rng.integers(0, 120, (1, Hkv, g, d), dtype=np.uint8)
        kn = rng.integers(0, 120, (1, Hkv, N, d), dtype=np.uint8)
        vn = rng.integers(0, 120, (1, Hkv, N, d), dtype=np.uint8)
        fn = np.ones((1, Hkv, nb), dtype=np.float32)
        t = time.perf_counter()
        from oracle import fp8 as F
        F.decode_fp8(qn, np.ones((1, Hkv), dtype=np.float32), kn, vn, fn, fn, [N], d ** -0.5, -(-nb // splits))
        sec = time.perf_counter() - t
        line["cpu"] = (2 * Hkv * N * d + 2 * Hkv * nb * 4) / sec / 1e9, sec
    return line


def decode_main(args, world, rank):
    import numpy as np
    wl = DECODE_WORKLOADS[args.workload]
    B, Hq, Hkv, N, d, splits = wl
    config = {"workload": args.workload, "B": B, "Hq": Hq, "Hkv": Hkv, "Nmax": N, "d": d, "splits": splits,
              "step": "attn_decode_fp8: one token per sequence over the whole FP8 cache (+ split combine)",
              "l2": f"cache ({2 * B * Hkv * N * d / 2**20:.0f} MiB) larger than L2 (no flush)",
              "parallelism": f"replicas x{world}"}
    metric = "FP8 KV-cache decode: cache bytes read per second on GB300"
    pk = peaks()
    if args.impl == "reference":
        if rank != 0:
            return
        from oracle import fp8 as F
        rng = np.random.default_rng(7)
        g, nb = Hq // Hkv, (N + 127) // 128
        q8 = rng.integers(0, 120, (1, Hkv, g, d), dtype=np.uint8)
        k8 = rng.integers(0, 120, (1, Hkv, N, d), dtype=np.uint8)
        v8 = rng.integers(0, 120, (1, Hkv, N, d), dtype=np.uint8)
        f = np.ones((1, Hkv, nb), dtype=np.float32)
        t = time.perf_counter()
        for _ in range(args.steps):
            F.decode_fp8(q8, np.ones((1, Hkv), dtype=np.float32), k8, v8, f, f, [N], d ** -0.5, -(-nb // splits))
        sec = time.perf_counter() - t
        val = args.steps * (2 * Hkv * N * d + 2 * Hkv * nb * 4) / sec / 1e9
        print(json.dumps({"impl": "reference", "metric": metric, "value": val, "unit": "GB/s", "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": config,
                          "cpu_baseline": {"kind": "oracle", "value": val, "unit": "GB/s", "cores": cpu_cores(),
                                           "sample": "one sequence (b = 0) of the workload per step"},
                          "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = bench_decode(args, wl, rank, world)
    gbs = world * r["bytes"] * args.steps / (r["ms_total"] * 1e-3) / 1e9
    line = {"metric": metric, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms_total"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic", "config": config,
            "tokens_per_s": world * B * args.steps / (r["ms_total"] * 1e-3),
            "roofline": {"bound": "hbm", "kernel": "attn_decode_fp8 (split kernel + combine)",
                         "achieved": gbs / world, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / world / pk["hbm_gbs"], "peak_source": pk["source"] + " copy bandwidth",
                         "traffic": measured_traffic(f"{args.workload}:decode")},
            "e2e": {"value": world * r["bytes"] * args.steps / (r["ms_e2e"] * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": 2 * 2 * args.steps, "clocks": r["clocks"]}   # device-timed and e2e steps
    if "cpu" in r:
        line["cpu_baseline"] = {"value": r["cpu"][0], "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": "one sequence of the workload (seeded E4M3 codes, unit factors): "
                                          f"{r['cpu'][1]:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bench_varlen(args, wl, rank, world):
    """Time attn_fwd_varlen + attn_bwd_varlen (causal, BF16) on resident packed
    inputs; returns the JSON line's fields."""
    import torch
    from exact_attention_73_gb300 import binding as L
    from exact_attention_73_gb300 import inputs
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    L.load(build_if_missing=True)
    seed, nseq, Hq, Hkv, d = wl
    lens = inputs.varlen_lengths(seed, nseq)
    cu = inputs.cu_seqlens(lens).to(dev)
    T, mx = int(sum(lens)), int(max(lens))
    gen = torch.Generator(device=dev).manual_seed(5)   # 2.7 GB of inputs are drawn on the device
    q = torch.randn((T, Hq, d), generator=gen, device=dev).to(torch.bfloat16)
    k = torch.randn((T, Hkv, d), generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn((T, Hkv, d), generator=gen, device=dev).to(torch.bfloat16)
    do = torch.randn((T, Hq, d), generator=gen, device=dev).to(torch.bfloat16)
    o, dq = torch.empty_like(q), torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    lse = torch.empty((Hq, T), device=dev)
    ws = torch.empty((L.attn_bwd_varlen_workspace_size(T, Hq, Hkv, d),), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(m=None):
        if m is not None:
            m[0].record(stream)
        L.attn_fwd_varlen(q, k, v, o, lse, cu, mx, causal=True)
        if m is not None:
            m[1].record(stream)
        L.attn_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, ws, cu, mx, causal=True)
        if m is not None:
            m[2].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = Clocks(dev.index)
    clocks.start()
    for _ in range(args.warmup):
        step()
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier()
    clocks.begin()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s_ in range(args.steps):
        step(marks[s_])
    t1.record(stream)
    barrier()
    clocks.end()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    stage = {n: sum(m[i].elapsed_time(m[i + 1]) for m in marks) / args.steps for i, n in enumerate(("fwd", "bwd"))}
    # end to end: Q, K, V, dO in from pinned host memory and O, LSE, dQ, dK, dV out, every step
    hin = [x.cpu().pin_memory() for x in (q, k, v, do)]
    hout = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (o, lse, dq, dk, dv)]
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        for dst, src in zip((q, k, v, do), hin):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(hout, (o, lse, dq, dk, dv)):
            dst.copy_(src, non_blocking=True)
    e1.record(stream)
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    if L.attn_get_device_status() != 0:
        raise RuntimeError("device-side wait timed out during the varlen run")
    ms, ms_e2e = max_over_ranks([ms, ms_e2e], world, dev)
    fwd_flops = sum(4.0 * Hq * n * n * d / 2 for n in lens)
    line = {"ms_total": ms, "ms_e2e": ms_e2e, "clocks": clk, "stage_ms": stage, "fwd_flops": fwd_flops,
            "h2d": sum(x.numel() * x.element_size() for x in hin),
            "d2h": sum(x.numel() * x.element_size() for x in hout), "lens": lens}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu"] = varlen_cpu_sample(min(lens), d)
    return line


def varlen_cpu_sample(n, d):
    """The oracle's forward and backward on one head of one sequence of n
    tokens (causal): (TFLOP/s, seconds)."""
    from exact_attention_73_gb300 import inputs
    from oracle import attention as A
    q, k, v, do = inputs.normal(5, [(1, 1, n, d)] * 4)
    t = time.perf_counter()
    A.forward(q, k, v, d ** -0.5, True)
    A.backward(q, k, v, do, d ** -0.5, True)
    sec = time.perf_counter() - t
    return 3.5 * 4.0 * n * n * d / 2 / sec / 1e12, sec


def varlen_main(args, world, rank):
    seed, nseq, Hq, Hkv, d = VARLEN_WORKLOADS[args.workload]
    from exact_attention_73_gb300 import inputs
    lens = [int(x) for x in inputs.varlen_lengths(seed, nseq)]
    config = {"workload": args.workload, "lengths": lens, "T": sum(lens), "Hq": Hq, "Hkv": Hkv, "d": d,
              "causal": True, "step": "attn_fwd_varlen + attn_bwd_varlen (BF16, packed [T, H, d])",
              "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}
    metric = "attention fwd+bwd (BF16, packed variable length) TFLOP/s on GB300"
    pk = peaks()
    if args.impl == "reference":
        if rank != 0:
            return
        n = min(lens)
        t = time.perf_counter()
        for _ in range(args.steps):
            varlen_cpu_sample(n, d)
        sec = time.perf_counter() - t
        val = args.steps * 3.5 * 4.0 * n * n * d / 2 / sec / 1e12
        print(json.dumps({"impl": "reference", "metric": metric, "value": val, "unit": "TFLOP/s", "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": config,
                          "cpu_baseline": {"kind": "oracle", "value": val, "unit": "TFLOP/s", "cores": cpu_cores(),
                                           "sample": f"one head of the {n}-token sequence per step"},
                          "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = bench_varlen(args, VARLEN_WORKLOADS[args.workload], rank, world)
    f = r["fwd_flops"]
    value = job_tflops(3.5 * f, args.steps, world, r["ms_total"])
    st = r["stage_ms"]
    line = {"metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms_total"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
            "stages": {"fwd_bf16": {"ms": st["fwd"], "tflops": f / st["fwd"] / 1e9,
                                    "frac_of_bf16_peak": f / st["fwd"] / 1e9 / pk["bf16_burst"]},
                       "bwd_bf16": {"ms": st["bwd"], "tflops": 2.5 * f / st["bwd"] / 1e9,
                                    "frac_of_bf16_peak": 2.5 * f / st["bwd"] / 1e9 / pk["bf16_burst"]}},
            "roofline": {"bound": "tensor", "kernel": "attn_bwd_varlen (main + 2 helpers)",
                         "achieved": 2.5 * f / st["bwd"] / 1e9, "peak": pk["bf16_burst"], "unit": "TFLOP/s",
                         "frac": 2.5 * f / st["bwd"] / 1e9 / pk["bf16_burst"], "peak_source": pk["source"],
                         "traffic": measured_traffic(f"{args.workload}:bwd")},
            "e2e": {"value": job_tflops(3.5 * f, args.steps, world, r["ms_e2e"]), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": 2 * 4 * args.steps, "clocks": r["clocks"]}   # device-timed and e2e steps
    if "cpu" in r:
        line["cpu_baseline"] = {"value": r["cpu"][0], "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": f"one head of the {min(r['lens'])}-token sequence, fwd + bwd: "
                                          f"{r['cpu'][1]:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


SWEEP = [  # (B, H, N, d): the BF16 sweep configuration, B * N = 16384 tokens
    (32, 16, 512, 128), (16, 16, 1024, 128), (8, 16, 2048, 128), (4, 16, 4096, 128), (2, 16, 8192, 128),
    (1, 16, 16384, 128), (2, 32, 8192, 64), (2, 8, 8192, 256)]


def sweep(args):
    """Forward (BF16 and FP8) and, at N = 8192, backward TFLOP/s of every sweep
    point, causal and not: `steps` launches each after 3 warm-up launches,
    CUDA events; inputs drawn on the device (N(0,1), bf16), above L2 at every
    point. Prints one JSON line per point (not the benchmark line)."""
    import torch
    from exact_attention_73_gb300 import binding as L
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L.load(build_if_missing=True)
    stream = torch.cuda.current_stream(dev)
    gen = torch.Generator(device=dev).manual_seed(1)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    for B, H, N, d in SWEEP:
        q, k, v, do = (torch.randn((B, H, N, d), generator=gen, device=dev).to(torch.bfloat16) for _ in range(4))
        o, lse = torch.empty_like(q), torch.empty((B, H, N), device=dev)
        nb = (N + 127) // 128
        codes = []
        for x in (q, k, v):
            x8, sc = torch.empty(x.shape, dtype=torch.uint8, device=dev), torch.empty((B, H, nb), device=dev)
            L.attn_quantize_fp8(x, x8, sc)
            codes += [x8, sc]
        q8, sq, k8, sk, v8, sv = codes
        row = {"B": B, "H": H, "N": N, "d": d}
        for causal in (False, True):
            f = fwd_flops(B, H, N, d, causal)
            tag = "causal" if causal else "non_causal"
            ms = timed(lambda: L.attn_fwd(q, k, v, o, lse, causal=causal))
            row[f"fwd_bf16_{tag}"] = round(f / ms / 1e9, 1)
            ms = timed(lambda: L.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, causal=causal))
            row[f"fwd_fp8_{tag}"] = round(f / ms / 1e9, 1)
            if N == 8192:
                L.attn_fwd(q, k, v, o, lse, causal=causal)
                dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                ws = torch.empty((L.attn_bwd_workspace_size(B, H, H, N, d),), dtype=torch.uint8, device=dev)
                ms = timed(lambda: L.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, causal=causal))
                row[f"bwd_bf16_{tag}"] = round(2.5 * f / ms / 1e9, 1)
        if L.attn_get_device_status() != 0:
            raise RuntimeError("device-side wait timed out during the sweep")
        print(json.dumps(row), flush=True)
        del q, k, v, do, o, lse, codes, q8, sq, k8, sk, v8, sv


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def kernel_source_sha16():
    """Hash of every kernel and launcher source of the library: a DRAM capture
    is valid only for the source it was taken from."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_73_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh")) +
                    glob.glob(os.path.join(csrc, "*.h"))):
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def measured_traffic(key):
    """DRAM bytes (read + write) per launch of one ncu capture (profiles/traffic.json),
    or None when the kernel has no capture or the capture was taken from other
    kernel sources than the current ones."""
    if not os.path.exists(TRAFFIC):
        return None
    t = json.load(open(TRAFFIC))
    e = t.get("launches", {}).get(key)
    if e is None or t.get("source_sha16") != kernel_source_sha16():
        return None
    return e


def write_traffic(csv_path, keys, step_launches, per_step):
    """Write profiles/traffic.json from an ncu --csv launch list holding
    dram__bytes_read.sum and dram__bytes_write.sum: `keys` maps a kernel-name
    regex to the traffic key. The first `step_launches` launches are the
    benchmark steps (before the FP8 configuration's), `per_step` of them per
    step; each key gets the summed bytes of its launches in the last of those
    steps (the backward's main kernel is two launches when its last wave is
    split). Records the current kernel source hash with the numbers."""
    import csv
    import re
    rows = list(csv.reader(l for l in open(csv_path) if l.startswith('"')))
    head = rows[0]
    ki, mi, vi, ui = head.index("Kernel Name"), head.index("Metric Name"), head.index("Metric Value"), \
        head.index("Metric Unit")
    ii = head.index("ID")
    rows = [r for r in rows[1:] if step_launches - per_step <= int(r[ii]) < step_launches]
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    per = {}
    for r in rows:
        for pat, key in keys.items():
            if re.search(pat, r[ki]) and r[mi] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                d = per.setdefault(key, {})
                d[r[mi]] = d.get(r[mi], 0.0) + float(r[vi].replace(",", "")) * scale[r[ui]]
    out = {"source_sha16": kernel_source_sha16(), "capture": os.path.basename(csv_path),
           "launches": {k: int(v["dram__bytes_read.sum"] + v["dram__bytes_write.sum"]) for k, v in per.items()}}
    with open(TRAFFIC, "w") as f:
        json.dump(out, f, indent=1)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(DECODE_WORKLOADS) + sorted(VARLEN_WORKLOADS),
                    default=DEFAULT)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle timing")
    ap.add_argument("--write-traffic", metavar="CSV",
                    help="write profiles/traffic.json from an ncu --csv capture of the default workload's "
                         "dram__bytes_read.sum/dram__bytes_write.sum, then exit")
    ap.add_argument("--sms", type=int, default=152,
                    help="SM count of the GPU the --write-traffic capture ran on")
    ap.add_argument("--sweep", action="store_true",
                    help="time the forward (BF16, FP8) and backward over the sweep points instead, one JSON line "
                         "per point")
    args = ap.parse_args()
    if args.sweep:
        return sweep(args)
    if args.write_traffic:
        # a capture of `bench.py --steps S --warmup W` on a GPU of `--sms` SMs:
        # (W + S + 2 + S) steps come before the FP8 configuration's launches
        steps = args.warmup + args.steps + 2 + args.steps
        B, Hq, Hkv, N, d, causal, window = WORKLOADS[DEFAULT]
        lps = launches_per_step(B, Hq, Hkv, N, d, causal, window, args.sms)
        print(json.dumps(write_traffic(args.write_traffic, {
            r"fwd_kernel<\(?int\)?0|fwd_kernel<0": f"{DEFAULT}:fwd", r"bwd_kernel": f"{DEFAULT}:bwd",
            r"fwd_kernel<\(?int\)?2|fwd_kernel<2": f"{DEFAULT}:fwd_fp8"}, steps * lps, lps)))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.workload in DECODE_WORKLOADS:
        return decode_main(args, world, rank)
    if args.workload in VARLEN_WORKLOADS:
        return varlen_main(args, world, rank)
    wl = WORKLOADS[args.workload]
    B, Hq, Hkv, N, d, causal, window = wl
    config = {"workload": args.workload, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "causal": causal,
              "step": "fwd bf16 + bwd bf16 + fp8 quantise (Q,K rotated) + fwd fp8",
              "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}
    metric = "attention fwd+bwd (BF16) + FP8 fwd TFLOP/s on GB300"
    step_flops = 4.5 * fwd_flops(B, Hq, N, d, causal)
    if window is not None:
        config["window"] = list(window)
        config["step"] = "fwd bf16 + bwd bf16, sliding window (FLOPs of visible pairs only)"
        metric = "attention fwd+bwd (BF16, sliding window) TFLOP/s on GB300"
        step_flops = 3.5 * fwd_flops(B, Hq, N, d, causal, window)

    if args.impl == "reference":
        if rank != 0:
            return
        # the oracle keeps no state between steps, so warm-up steps are not run
        fl, sec = cpu_sample(wl, steps=args.steps)
        val = fl / sec / 1e12
        line = {"impl": "reference", "metric": metric, "value": val, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"kind": "oracle", "value": val, "unit": "TFLOP/s", "cores": cpu_cores(),
                                 "sample": f"one head (b=0,h=0) of the workload per step: fwd + bwd + FP8 emulation"},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = bench_ours(args, wl, rank, world)
    pk = peaks()
    ms_step = r["ms_total"] / args.steps
    value = job_tflops(step_flops, args.steps, world, r["ms_total"])
    e2e_val = job_tflops(step_flops, args.steps, world, r["ms_e2e"])
    st = r["stage_ms"]
    f = fwd_flops(B, Hq, N, d, causal, window)
    stages = {
        "fwd_bf16": {"ms": st["fwd"], "tflops": f / st["fwd"] / 1e9, "frac_of_bf16_peak": f / st["fwd"] / 1e9 / pk["bf16_burst"]},
        "bwd_bf16": {"ms": st["bwd"], "tflops": 2.5 * f / st["bwd"] / 1e9,
                     "frac_of_bf16_peak": 2.5 * f / st["bwd"] / 1e9 / pk["bf16_burst"]},
        "quant_fp8": {"ms": st["quant"], "gbs": ((Hq + 2 * Hkv) * B * N * d * 3) / st["quant"] / 1e6},
        "fwd_fp8": {"ms": st["fwd_fp8"], "tflops": f / st["fwd_fp8"] / 1e9,
                    "frac_of_fp8_peak": f / st["fwd_fp8"] / 1e9 / (2 * pk["bf16_burst"])},
    }
    # dominant kernel: the stage with the longest time (the backward call
    # holds its main kernel plus two HBM-bound helpers of a few percent)
    if window is not None:
        del stages["quant_fp8"], stages["fwd_fp8"]
    dom = max(("fwd", "bwd", "fwd_fp8"), key=lambda n: st[n])
    dom_flops = {"fwd": f, "bwd": 2.5 * f, "fwd_fp8": f}[dom]
    dom_peak = pk["bf16_burst"] * (2 if dom == "fwd_fp8" else 1)
    achieved = dom_flops / st[dom] / 1e9
    traffic = measured_traffic(f"{args.workload}:{dom}")
    line = {
        "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if window is not None else "bf16+e4m3", "data": "synthetic",
        "config": config, "stages": stages,
        "roofline": {"bound": "tensor", "kernel": {"fwd": "attn_fwd", "bwd": "attn_bwd (main kernel, its last wave split into a second launch where that pays, + 2 helpers)",
                                                    "fwd_fp8": "attn_fwd_fp8"}[dom],
                     "achieved": achieved, "peak": dom_peak, "unit": "TFLOP/s", "frac": achieved / dom_peak,
                     "peak_source": pk["source"] + (" bf16 burst x2 (fp8 nominal ratio)" if dom == "fwd_fp8" else " bf16 burst"),
                     "traffic": traffic,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, captured "
                                       "from the current kernel sources" if traffic is not None else
                                       "no ncu capture of the current kernel sources"},
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        # the library's launches inside the timed regions: the device-timed
        # steps and the end-to-end steps (plus the FP8 config's launches below)
        "gpu_launches": 2 * launches_per_step(B, Hq, Hkv, N, d, causal, window, sm_count()) * args.steps,
        "clocks": r["clocks"],
    }
    if r.get("fp8_config"):
        fb, fh, fn, fd = FP8_CONFIG
        ff = fwd_flops(fb, fh, fn, fd, False)
        line["fp8_config"] = {
            "workload": f"fp8_b{fb}_h{fh}_n{fn}_d{fd}_outliers_rotated",
            "kernel": "attn_fwd_fp8", "peak": 2 * pk["bf16_burst"],
            "peak_source": pk["source"] + " bf16 burst x2 (fp8 nominal ratio)",
            **{name: {"ms": ms, "tflops": ff / (2 if c else 1) / ms / 1e9,
                      "frac_of_fp8_peak": ff / (2 if c else 1) / ms / 1e9 / (2 * pk["bf16_burst"])}
               for c, name, ms in ((False, "non_causal", r["fp8_config"][False]),
                                   (True, "causal", r["fp8_config"][True]))}}
        line["gpu_launches"] += 2 * args.steps
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, sec = cpu_sample(wl)
        line["cpu_baseline"] = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": f"one head of the workload (N={N}, d={d}): fwd + bwd + FP8 emulation, "
                                          f"{sec:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
