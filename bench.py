"""Benchmark of the streaming attention forward on one node.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one attention forward over the workload (one call of the library's
C ABI; inputs resident in HBM). The headline times K steps back to back: one
CUDA graph holds all K calls, each call on the next of R copies of the inputs
in rotation, the R copies together several times the L2 size, so no step finds
its inputs in L2; CUDA events on the launching stream bracket the replay.
Separately, a single call is timed cold (graph replay of one call, an L2 flush
by reading a buffer twice the L2 size before each, outside the events): the
latency of one call including its launch. Under torchrun each rank runs the
same per-rank workload (weak scaling, no collective on the data path); the
step time is the maximum over ranks.

``--impl reference`` times the FP64 CPU oracle (the only reference this
project has) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from streaming_attention_gb300.inputs import (  # noqa: E402
    DECODE_GQA, LONG_CAUSAL, PREFILL_D64, PREFILL_D128, WORKLOADS, workload_inputs)

# the D=128 prefill shape in FP16 (same seed and sizes)
FP16_D128 = PREFILL_D128.with_(dtype=torch.float16, name="prefill_b2_h32_4096x4096_d128_fp16_causal")
# the GQA decode shape at head dimension 64 (same seed)
DECODE_D64 = DECODE_GQA.with_(D=64, name="decode_gqa_b8_hq32_hkv8_m1_n8192_w4096_d64_bf16")

METRIC = "attention fwd TFLOP/s (decode: GB/s) and % of GB300 roofline, 1 GPU"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DEFAULT_WORKLOAD = PREFILL_D128.name


# ----------------------------------------------------------------------------
# Work accounting (algorithmic, allowed pairs only)
# ----------------------------------------------------------------------------
def visible_keys(i, M, N, causal, window):
    p = i + N - M
    hi = min(N, p + 1) if causal else N
    lo = max(0, p - window + 1) if window > 0 else 0
    return max(0, hi - lo)


def allowed_pairs(M, N, causal, window):
    if not causal and window <= 0:
        return M * N
    return sum(visible_keys(i, M, N, causal, window) for i in range(M))


def flops(w, causal=None, window=None):
    causal = w.causal if causal is None else causal
    window = w.window if window is None else window
    return 4.0 * w.D * w.B * w.Hq * allowed_pairs(w.M, w.N, causal, window)


def decode_bytes(w, in_bytes=2):
    """Q + O + the K and V rows that any query row may see, each read once
    (Q, K, V of in_bytes per element; O always 16-bit)."""
    lo = max(0, (w.N - w.M) - w.window + 1) if w.window > 0 else 0
    hi = w.N  # the last row sits at position N-1
    kv = 2 * w.B * w.Hkv * (hi - lo) * w.D * in_bytes
    qo = w.B * w.Hq * w.M * w.D * (in_bytes + 2)
    return float(kv + qo)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------
# Distributed helpers (torchrun: one process per GPU)
# ----------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job(work_per_rank, ms_per_step, world, device, scale):
    """(slowest rank's ms per step, whole-job throughput): every rank does the
    same work per step, so the job's rate is world x work over the slowest rank."""
    ms_max = max_over_ranks(ms_per_step, world, device)
    return ms_max, world * work_per_rank / (ms_max * 1e-3) / scale


# ----------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------
def time_calls(fn, steps, warmup, stream, flush):
    """Per-step device time (ms) of fn(stream) with an L2 flush between steps,
    timed with CUDA events on the launching stream."""
    for _ in range(warmup):
        fn(stream)
        flush()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn(stream)
        e.record(stream)
        flush()
        times.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in times]


def capture(fn, warmup):
    """One call of fn captured in a CUDA graph (after warm-up on a side stream)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            fn(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(torch.cuda.current_stream())
    torch.cuda.synchronize()
    return g


def time_steady(step, sets, steps, warmup, stream, replays=1, samples=None):
    """Device time (ms) per step of `steps` calls back to back, call i on input
    set i % len(sets), all captured in one CUDA graph (launches inside a graph
    keep their programmatic overlap); `warmup` untimed calls first. The graph is
    replayed `replays` times, each replay timed on its own; the median replay
    divided by `steps` is returned and the per-replay figures are appended to
    `samples` when given."""

    def seq(n, st):
        for i in range(n):
            step(sets[i % len(sets)], st)

    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        seq(warmup, side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    gw, gk = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(gw):
        seq(warmup, torch.cuda.current_stream())
    with torch.cuda.graph(gk):
        seq(steps, torch.cuda.current_stream())
    torch.cuda.synchronize()
    gw.replay()
    torch.cuda.synchronize()
    evs = []
    for _ in range(max(1, replays)):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        gk.replay()
        e.record(stream)
        evs.append((s, e))
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) / steps for s, e in evs]
    if samples is not None:
        samples.extend(per)
    return statistics.median(per)


def time_eager_steady(step, sets, steps, warmup, stream):
    """As time_steady, but plain C-ABI calls on the stream (no graph)."""
    for i in range(warmup):
        step(sets[i % len(sets)], stream)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for i in range(steps):
        step(sets[i % len(sets)], stream)
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps


def rotation(w, dev, l2_bytes):
    """Device copies of the workload's inputs (and an output each), enough that
    the copies a step does not use fill several times the L2 size."""
    q, k, v = workload_inputs(w)
    per_set = 2 * q.numel() * q.element_size() + 2 * k.numel() * k.element_size()
    r = max(2, min(8, math.ceil(3 * l2_bytes / per_set) + 1))
    sets = []
    for _ in range(r):
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        sets.append((qd, kd, vd, torch.empty_like(qd)))
    return (q, k, v), sets, per_set


def time_graph(fn, steps, warmup, flush):
    """Per-step device time (ms) of the captured call replayed, L2 flushed between replays."""
    g = capture(fn, warmup)
    return time_calls(lambda st: g.replay(), steps, warmup, torch.cuda.current_stream(), flush)


def l2_flusher(dev):
    """Evicts L2 by reading a buffer twice the L2 size. Reading leaves clean
    lines, so the next step pays no write-back of the flush's own data."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    buf = torch.ones(2 * max(l2, 64 << 20) // 8, dtype=torch.int64, device=dev)

    def flush():
        buf.sum()

    return flush


def decode_splits(w, sms):
    """The library's split plan for the decode path: as many splits per (KV group,
    block of 16 grouped rows) as fill two CTAs per SM, at most one per 128-key
    tile of the visible range."""
    lo = max(0, (w.N - w.M) - w.window + 1) if w.window > 0 else 0
    tiles = max(1, -(-(w.N - (lo // 128) * 128) // 128))
    groups = w.B * w.Hkv * -(-(w.Hq // w.Hkv) * w.M // 16)
    s = max(1, min(2 * sms // groups, tiles, 4096))
    per = -(-tiles // s)
    return -(-tiles // per)


def path_launches(path_name, w=None, sms=152):
    """Kernel launches per call: prefill one; decode one when a group's splits
    fit a thread-block cluster (they merge in the kernel), else split + merge."""
    if path_name != "decode":
        return 1
    return 1 if w is not None and decode_splits(w, sms) <= 8 else 2


def chosen_path(w):
    import streaming_attention_gb300 as sa

    G = w.Hq // w.Hkv
    lo = max(0, (w.N - w.M) - w.window + 1) if w.window > 0 else 0
    if w.D in (64, 128) and G * w.M <= 16 and (w.N - lo) >= 512:
        return sa.PATH_DECODE, "decode"
    return sa.PATH_AUTO, "prefill_or_simt"


def run_ours(args):
    import streaming_attention_gb300 as sa
    from streaming_attention_gb300 import build as sab

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    sab.build()
    w = WORKLOADS[args.workload]
    stream = torch.cuda.current_stream(dev)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    (q, k, v), sets, per_set = rotation(w, dev, l2)
    qd, kd, vd, od = sets[0]
    path, path_name = chosen_path(w)
    nbytes = sa.attn_workspace_bytes_ex(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, w.causal, w.window, path)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    flush = l2_flusher(dev)

    def step_on(t, st):
        sa.attn_fwd_ex(t[0], t[1], t[2], t[3], w.causal, w.window, 0.0, path, ws if nbytes else None, st)

    def step(st):
        step_on(sets[0], st)

    decode = path_name == "decode"
    work = decode_bytes(w) if decode else flops(w)
    unit = "GB/s" if decode else "TFLOP/s"
    scale = 1e9 if decode else 1e12

    barrier(world)
    torch.cuda.synchronize()
    replay_ms = []
    with ClockSampler(local) as clk:
        ms = time_steady(step_on, sets, args.steps, args.warmup, stream, replays=args.replays, samples=replay_ms)
        eager_ms = time_eager_steady(step_on, sets, args.steps, args.warmup, stream)
        cold = time_graph(step, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    barrier(world)
    clocks = clk.summary()
    ms_max, value = whole_job(work, ms, world, dev, scale)
    status = sa.last_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # end to end: host (pinned) buffers through the C ABI, copies inside the timed region
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    e2e_times = []
    for i in range(args.warmup + args.steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        sa.attn_fwd_host(qh, kh, vh, oh, qd, kd, vd, od, w.causal, w.window, 0.0, ws if nbytes else None, stream)
        t1 = time.perf_counter()
        if i >= args.warmup:
            e2e_times.append(t1 - t0)
    e2e_s = max_over_ranks(statistics.mean(e2e_times), world, dev)
    h2d = (q.numel() + k.numel() + v.numel()) * q.element_size()
    d2h = od.numel() * od.element_size()

    pk, pk_src = peaks()
    if decode:
        peak, bound, r_unit = pk["hbm_gbs"], "hbm", "GB/s"
    else:
        peak, bound, r_unit = pk["bf16_tflops"], "tensor", "TFLOP/s"
        if w.dtype == torch.float16:
            peak = pk["bf16_tflops"]  # fp16 and bf16 share the dense tensor rate
    achieved = work / (ms * 1e-3) / scale  # per-rank step time: one launch (prefill; decode with <= 8 splits per KV head)
    traffic = stored_traffic(w.name)

    also = {}
    if not args.no_extra and world == 1:
        also = extra_measurements(args, dev, stream, flush)

    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "fp16",
        "data": "synthetic (seeded N(0,1), rounded to the input dtype)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "M": w.M, "N": w.N, "D": w.D,
                   "causal": w.causal, "window": w.window, "path": path_name,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": (f"inputs larger than L2: steps rotate over {len(sets)} input copies of "
                          f"{per_set / 1e6:.0f} MB each (L2 {l2 / 1e6:.0f} MB)"),
                   "timing": (f"CUDA events around each of {args.replays} replays of one CUDA graph of K "
                              "back-to-back C-ABI calls; ms_per_step is the median replay / K"),
                   "replay_ms_per_step": [round(x, 4) for x in replay_ms],
                   "eager_ms_per_step": round(eager_ms, 4),
                   # causal prefill also counted the other common way (half the noncausal FLOPs)
                   **({"tflops_as_noncausal_half": round(
                       0.5 * 4.0 * w.D * w.B * w.Hq * w.M * w.N / (ms_max * 1e-3) / 1e12, 2)}
                      if not decode and w.causal and w.window <= 0 else {}),
                   "cold_call_us": {"median": round(statistics.median(cold) * 1e3, 2),
                                    "samples": [round(x * 1e3, 2) for x in cold],
                                    "protocol": "graph replay of one call, L2 flushed (2x-L2 read) before each"}},
        "e2e": {"value": round(world * work / e2e_s / scale, 3), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        # launches inside the timed region: every replay runs the K calls of the graph
        "gpu_launches": path_launches(path_name, w, torch.cuda.get_device_properties(dev).multi_processor_count)
        * args.steps * max(1, args.replays),
        "roofline": {"bound": bound, "achieved": round(achieved, 3), "peak": peak, "unit": r_unit,
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": pk_src},
        "clocks": clocks,
    }
    if also:
        line["also"] = also
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def stored_traffic(workload_name):
    """DRAM bytes per launch from a committed ncu capture, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(workload_name)
    if not ent:
        return None
    src = os.path.join(ROOT, ent["source"])
    import hashlib

    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != ent["source_sha"]:
        return None
    return ent["bytes_per_launch"]


def extra_measurements(args, dev, stream, flush):
    """Secondary figures on the same box: noncausal D=128 prefill and GQA decode."""
    import streaming_attention_gb300 as sa

    out = {}
    steps = max(3, min(args.steps, 10))
    for name, w, causal in (("prefill_d128_bf16_noncausal", PREFILL_D128, False),
                            ("prefill_d128_fp16_causal", FP16_D128, True),
                            ("prefill_d64_bf16_noncausal", PREFILL_D64, False),
                            ("prefill_d64_bf16_causal", PREFILL_D64, True),
                            ("long_causal_16k_fp16", LONG_CAUSAL, True),
                            # the pair-MMA prefill (explicit path; AUTO runs the one-CTA kernel)
                            ("prefill_d128_bf16_causal_pair", PREFILL_D128, True),
                            ("prefill_d128_bf16_noncausal_pair", PREFILL_D128, False),
                            ("decode_gqa", DECODE_GQA, DECODE_GQA.causal),
                            ("decode_gqa_d64", DECODE_D64, DECODE_GQA.causal)):
        if name.startswith(("prefill", "long")) and args.workload != PREFILL_D128.name:
            continue
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        _, sets, _ = rotation(w, dev, l2)
        path, pname = chosen_path(w)
        if name.endswith("_pair"):
            path, pname = sa.PATH_PREFILL_PAIR, "prefill pair MMA (cta_group::2)"
        nb = sa.attn_workspace_bytes_ex(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, causal, w.window, path)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)

        def fn_on(t, st, causal=causal, w=w, path=path, nb=nb, ws=ws):
            sa.attn_fwd_ex(t[0], t[1], t[2], t[3], causal, w.window, 0.0, path, ws if nb else None, st)

        ms = time_steady(fn_on, sets, steps, 3, stream)
        cold = statistics.median(time_graph(lambda st: fn_on(sets[0], st), steps, 3, flush))
        if pname == "decode":
            gbs = decode_bytes(w) / (ms * 1e-3) / 1e9
            out[name] = {"GB/s": round(gbs, 1), "us": round(ms * 1e3, 2), "cold_call_us": round(cold * 1e3, 2),
                         "frac_of_hbm": round(gbs / peaks()[0]["hbm_gbs"], 4), "path": pname,
                         "shape": {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "M": w.M, "N": w.N, "window": w.window,
                                   "D": w.D}}
        else:
            out[name] = {"TFLOP/s": round(flops(w, causal) / (ms * 1e-3) / 1e12, 2), "us": round(ms * 1e3, 1),
                         "cold_call_us": round(cold * 1e3, 1), "path": pname}
        del sets, ws
    if args.workload == PREFILL_D128.name:
        for causal in (True, False):
            name = "prefill_d128_e4m3_" + ("causal" if causal else "noncausal")
            out[name] = fp8_measure(PREFILL_D128, causal, steps, dev, stream, flush)
        # D = 64 in E4M3: the 128-column kernel with the upper half of every tile zero
        for causal in (False, True):
            name = "prefill_d64_e4m3_" + ("causal" if causal else "noncausal")
            out[name] = fp8_measure(PREFILL_D64, causal, steps, dev, stream, flush)
    if args.workload == PREFILL_D128.name:
        out["prefill_d128_bf16_causal_backward"] = backward_measure(PREFILL_D128, True, steps, dev, stream)
        out["prefill_d128_bf16_noncausal_backward"] = backward_measure(PREFILL_D128, False, steps, dev, stream)
        # the CUDA-core backward of the small head dimensions (a covering path), on a 1024-row shape
        small = PREFILL_D64.with_(D=32, name="prefill_b4_h16_1024x1024_d32_bf16")
        out["prefill_d32_bf16_causal_backward"] = backward_measure(small, True, steps, dev, stream)
    if args.workload == PREFILL_D128.name:
        out["split_softmax_bf16_m1024_n131072"] = split_softmax_measure(1024, 131072, 4096, steps, dev, stream)
        out["split_softmax_bf16_m1024_n131072_resident"] = split_softmax_measure(1024, 131072, 0, steps, dev,
                                                                                  stream)
    if args.workload in (PREFILL_D128.name, DECODE_GQA.name):
        out["decode_gqa_e4m3"] = fp8_decode_measure(DECODE_GQA, None, steps, dev, stream, flush)
        out["decode_gqa_e4m3_paged128"] = fp8_decode_measure(DECODE_GQA, 128, steps, dev, stream, flush)
    if args.workload in (PREFILL_D128.name, DECODE_GQA.name):
        for ps in (16, 128):
            out[f"decode_gqa_paged{ps}"] = paged_decode_measure(DECODE_GQA, ps, steps, dev, stream, flush)
        # D = 64 (upper half of each tile read as zeros), and 8 speculative rows
        # per sequence (32 grouped rows per KV head: two CTAs of 16) at D = 128
        import dataclasses
        out["decode_gqa_d64_paged16"] = paged_decode_measure(DECODE_D64, 16, steps, dev, stream, flush)
        m8 = dataclasses.replace(DECODE_GQA, name="decode_gqa_b8_hq32_hkv8_m8_n8192_w4096_d128_bf16", M=8)
        out["decode_gqa_m8_paged16"] = paged_decode_measure(m8, 16, steps, dev, stream, flush)
        # the grouped CUDA-core paged kernel (D = 32, a covering path)
        d32 = DECODE_GQA.with_(D=32, name="decode_gqa_b8_hq32_hkv8_m1_n8192_w4096_d32_bf16")
        out["decode_gqa_d32_paged16"] = paged_decode_measure(d32, 16, steps, dev, stream, flush)
    return out


def fp8_measure(w, causal, steps, dev, stream, flush):
    """attn_fwd_fp8 on the workload's shape with seeded E4M3 inputs (descale 1)
    and a BF16 output; the same algorithmic FLOPs as the 16-bit forward, and the
    roofline peak is the 8-bit dense rate: the measured BF16 peak times the
    nominal 8-bit / 16-bit ratio of 2."""
    import streaming_attention_gb300 as sa
    from streaming_attention_gb300.inputs import make_qkv_fp8

    q, k, v = make_qkv_fp8(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, w.seed)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_set = q.numel() * 3 + k.numel() * 2
    r = max(2, min(8, math.ceil(3 * l2 / per_set) + 1))
    sets = [(q.to(dev), k.to(dev), v.to(dev), torch.empty(q.shape, dtype=torch.bfloat16, device=dev))
            for _ in range(r)]

    def fn_on(t, st):
        sa.attn_fwd_fp8(t[0], t[1], t[2], t[3], None, causal, w.window, 0.0, 1.0, 1.0, 1.0, path=sa.PATH_PREFILL,
                        stream=st)

    ms = time_steady(fn_on, sets, steps, 3, stream)
    cold = statistics.median(time_graph(lambda st: fn_on(sets[0], st), steps, 3, flush))
    tf = flops(w, causal) / (ms * 1e-3) / 1e12
    pk, pk_src = peaks()
    fp8_peak = 2.0 * pk["bf16_tflops"] if pk.get("bf16_tflops") else None
    del sets
    return {"TFLOP/s": round(tf, 2), "us": round(ms * 1e3, 1), "cold_call_us": round(cold * 1e3, 1),
            "frac_of_fp8_peak": round(tf / fp8_peak, 4) if fp8_peak else None,
            "fp8_peak_tflops": round(fp8_peak, 1) if fp8_peak else None,
            "peak_source": f"derived: 2 x {pk_src} bf16 (nominal 8-bit / 16-bit dense ratio)",
            "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4) if pk.get("bf16_tflops") else None,
            "path": "prefill tcgen05 kind::f8f6f4 (E4M3 Q, K, V and P)"
            + (", D = 64 read as 128 with the upper half zero" if w.D == 64 else "")}


def fp8_decode_measure(w, page_size, steps, dev, stream, flush):
    """The decode workload on E4M3 inputs (descale 1, BF16 output): contiguous
    (attn_fwd_fp8, decode path) or a paged cache of `page_size`-key pages in a
    shuffled pool (attn_decode_paged_fp8). Bytes count 1 per Q/K/V element."""
    import numpy as np

    import streaming_attention_gb300 as sa
    from streaming_attention_gb300.inputs import make_qkv_fp8

    q, k, v = make_qkv_fp8(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, w.seed)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_set = 2 * k.numel() + 3 * q.numel()
    r = max(2, min(8, math.ceil(3 * l2 / per_set) + 1))
    if page_size:
        npg = w.N // page_size
        perm = torch.from_numpy(np.random.default_rng(w.seed).permutation(w.B * npg))

        def pool(x):  # page i of the cache stored at pool slot perm[i] (rearranged as raw bytes)
            x = x.view(torch.uint8)
            pg = x.reshape(w.B, w.Hkv, npg, page_size, w.D).permute(0, 2, 1, 3, 4).reshape(
                w.B * npg, w.Hkv, page_size, w.D)
            out = torch.empty_like(pg)
            out[perm] = pg
            return out.view(torch.float8_e4m3fn)

        k, v = pool(k), pool(v)
        td = perm.reshape(w.B, npg).to(torch.int32).to(dev)
        lens = torch.full((w.B,), w.N, dtype=torch.int32, device=dev)
        nb = sa.attn_decode_paged_fp8_workspace_bytes(w.B, w.Hq, w.Hkv, w.M, w.D, page_size, npg, w.N, w.causal,
                                                      w.window)
    else:
        nb = sa.attn_fwd_fp8_workspace_bytes(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, w.causal, w.window, sa.PATH_DECODE)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
    sets = [(q.to(dev), k.to(dev), v.to(dev), torch.empty(q.shape, dtype=torch.bfloat16, device=dev))
            for _ in range(r)]

    def fn_on(t, st):
        if page_size:
            sa.attn_decode_paged_fp8(t[0], t[1], t[2], td, lens, t[3], w.N, w.causal, w.window, 0.0, 1.0, 1.0,
                                     1.0, ws, st)
        else:
            sa.attn_fwd_fp8(t[0], t[1], t[2], t[3], None, w.causal, w.window, 0.0, 1.0, 1.0, 1.0, sa.PATH_DECODE,
                            ws, st)

    ms = time_steady(fn_on, sets, steps, 3, stream)
    cold = statistics.median(time_graph(lambda st: fn_on(sets[0], st), steps, 3, flush))
    del sets
    pk, pk_src = peaks()
    gbs = decode_bytes(w, 1) / (ms * 1e-3) / 1e9
    return {"GB/s": round(gbs, 1), "us": round(ms * 1e3, 2), "cold_call_us": round(cold * 1e3, 2),
            "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "peak_source": pk_src,
            "bytes": "E4M3 Q, K, V (1 byte each) + BF16 O",
            "path": (f"paged decode, {page_size}-key pages, shuffled pool" if page_size else "decode") + ", E4M3"}


def backward_measure(w, causal, steps, dev, stream):
    """attn_bwd on the workload (forward output and log-sum-exp from attn_fwd_lse,
    a seeded N(0,1) dO); algorithmic FLOPs 2.5x the forward's (five products of
    the forward's size over the allowed pairs: dV, dP, dS*K, dS^T*Q and the
    recomputed S)."""
    import streaming_attention_gb300 as sa

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    _, sets, _ = rotation(w, dev, l2)
    bsets = []
    for qd, kd, vd, od in sets:
        lse = torch.empty(qd.shape[:3], dtype=torch.float32, device=dev)
        sa.attn_fwd_lse(qd, kd, vd, od, lse, causal, w.window)
        d_o = torch.randn(qd.shape, generator=torch.Generator().manual_seed(12)).to(w.dtype).to(dev)
        bsets.append((qd, kd, vd, od, d_o, lse, torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)))
    del sets
    ws = torch.empty(max(sa.attn_bwd_workspace_bytes(w.B, w.Hq, w.M), 1), dtype=torch.uint8, device=dev)

    def fn_on(t, st):
        sa.attn_bwd(*t, causal=causal, window=w.window, workspace=ws, stream=st)

    ms = time_steady(fn_on, bsets, steps, 3, stream)
    work = 2.5 * flops(w, causal)
    del bsets
    kern = "tcgen05 dK/dV kernel + dQ kernel" if w.D in (64, 128) else "CUDA-core dK/dV kernel + dQ kernel"
    return {"TFLOP/s": round(work / (ms * 1e-3) / 1e12, 2), "us": round(ms * 1e3, 1),
            "flops": "2.5x forward (five products over allowed pairs)", "path": f"backward ({kern})",
            "shape": {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "M": w.M, "N": w.N, "D": w.D}}


def split_softmax_measure(M, N, chunk, steps, dev, stream):
    """Wide-row split softmax of a seeded N(0,1) [M, N] BF16 matrix; bytes are the
    form's own traffic: x read twice (statistics, then normalization) and y
    written once for the three-kernel form (chunk > 0); x read once and y
    written once for the row-resident form (chunk 0)."""
    import streaming_attention_gb300 as sa

    x = (torch.randn(M, N, generator=torch.Generator().manual_seed(7)) * 4).to(torch.bfloat16)
    sets = [(x.to(dev), torch.empty(M, N, dtype=torch.bfloat16, device=dev)) for _ in range(3)]
    ws = torch.empty(sa.attn_split_softmax_workspace_bytes(M, N, chunk), dtype=torch.uint8, device=dev)

    def fn_on(t, st):
        sa.split_softmax(t[0], chunk, y=t[1], workspace=ws, stream=st)

    ms = time_steady(fn_on, sets, steps, 3, stream)
    nbytes = (3.0 if chunk else 2.0) * M * N * 2
    del sets
    return {"GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "us": round(ms * 1e3, 1),
            "bytes": "x read twice + y written once" if chunk else "x read once + y written once",
            "path": f"split softmax, chunk {chunk}" if chunk else "split softmax, row-resident clusters"}


def paged_decode_measure(w, page_size, steps, dev, stream, flush):
    """The decode workload with its cache cut into pages of `page_size` keys,
    stored in a shuffled order in the pool (attn_decode_paged)."""
    import numpy as np

    import streaming_attention_gb300 as sa

    q, k, v = workload_inputs(w)
    npg = w.N // page_size
    perm = torch.from_numpy(np.random.default_rng(w.seed).permutation(w.B * npg))

    def pool(x):  # [B, Hkv, N, D] -> [B * npg, Hkv, page_size, D], page i stored at slot perm[i]
        pg = x.reshape(w.B, w.Hkv, npg, page_size, w.D).permute(0, 2, 1, 3, 4).reshape(w.B * npg, w.Hkv,
                                                                                   page_size, w.D)
        out = torch.empty_like(pg)
        out[perm] = pg
        return out

    table = perm.reshape(w.B, npg).to(torch.int32)
    per_set = 2 * q.numel() * 2 + 2 * k.numel() * 2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    r = max(2, min(8, math.ceil(3 * l2 / per_set) + 1))
    kp, vp = pool(k), pool(v)
    sets = [(q.to(dev), kp.to(dev), vp.to(dev), torch.empty_like(q, device=dev)) for _ in range(r)]
    td = table.to(dev)
    lens = torch.full((w.B,), w.N, dtype=torch.int32, device=dev)
    nb = sa.attn_decode_paged_workspace_bytes(w.B, w.Hq, w.Hkv, w.M, w.D, page_size, npg, w.N, w.causal, w.window)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)

    def fn_on(t, st):
        sa.attn_decode_paged(t[0], t[1], t[2], td, lens, t[3], w.N, w.causal, w.window, 0.0, ws, st)

    ms = time_steady(fn_on, sets, steps, 3, stream)
    cold = statistics.median(time_graph(lambda st: fn_on(sets[0], st), steps, 3, flush))
    gbs = decode_bytes(w) / (ms * 1e-3) / 1e9
    pk, pk_src = peaks()
    kernel = "tcgen05 split" if w.D in (64, 128) else "grouped CUDA-core"
    return {"GB/s": round(gbs, 1), "us": round(ms * 1e3, 2), "cold_call_us": round(cold * 1e3, 2),
            "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "peak_source": pk_src,
            "path": f"paged decode ({kernel} kernel), {page_size}-key pages, shuffled pool",
            "shape": {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "M": w.M, "N": w.N, "window": w.window, "D": w.D}}


# ----------------------------------------------------------------------------
# CPU baseline / reference arm: the FP64 oracle on a bounded sample
# ----------------------------------------------------------------------------
def oracle_sample(w, seconds, seed=0):
    """Times the oracle on random rows of the workload until about `seconds`
    of CPU work; returns (flops done, wall seconds, rows, threads)."""
    import numpy as np

    import oracle

    q, k, v = workload_inputs(w)
    q64, k64, v64 = (t.to(torch.float64).numpy() for t in (q, k, v))
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.Hq * w.M
    threads = oracle.cpu_threads()
    done_flops, wall, nrows = 0.0, 0.0, 0
    batch = max(threads * 4, 64)
    while wall < seconds:
        rows = rng.integers(0, total_rows, batch)
        t0 = time.perf_counter()
        oracle.attention_rows(q64, k64, v64, rows, causal=w.causal, window=w.window, nthreads=threads)
        dt = time.perf_counter() - t0
        wall += dt
        nrows += len(rows)
        done_flops += sum(4.0 * w.D * visible_keys(int(r) % w.M, w.M, w.N, w.causal, w.window) for r in rows)
        if dt < seconds / 8:
            batch *= 2
    return done_flops, wall, nrows, threads


def cpu_baseline(w, seconds):
    """The oracle's throughput in the bench line's unit (GB/s pro rata by rows for decode)."""
    fl, wall, nrows, threads = oracle_sample(w, seconds)
    if chosen_path(w)[1] == "decode":
        value, unit = decode_bytes(w) * nrows / (w.B * w.Hq * w.M) / wall / 1e9, "GB/s"
    else:
        value, unit = fl / wall / 1e12, "TFLOP/s"
    return {"value": round(value, 6), "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"{nrows} random query rows of {w.name} ({fl / 1e9:.1f} GFLOP FP64, {wall:.1f} s)"}


def run_reference(args):
    rank, local, world = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        oracle_sample(w, min(1.0, per_step), seed=1)
    fl_tot, wall_tot, rows_tot, threads = 0.0, 0.0, 0, 1
    for s in range(args.steps):
        fl, wall, nrows, threads = oracle_sample(w, per_step, seed=100 + s)
        fl_tot += fl
        wall_tot += wall
        rows_tot += nrows
    _, path_name = chosen_path(w)
    if path_name == "decode":
        # the same algorithmic bytes as our arm, pro rata for the rows sampled
        value = decode_bytes(w) * rows_tot / (w.B * w.Hq * w.M) / wall_tot / 1e9
        unit = "GB/s"
    else:
        value = fl_tot / wall_tot / 1e12
        unit = "TFLOP/s"
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(wall_tot / args.steps * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1), rounded to the input dtype, widened to FP64)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "M": w.M, "N": w.N, "D": w.D,
                   "causal": w.causal, "window": w.window},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": f"{rows_tot} random query rows over {args.steps} steps"},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--replays", type=int, default=300,
                    help="timed replays of the K-call graph (median reported, all kept)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
