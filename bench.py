"""Benchmark: one training step of sharded causal attention per timed step.

A step is one pass of the whole hot path on device-resident inputs: P ring
steps of per-block (o, lse) partials with double-buffered key/value staging,
the exact lse merge, delta, the fp16 cast of the queries and the P ring
steps of the backward.  Rows are addressed by their global positions, so the
zigzag map needs no copy; with --addressing permuted the step also permutes
Q/K/V and inverse-permutes the outputs.  Default workload: B=1, H=16,
S=32768, D=128 bf16, P=4 zigzag shards (the training-step case);
--workload picks another of seeded_inputs.

FLOPs: forward 2*B*H*S^2*D, backward 5*B*H*S^2*D (causal; five matmuls in
the backward including the recompute of S).

Multi-GPU: the path is computed on one GPU per process; with torchrun each
rank runs an independent replica (no data-path collective) and the rank-0
line reports the whole job's FLOPs over the slowest rank's time.

--impl reference times the fp64 CPU oracle instead (the deliberately slow
plain implementation), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import atexit
import dataclasses
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

import torch  # noqa: E402

import seeded_inputs  # noqa: E402
from seeded_inputs import WORKLOADS  # noqa: E402

METRIC = "causal attn fwd/bwd TFLOP/s and % of BF16 tensor peak, S=8K–128K, 1×GB300"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
L2_BYTES = 129 * 2 ** 20


def flops(w, fwd=True, bwd=True):
    if w.method == "lasp":
        # the chunked linear-attention algorithm with blocks of C rows, per row:
        # forward K^T V and Q.state (2 D^2 each) and the block's left product
        # (2 C D twice); backward two state products more and six block ones
        C, rows = 64.0, w.B * w.H * w.S
        f = rows * (4.0 * w.D * w.D + 4.0 * C * w.D) if fwd else 0.0
        if bwd and w.backward:
            f += rows * (8.0 * w.D * w.D + 12.0 * C * w.D)
        return f
    f = 2.0 * w.B * w.H * w.S * w.S * w.D if fwd else 0.0
    if bwd and w.backward:
        f += 5.0 * w.B * w.H * w.S * w.S * w.D
    return f


def workload_config(w, ws: int, visit: str = "ring", inner: int = 0) -> dict:
    """The `config` object both arms print for a workload."""
    from sharded_causal_softmax_gb300.sharded import AUTO_FUSED_MAX_ROWS, resolve_schedule
    sched = (resolve_schedule(w.schedule, w.S, w.P, visit) if w.method == "softmax"
             else "state passed shard to shard")
    cfg = {"workload": w.description, "name": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "P": w.P,
           "method": w.method, "layout": w.layout, "schedule": sched, "kv_heads": w.kv_heads or w.H,
           "head_groups": w.head_groups, "step": "fwd+bwd" if w.backward else "fwd", "flops_per_step": flops(w),
           "parallelism": f"{ws} independent replica(s), one per GPU"}
    if visit == "double_ring":
        cfg["visit"] = f"double_ring (inner rings of {inner})"
    if w.schedule == "auto" and w.method == "softmax":
        cfg["schedule_choice"] = (f"auto: fused (one launch per direction) up to {AUTO_FUSED_MAX_ROWS} rows per "
                                  "shard, ring above")
    return cfg


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if ws <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every `period_ms` from
    before the warm-up on; summary() keeps the samples taken inside a host
    time window (the timed region)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []   # (host monotonic time, csv line)

    def start(self, wait_s: float = 5.0):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        atexit.register(self.stop)   # never leave the sampler running
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        t_end = time.monotonic() + wait_s   # let it start sampling before the region opens
        while not self.lines and time.monotonic() < t_end:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = [ln for t, ln in self.lines if t0 <= t <= t1]
        for line in window:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "period_ms": self.period_ms}


def choose_bf16_peak(peaks, region_ms, clocks):
    """The measured bf16 peak that matches how the kernel was timed: the
    burst figure (a short cuBLAS run at full clock) when the timed region is
    short (< 1 s) and the SM clock held at its maximum, else the sustained
    one (a seconds-long run under the power cap).  Returns (peak, name)."""
    burst = peaks.get("bf16_tflops")
    sustained = peaks.get("bf16_tflops_sustained", burst)
    mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    at_max = mhz is not None and mx is not None and mhz >= 0.97 * mx
    if burst is not None and region_ms < 1000.0 and at_max:
        return burst, "burst"
    return sustained, "sustained"


def pinned_copy_gbs(device, nbytes=256 << 20, reps=5):
    """Host<->device copy bandwidth from pinned memory on this machine (best of
    `reps` copies of `nbytes`, CUDA events), in GB/s per direction."""
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dev = torch.empty(nbytes, dtype=torch.uint8, device=device)
    out = {}
    for name, dst, src in (("h2d", dev, host), ("d2h", host, dev)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            dst.copy_(src, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out[name] = round(nbytes / (best * 1e-3) / 1e9, 1)
    return out


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "sharded_causal_softmax_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, sources, workload: str):
    """dram bytes per launch from a committed ncu summary, if it was taken
    on the current source of the kernel; else None."""
    try:
        with open(TRAFFIC_PATH) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(sources) or rec.get("workload") != workload:
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------ GPU arm ----

def run_gpu(args):
    import sharded_causal_softmax_gb300 as sca
    from sharded_causal_softmax_gb300 import build as sca_build

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    if rank == 0 or ws == 1:
        sca_build.build()
    barrier(ws)
    w = WORKLOADS[args.workload]
    if args.heads:   # a smaller case of the same kernels, for profiler captures
        kvh = None if w.kv_heads is None else max(1, args.heads * w.kv_heads // w.H)
        w = dataclasses.replace(w, H=args.heads, kv_heads=kvh,
                                head_groups=1 if args.heads % w.head_groups else w.head_groups,
                                description=w.description + f" (profiling case: H={args.heads})")
    dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inputs = seeded_inputs.workload_inputs(w)
    dev_in = [x.to(device) for x in inputs]
    if args.schedule:
        w = dataclasses.replace(w, schedule=args.schedule)
    visit = {"visit": "double_ring", "inner": args.inner} if args.visit == "double_ring" else {}

    def make_plan(**over):
        if w.method == "lasp":
            return sca.ShardedLinearAttention(w.B, w.H, w.S, w.D, w.P, dtype=dtype, backward=w.backward,
                                              block=args.lasp_block or None)
        kw = dict(layout=w.layout, dtype=dtype, head_groups=w.head_groups, schedule=w.schedule,
                  backward=w.backward, addressing=args.addressing, kv_heads=w.kv_heads, **visit)
        kw.update(over)
        return sca.ShardedCausalAttention(w.B, w.H, w.S, w.D, w.P, **kw)

    plan = make_plan()
    stream = torch.cuda.current_stream(device)

    # per-launch timing of the attention kernels (same stream they run on)
    timing = {"fwd": [], "bwd": []}
    orig_fwd, orig_bwd = sca.capi.attn_fwd_shard, sca.capi.attn_bwd_shard

    def timed(kind, fn):
        def wrapper(*a, **k):
            if not timing_on[0]:
                return fn(*a, **k)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            r = fn(*a, **k)
            e1.record(stream)
            timing[kind].append((e0, e1))
            return r
        return wrapper

    timing_on = [False]
    sca.sharded.capi.attn_fwd_shard = timed("fwd", orig_fwd)
    sca.sharded.capi.attn_bwd_shard = timed("bwd", orig_bwd)
    sca.capi.lasp_fwd = timed("fwd", sca.capi.lasp_fwd)
    sca.capi.lasp_bwd = timed("bwd", sca.capi.lasp_bwd)

    # HBM-bound kernels: events around each call, algorithmic bytes from its
    # arguments (read + written once)
    hbm = {"zigzag_permute_kernel": [], "merge_lse_kernel": [], "delta_kernel": []}

    def timed_hbm(name, fn, nbytes):
        def wrapper(*a, **k):
            if not timing_on[0]:
                return fn(*a, **k)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            r = fn(*a, **k)
            e1.record(stream)
            hbm[name].append((e0, e1, nbytes(*a)))
            return r
        return wrapper

    def permute_bytes(src, dst, outer, S, row_bytes, *rest):   # (P, inverse, status, stream follow)
        return 2 * outer * S * row_bytes

    def merge_bytes(o_parts, lse_parts, n, rows, D, o_stride, lse_stride, o_out, lse_out, o_bf16, *rest):
        return (n + 1) * rows * (4 * D + 4) + (2 * rows * D if o_bf16 else 0)

    def delta_bytes(o, dout, dout_dtype, delta, rows, D, *rest):
        return rows * (4 * D + (2 if dout_dtype == 0 else 4) * D + 4)

    sca.sharded.capi.zigzag_permute = timed_hbm("zigzag_permute_kernel", sca.capi.zigzag_permute, permute_bytes)
    sca.sharded.capi.attn_merge_lse = timed_hbm("merge_lse_kernel", sca.capi.attn_merge_lse, merge_bytes)
    sca.sharded.capi.attn_bwd_delta = timed_hbm("delta_kernel", sca.capi.attn_bwd_delta, delta_bytes)

    staged = {"bytes": 0}

    def step(p=None):
        p = plan if p is None else p
        p.forward(*dev_in[:3])
        kern = p.kernels
        staged["bytes"] += getattr(p, "staged_bytes", 0)
        if w.backward:
            p.backward(dev_in[3])
            kern += p.kernels
            staged["bytes"] += getattr(p, "staged_bytes", 0)
        return kern

    clocks = ClockSampler(local).start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if plan.read_status() != 0:
        raise RuntimeError("device status word reports a failure")

    # timed region: inputs (> L2) resident in HBM
    barrier(ws)
    torch.cuda.synchronize()
    timing_on[0] = True
    ring_staged = getattr(plan, "stage_k", None) is not None
    if ring_staged:
        plan.stage_events = []
    staged["bytes"] = 0
    launches = 0
    h0 = time.monotonic()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        launches += step()
    t1.record(stream)
    torch.cuda.synchronize()
    h1 = time.monotonic()
    clocks.stop()
    timing_on[0] = False
    barrier(ws)
    ms = t0.elapsed_time(t1)
    ms_max = max_over_ranks(ms, ws, device)
    ms_per_step = ms_max / args.steps
    step_flops = flops(w)
    value = step_flops * args.steps * ws / (ms_max * 1e-3) / 1e12
    clock_summary = clocks.summary(h0, h1)

    # What the ring's staging costs the step: its copy-engine time per step,
    # and the step time of the same launches reading every block from its
    # home rows (no staging copies), timed the same way right after.
    staging = None
    if ring_staged:
        copy_ms = sum(a.elapsed_time(b) for a, b in plan.stage_events) / args.steps
        plan.stage_events = None
        home = make_plan(schedule="direct", group_steps=False)
        for _ in range(max(1, args.warmup)):
            step(home)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(args.steps):
            step(home)
        a1.record(stream)
        torch.cuda.synchronize()
        if home.read_status() != 0:
            raise RuntimeError("device status word reports a failure")
        home_ms = max_over_ranks(a0.elapsed_time(a1), ws, device) / args.steps
        del home
        # one hand-off alone (the rotation of staged blocks between two ring
        # steps, nothing else running): the copy engine's own rate
        cs = plan.copy_stream
        plan.staged_bytes = 0
        h0e, h1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(cs):
            h0e.record(cs)
            plan._stage(dev_in[1], dev_in[2], 2 if w.P > 2 else 1)
            h1e.record(cs)
        torch.cuda.synchronize()
        handoff_ms = h0e.elapsed_time(h1e)
        handoff_bytes = plan.staged_bytes
        staging = {"bytes_per_step": staged["bytes"] // args.steps, "copy_ms_per_step": round(copy_ms, 4),
                   "ring_ms_per_step": round(ms_per_step, 4), "home_read_ms_per_step": round(home_ms, 4),
                   "exposed_ms_per_step": round(ms_per_step - home_ms, 4),
                   "exposed_frac_of_step": round((ms_per_step - home_ms) / ms_per_step, 4),
                   "handoff_alone_ms": round(handoff_ms, 4), "handoff_bytes": handoff_bytes,
                   "handoff_alone_gbs": round(handoff_bytes / (handoff_ms * 1e-3) / 1e9, 1),
                   "note": "home_read: the same per-step launches with every block read from its home rows"}

    # end to end through the public API with host buffers: every step copies
    # its inputs in from pinned host memory and all its results (O, lse and
    # the gradients) back out.  Steps are pipelined the way a training loop
    # runs them: two plans double-buffer the device inputs and outputs, so
    # step i+1's host->device copy and step i-1's device->host copy run on
    # copy streams while step i computes.
    pinned = [x.pin_memory() for x in inputs]
    h2d = sum(x.numel() * x.element_size() for x in pinned)
    plans = [plan, make_plan()]
    dins = [dev_in, [torch.empty_like(x) for x in dev_in]]

    def results(p):
        out = [p.o] + ([p.lse] if hasattr(p, "lse") else [])
        return out + ([p.dq, p.dk, p.dv] if w.backward else [])

    outs_host = [[torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in results(p)] for p in plans]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_steps_run(n, start_ev=None):
        for i in range(n):
            j = i % 2
            p, din = plans[j], dins[j]
            if i == 0 and start_ev is not None:
                s_in.wait_event(start_ev)
            if i >= 2:
                s_in.wait_event(ev_comp[j])     # step i-2 has read slot j's inputs
            with torch.cuda.stream(s_in):
                for d, h in zip(din, pinned):
                    d.copy_(h, non_blocking=True)
            ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            if i >= 2:
                stream.wait_event(ev_out[j])    # slot j's results of step i-2 are on the host
            p.forward(*din[:3])
            if w.backward:
                p.backward(din[3])
            ev_comp[j].record(stream)
            s_out.wait_event(ev_comp[j])
            with torch.cuda.stream(s_out):
                for hst, r in zip(outs_host[j], results(p)):
                    hst.copy_(r, non_blocking=True)
            ev_out[j].record(s_out)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    e2e_steps_run(2)   # untimed: both plans warm
    barrier(ws)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps = max(2, min(args.steps, 6))
    e2e_steps_run(e2e_steps, start_ev=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    if any(p.read_status() != 0 for p in plans):
        raise RuntimeError("device status word reports a failure")
    d2h = sum(x.numel() * x.element_size() for x in outs_host[0])
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, device)
    e2e_value = step_flops * e2e_steps * ws / (e2e_ms * 1e-3) / 1e12
    # the copies' own limit on this machine: each direction on its own copy
    # engine, so a step can go no faster than the slower direction's bytes
    # at its measured pinned bandwidth, nor than the device-side step
    del plans, dins
    copy_gbs = pinned_copy_gbs(device)
    copy_ms = max(h2d / (copy_gbs["h2d"] * 1e9), d2h / (copy_gbs["d2h"] * 1e9)) * 1e3
    bound_ms = max(copy_ms, ms_per_step)
    e2e_ms_step = e2e_ms / e2e_steps

    # dominant kernel and its roofline
    per = {}
    for kind, evs in timing.items():
        if evs:
            durs = [a.elapsed_time(b) for a, b in evs]
            per[kind] = (sum(durs), len(durs))
    peaks, peak_src = load_peaks()
    bf16_peak, bf16_regime = choose_bf16_peak(peaks, ms_max, clock_summary)
    other_regime = "sustained" if bf16_regime == "burst" else "burst"
    other_peak = peaks.get("bf16_tflops_sustained" if other_regime == "sustained" else "bf16_tflops", bf16_peak)
    kind = max(per, key=lambda k: per[k][0])
    total_ms, n = per[kind]
    avg_s = total_ms / n * 1e-3
    # the FLOPs of that direction over the timed steps, shared by its launches
    # (P per direction on the ring, one when fused)
    launch_flops = flops(w, fwd=(kind == "fwd"), bwd=(kind == "bwd")) * args.steps / n
    tc = plan.uses_tensor_cores(kind)
    bound_of = getattr(plan, "roofline_bound", None)
    if bound_of is not None and bound_of(kind) == "hbm":
        # bytes-bound kernels: algorithmic bytes of one call over its time
        peak = peaks.get("hbm_gbs", 6800.0)
        bound, unit = "hbm", "GB/s"
        peak_note = f"{peak_src} copy bandwidth"
    elif tc:
        peak = bf16_peak
        bound, unit = "tensor", "TFLOP/s"
        peak_note = (f"{peak_src} bf16 {bf16_regime} (timed region {ms_max:.0f} ms at median SM "
                     f"{clock_summary.get('sm_mhz')} of {clock_summary.get('sm_max_mhz')} MHz)")
    else:
        # fp32 FMA issue: 152 SMs x 128 FMA/clk x 2 flop x measured max SM clock
        mhz = peaks.get("sm_max_mhz", 2070.0)
        peak = 152 * 128 * 2 * mhz * 1e6 / 1e12
        bound, unit = "alu", "TFLOP/s"
        peak_note = "derived fp32 FMA peak (152 SM x 128 FMA/clk x 2 x max SM clock)"
    if bound == "hbm":
        launch_bytes = plan.algorithmic_bytes(kind)
        achieved = launch_bytes / avg_s / 1e9
    else:
        achieved = launch_flops / avg_s / 1e12
    src = plan.kernel_sources(kind)
    traffic = measured_traffic(plan.kernel_name(kind), src, w.name)
    roofline = {"kernel": plan.kernel_name(kind), "bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 1),
                "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": peak_note, "launches_timed": n, "avg_launch_ms": round(avg_s * 1e3, 4),
                "flops_per_launch": launch_flops}
    if bound == "hbm":
        roofline["bytes_per_launch"] = launch_bytes
        roofline["tflops"] = round(launch_flops / avg_s / 1e12, 2)
    # the tensor pipe's own dense rate at the clock the region ran at: one
    # M=128, N=128, K=16 bf16 MMA every 64 clk per SM (measured by a probe),
    # 8192 FLOP/clk x 152 SMs; the measured cuBLAS peaks above sit below it
    pipe_mhz = clock_summary.get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
    pipe_peak = 8192 * 152 * pipe_mhz * 1e6 / 1e12
    if bound == "tensor":
        roofline["peak_regime"] = bf16_regime
        roofline[f"frac_{other_regime}"] = round(achieved / other_peak, 4)
        roofline[f"peak_{other_regime}"] = other_peak
        roofline["sm_mhz_median"] = clock_summary.get("sm_mhz")
        roofline["frac_of_tensor_pipe"] = round(achieved / pipe_peak, 4)
        roofline["tensor_pipe_peak"] = round(pipe_peak, 1)
        roofline["tensor_pipe_peak_source"] = (f"8192 FLOP/clk/SM x 152 SMs x {pipe_mhz:.0f} MHz "
                                               "(the region's median SM clock, else the maximum)")
    permute_alone = not hbm["zigzag_permute_kernel"] and w.layout == "zigzag"
    if permute_alone:
        # the step addresses rows by position and runs no permute: time the
        # permute kernel alone on one input (forward and inverse), untimed
        # for the step
        src = dev_in[0]
        scratch = torch.empty_like(src)
        timing_on[0] = True
        for inv in (0, 1, 0, 1):
            # a short spin keeps the stream busy while the host issues the
            # call, so the events bracket the kernel and not the host's
            # latency (the step's kernels are always queued behind others)
            torch.cuda._sleep(200_000)
            sca.sharded.capi.zigzag_permute(src.data_ptr() if inv == 0 else scratch.data_ptr(),
                                            scratch.data_ptr() if inv == 0 else src.data_ptr(),
                                            w.B * w.H, w.S, w.D * src.element_size(), w.P, inv,
                                            plan.status.data_ptr(), stream.cuda_stream)
        timing_on[0] = False
        # reference: a plain device copy of the same bytes, timed the same
        # way (the measured copy peak comes from copies several times larger)
        ref_ms = []
        for _ in range(4):
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(200_000)
            r0.record(stream)
            scratch.copy_(src)
            r1.record(stream)
            ref_ms.append((r0, r1))
        torch.cuda.synchronize()
        same_size_copy_ms = sum(a.elapsed_time(b) for a, b in ref_ms) / len(ref_ms)
        del scratch
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    hbm_stats = {}
    for name, evs in hbm.items():
        if evs:
            t = sum(a.elapsed_time(b) for a, b, _ in evs) * 1e-3
            nb = sum(x for _, _, x in evs)
            hbm_stats[name] = {"launches": len(evs), "avg_launch_ms": round(t / len(evs) * 1e3, 4),
                               "gbs": round(nb / t / 1e9, 1), "frac": round(nb / t / 1e9 / hbm_peak, 4),
                               "bytes_per_launch": nb // len(evs)}
    if permute_alone and "zigzag_permute_kernel" in hbm_stats:
        ps = hbm_stats["zigzag_permute_kernel"]
        ps["note"] = "timed alone: the step addresses rows by position"
        ps["same_size_copy_gbs"] = round(ps["bytes_per_launch"] / (same_size_copy_ms * 1e-3) / 1e9, 1)
        ps["frac_of_same_size_copy"] = round(ps["gbs"] / ps["same_size_copy_gbs"], 4)
    other = {}
    for k, v in per.items():
        tf = flops(w, fwd=(k == "fwd"), bwd=(k == "bwd")) * args.steps / v[0] * 1e-9
        other[k] = {"kernel": plan.kernel_name(k), "avg_launch_ms": round(v[0] / v[1], 4), "launches": v[1],
                    "tflops": round(tf, 2)}
        if plan.uses_tensor_cores(k) and not (bound_of is not None and bound_of(k) == "hbm"):
            other[k][f"frac_{bf16_regime}"] = round(tf / bf16_peak, 4)
            other[k][f"frac_{other_regime}"] = round(tf / other_peak, 4)
            other[k]["frac_of_tensor_pipe"] = round(tf / pipe_peak, 4)

    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1))",
        "config": dict(workload_config(w, ws, args.visit, args.inner), addressing=plan.addressing,
                       l2="inputs larger than L2 (no flush)"
                       if sum(x.numel() * x.element_size() for x in inputs) > L2_BYTES else "inputs fit in L2"),
        "clocks": clock_summary,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": round(e2e_ms_step, 4),
                "copy_gbs": copy_gbs, "copy_bound_ms_per_step": round(copy_ms, 4),
                "bound_ms_per_step": round(bound_ms, 4), "frac_of_bound": round(bound_ms / e2e_ms_step, 4),
                "pipeline": "two plans; each step's H2D and D2H run on copy streams beside the compute",
                "bound": "max(device step, the slower copy direction's bytes at its measured pinned bandwidth)"},
        "gpu_launches": launches,
        "roofline": roofline,
        "kernels": other,
        "hbm_kernels": {"peak_gbs": hbm_peak, "peak_source": f"{peak_src} copy bandwidth", **hbm_stats},
    }
    if staging is not None:
        line["staging"] = staging
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------ CPU oracle ----

def oracle_sample(w, S_sample):
    """One head of the workload over its first S_sample positions (a causal
    prefix is itself a causal attention problem): inputs and FLOPs."""
    ins = seeded_inputs.workload_inputs(w)
    head = [x[:1, :1, :S_sample] for x in ins]
    f = flops(dataclasses.replace(w, B=1, H=1, S=S_sample))
    return head, f


def run_oracle_once(w, head):
    import oracle
    scale = 1.0 / math.sqrt(w.D)
    if w.method == "lasp":
        oracle.linear_attention(head[0], head[1], head[2], scale)
        if w.backward:
            oracle.linear_attention_backward(head[0], head[1], head[2], head[3], scale)
        return
    o, lse = oracle.attention(head[0], head[1], head[2], scale)
    if w.backward:
        oracle.attention_backward(head[0], head[1], head[2], head[3], scale, o=o, lse=lse)


def pick_sample(w, budget_s):
    S_sample = min(w.S, 4096)
    head, f = oracle_sample(w, S_sample)
    t = time.perf_counter()
    run_oracle_once(w, head)
    dt = time.perf_counter() - t
    # scale the prefix (work ~ S^2) to roughly the budget
    target = S_sample * math.sqrt(max(1.0, budget_s / max(dt, 1e-3)))
    S2 = int(min(w.S, max(S_sample, 2 ** int(math.log2(target)))))
    return S2


def cpu_baseline(w, budget_s=15.0):
    S2 = pick_sample(w, budget_s)
    head, f = oracle_sample(w, S2)
    t = time.perf_counter()
    run_oracle_once(w, head)
    dt = time.perf_counter() - t
    return {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"fp64 numpy oracle, {'fwd+bwd' if w.backward else 'fwd'} of one head (b=0, h=0) over the "
                      f"first {S2} positions ({f / 1e9:.1f} GFLOP, {dt:.1f} s)"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    if args.schedule:   # the same config object as the GPU arm (the oracle's math does not depend on it)
        w = dataclasses.replace(w, schedule=args.schedule)
    S2 = pick_sample(w, budget_s=min(12.0, 150.0 / max(1, args.steps + args.warmup)))
    head, f = oracle_sample(w, S2)
    for _ in range(args.warmup):
        run_oracle_once(w, head)
    t = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_once(w, head)
    dt = time.perf_counter() - t
    value = f * args.steps / dt / 1e12
    sample = (f"fp64 numpy oracle, {'fwd+bwd' if w.backward else 'fwd'} of one head over the first {S2} "
              f"positions per step ({f / 1e9:.1f} GFLOP)")
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
            "impl": "reference",
            "config": workload_config(w, ws, args.visit, args.inner),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="train_s32k")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--schedule", choices=["auto", "ring", "direct", "fused"], default=None,
                    help="override the workload's schedule")
    ap.add_argument("--addressing", choices=["auto", "position", "permuted"], default="auto")
    ap.add_argument("--visit", choices=["ring", "double_ring"], default="ring",
                    help="order in which each shard visits the key/value blocks")
    ap.add_argument("--inner", type=int, default=2, help="double ring: shards per inner ring")
    ap.add_argument("--lasp-block", type=int, default=0,
                    help="linear attention: rows per stored state (64: CUDA cores; a multiple of 128: tensor cores)")
    ap.add_argument("--heads", type=int, default=0,
                    help="override the head count (profiler captures of a smaller case; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
