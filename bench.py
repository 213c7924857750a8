#!/usr/bin/env python3
"""Throughput bench for the GLA prefill forward (one JSON line on rank 0).

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

A step is one gla_fwd call over the whole workload (B=1, H=16, T=16384, Dk=Dv=128,
bf16 q/k/v/o, fp32 log-gates), inputs resident in HBM. L2 is flushed (a 256 MiB
device write) before every step, outside the timed events. Each step is timed with
CUDA events on the launching stream; value = tokens (B*T, summed over ranks) / the
max over ranks of the summed step times.

Under torchrun (N > 1) every rank runs its own copy of the workload on its own GPU
(weak scaling, no collective on the data path; the (batch, head) problems are
independent). The reference arm (--impl reference) times the fp64 CPU oracle on a
bounded sample of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GLA prefill fwd tokens/s (B·T, H=16 D=128 bf16) and % of HBM/tensor roofline"
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20
NOMINAL_HBM_GBS = 8000.0   # nominal HBM3e bandwidth of the part, for a second fraction
KERNEL_SOURCES = {
    "tc": ["chunkwise_recurrent_prefill_gb300/csrc/gla_tc.cu"],
    "exact": ["chunkwise_recurrent_prefill_gb300/csrc/gla_exact.cu"],
    "gdn": ["chunkwise_recurrent_prefill_gb300/csrc/gdn.cu"],
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--path", default="auto", choices=["auto", "tc", "exact"])
    ap.add_argument("--seq-splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU work of the oracle baseline sample")
    ap.add_argument("--op", default="prefill", choices=["prefill", "step", "gdn"],
                    help="prefill (the headline), one decode step on a resident state, or the "
                         "gated delta rule forward")
    return ap.parse_args()


# ------------------------------------------------------------------ workload arithmetic

def algorithmic_bytes(w) -> int:
    """Bytes a forward must move at least: q, k, v read, o written (io dtype), g read
    (fp32), plus h0 read / hT written when the workload carries them."""
    es = 2 if w.io == "bf16" else 4
    gate_bytes = w.Dk * 4 if getattr(w, "gate", "key") == "key" else 4
    per_token_head = 2 * w.Dk * es + w.Dv * es + w.Dv * es + gate_bytes
    n = w.B * w.T * w.H * per_token_head
    state = w.B * w.H * w.Dk * w.Dv * 4
    return n + (state if w.with_h0 else 0) + (state if w.want_hT else 0)


def algorithmic_flops(w, C: int = 64) -> int:
    """Chunkwise flops (causal half of the in-chunk products): per token and head
    4*Dk*Dv (state contribution and q.S) + (C+1)*(Dk+Dv) (q.k^T and P.v)."""
    return w.B * w.T * w.H * (4 * w.Dk * w.Dv + (C + 1) * (w.Dk + w.Dv))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def source_sha(path_kind: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(path_kind, []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def committed_traffic(kernel_kind: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, or None if the kernel source
    changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        entries = json.load(f)
    sha = source_sha(kernel_kind)
    for e in entries:
        if e.get("kernel_kind") == kernel_kind and e.get("workload") == workload \
                and e.get("source_sha256") == sha:
            return int(e["dram_bytes_per_launch"])
    return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.t_lo = self.t_hi = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, lo, hi):
        self.t_lo, self.t_hi = lo, hi

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def count_in(self, lo, hi):
        return sum(1 for t, _ in self.samples if lo <= t <= hi)

    def summary(self, source="timed region"):
        rows = []
        for t, line in self.samples:
            if self.t_lo is not None and not (self.t_lo <= t <= self.t_hi):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append(dict(sm=float(parts[0]), smax=float(parts[1]), hw=parts[4],
                                 hwt=parts[5], swt=parts[6], swp=parts[7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in timed region"]}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "source": source}


# ------------------------------------------------------------------ arms

def per_key_gates(w, g):
    """The oracle's gate layout [B,T,H,Dk]: a scalar gate is the same in every key dim."""
    if getattr(w, "gate", "key") == "key":
        return g.numpy()
    return g[..., None].expand(*g.shape, w.Dk).contiguous().numpy()


def cpu_oracle_sample(w, x_cpu, target_s: float):
    """Time the fp64 C oracle on a bounded sample of the workload: the first T_s tokens of
    every (batch, head) pair, repeated until ~target_s of CPU time has been spent (T_s is the
    whole sequence when one pass is shorter than the target)."""
    import numpy as np
    import oracle
    oracle.build()
    q = x_cpu["q"].float().numpy()
    k = x_cpu["k"].float().numpy()
    v = x_cpu["v"].float().numpy()
    g = per_key_gates(w, x_cpu["g"])
    h0 = None if x_cpu["h0"] is None else x_cpu["h0"].numpy()
    cal_T = min(w.T, 256)
    t0 = time.perf_counter()
    oracle.recurrent(q[:, :cal_T], k[:, :cal_T], v[:, :cal_T], g[:, :cal_T], x_cpu["scale"], h0)
    rate = (w.B * cal_T) / max(time.perf_counter() - t0, 1e-6)   # tokens/s (all heads)
    T_s = int(min(w.T, max(64, (target_s * rate) / w.B)))
    sl = [np.ascontiguousarray(a[:, :T_s]) for a in (q, k, v, g)]
    reps, dt = 0, 0.0
    while reps == 0 or dt < target_s:
        t0 = time.perf_counter()
        oracle.recurrent(*sl, x_cpu["scale"], h0)
        dt += time.perf_counter() - t0
        reps += 1
    return {"value": reps * (w.B * T_s) / dt, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"first {T_s} of {w.T} tokens of all {w.B}x{w.H} (batch, head) pairs, "
                      f"{reps} pass(es), fp64 C recurrence, {dt:.2f} s"}


def run_reference(args, w, rank, world):
    """--impl reference: the fp64 CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs
    oracle.build()
    x = make_inputs(w)
    q = x["q"].float().numpy()
    k = x["k"].float().numpy()
    v = x["v"].float().numpy()
    g = per_key_gates(w, x["g"])
    h0 = None if x["h0"] is None else x["h0"].numpy()
    # size each step so that warmup + steps take ~150 s of CPU time in total
    cal_T = min(w.T, 128)
    t0 = time.perf_counter()
    oracle.recurrent(q[:, :cal_T], k[:, :cal_T], v[:, :cal_T], g[:, :cal_T], x["scale"], h0)
    rate = (w.B * cal_T) / max(time.perf_counter() - t0, 1e-6)
    per_step_s = 150.0 / max(1, args.steps + args.warmup)
    T_s = int(min(w.T, max(1, per_step_s * rate / w.B)))
    sl = [np.ascontiguousarray(a[:, :T_s]) for a in (q, k, v, g)]
    for _ in range(args.warmup):
        oracle.recurrent(*sl, x["scale"], h0)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.recurrent(*sl, x["scale"], h0)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * w.B * T_s / total
    sample = (f"each step: first {T_s} of {w.T} tokens of all {w.B}x{w.H} (batch, head) "
              f"pairs, fp64 C recurrence on host cores")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, "oracle"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def max_over_ranks(seconds: float, dist, device) -> float:
    """The slowest rank's time (every rank gets the same number)."""
    if dist is None:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank processed `steps` x its own workload."""
    return world * tokens_per_rank * steps / max_seconds


def workload_config(w, path):
    l2 = ("n/a (host CPU)" if path == "oracle"
          else "flushed by a 256 MiB device write before every timed step")
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Dk": w.Dk, "Dv": w.Dv,
            "io": w.io, "gate": ("fp32 log-gate logsigmoid(u)/16, "
                                 + ("one per key dim" if w.gate == "key" else "one per token and head")),
            "path": path,
            "h0": w.with_h0, "hT": w.want_hT, "l2": l2}


def run_ours(args, w, rank, world, dist):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from chunkwise_recurrent_prefill_gb300 import gla
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs

    dev = torch.device("cuda", torch.cuda.current_device())
    x_cpu = make_inputs(w)
    x = {k_: (v_.to(dev) if hasattr(v_, "to") else v_) for k_, v_ in x_cpu.items()}
    o = torch.empty((w.B, w.T, w.H, w.Dv), dtype=x["q"].dtype, device=dev)
    hT = torch.empty((w.B, w.H, w.Dk, w.Dv), dtype=torch.float32, device=dev) \
        if w.want_hT else None
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        gla.gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], o=o, hT=hT,
                    path=args.path, seq_splits=args.seq_splits, gate=w.gate, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert gla.last_device_status() == 0, "device error during warm-up"

    gid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gid if gid.startswith("GPU-") else "GPU-" + gid)
    sampler.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = gla.launch_counter()
    t_lo = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_hi = time.time()
    if dist:
        dist.barrier()
    launches = gla.launch_counter() - launches0
    time.sleep(0.1)
    clock_source = "timed region"
    if sampler.count_in(t_lo, t_hi) < 3:
        # the timed region was shorter than a few sampling periods: run the same step (flush
        # included) back to back for ~0.6 s right after it and read the clocks there
        t_lo = time.time()
        while time.time() - t_lo < 0.6:
            for _ in range(20):
                flush.zero_()
                step()
            torch.cuda.synchronize()
        t_hi = time.time()
        clock_source = ("the same step run back to back for 0.6 s right after the timed "
                        "region (which was shorter than the 20 ms sampling period allows)")
        time.sleep(0.1)
    sampler.mark(t_lo, t_hi)
    sampler.stop()
    assert gla.last_device_status() == 0, "device error during the timed region"
    ms = [a.elapsed_time(b) for a, b in evs]
    total_s = max_over_ranks(sum(ms) / 1e3, dist, dev)
    tokens = w.B * w.T
    value = weak_scaling_value(tokens, args.steps, world, total_s)
    ms_sorted = sorted(ms)
    per_launch_s = total_s / args.steps

    # roofline of the dominant (only) kernel of the call
    hbm_gbs, bf16_tflops, peak_src = load_peaks()
    abytes = algorithmic_bytes(w)
    aflops = algorithmic_flops(w)
    achieved = abytes / per_launch_s / 1e9
    kind = gla.path_for(w.B, w.T, w.H, w.Dk, w.Dv, w.io, args.path)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                "traffic": committed_traffic(kind, w.name),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)",
                "algorithmic_bytes_per_launch": abytes,
                "tensor_frac": (aflops / per_launch_s / 1e12) / bf16_tflops,
                "kernel": kind}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, x_cpu, dev, stream, gla, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(w, x_cpu, args.cpu_seconds)

    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per_launch_s,
            "ms_p50": ms_sorted[len(ms) // 2], "ms_p95": ms_sorted[int(0.95 * (len(ms) - 1))],
            "ms_p99": ms_sorted[int(0.99 * (len(ms) - 1))],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) q/k/v, logsigmoid(N(0,1))/16 gates)",
            "config": workload_config(w, kind), "clocks": sampler.summary(clock_source),
            "gpu_launches": launches, "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
        }), flush=True)


def run_e2e(args, w, x_cpu, dev, stream, gla, world, dist):
    """End to end through the public API: every step copies its inputs from pinned host
    memory to the device, runs the forward and copies its output (and final state) back to
    pinned host memory. Steps are pipelined two deep on three streams, as a serving loop
    would run them: step i+1's inputs upload while step i computes and step i-1's output
    downloads (the host link is full duplex). The timed region spans the first upload to the
    last download."""
    import torch
    steps = max(3, min(args.steps, 50))
    names = [k_ for k_ in ("q", "k", "v", "g", "h0") if x_cpu.get(k_) is not None]
    host = {k_: x_cpu[k_].pin_memory() for k_ in names}
    slots = []
    for _ in range(2):
        dbuf = {k_: torch.empty_like(host[k_], device=dev) for k_ in names}
        o = torch.empty((w.B, w.T, w.H, w.Dv), dtype=x_cpu["q"].dtype, device=dev)
        hT = (torch.empty((w.B, w.H, w.Dk, w.Dv), dtype=torch.float32, device=dev)
              if w.want_hT else None)
        o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hT_host = torch.empty(hT.shape, dtype=hT.dtype).pin_memory() if hT is not None else None
        ev = {n: torch.cuda.Event() for n in ("up", "fwd", "down")}
        slots.append(dict(d=dbuf, o=o, hT=hT, o_host=o_host, hT_host=hT_host, ev=ev,
                          used=False))
    s_up, s_fwd, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    h2d = sum(host[k_].numel() * host[k_].element_size() for k_ in names)
    d2h = slots[0]["o"].numel() * slots[0]["o"].element_size() + \
        (slots[0]["hT"].numel() * 4 if w.want_hT else 0)

    def step(i):
        sl = slots[i % 2]
        with torch.cuda.stream(s_up):
            if sl["used"]:
                s_up.wait_event(sl["ev"]["fwd"])       # the slot's last forward read its inputs
            for k_ in names:
                sl["d"][k_].copy_(host[k_], non_blocking=True)
            sl["ev"]["up"].record(s_up)
        with torch.cuda.stream(s_fwd):
            s_fwd.wait_event(sl["ev"]["up"])
            if sl["used"]:
                s_fwd.wait_event(sl["ev"]["down"])     # the slot's last output was copied out
            d = sl["d"]
            gla.gla_fwd(d["q"], d["k"], d["v"], d["g"], x_cpu["scale"], d.get("h0"),
                        o=sl["o"], hT=sl["hT"], path=args.path, seq_splits=args.seq_splits,
                        gate=w.gate, stream=s_fwd)
            sl["ev"]["fwd"].record(s_fwd)
        with torch.cuda.stream(s_down):
            s_down.wait_event(sl["ev"]["fwd"])
            sl["o_host"].copy_(sl["o"], non_blocking=True)
            if sl["hT"] is not None:
                sl["hT_host"].copy_(sl["hT"], non_blocking=True)
            sl["ev"]["down"].record(s_down)
        sl["used"] = True

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    for i in range(steps):
        step(i)
    b.record(s_down)   # ordered after every download, which waited on every forward and upload
    torch.cuda.synchronize()
    total_s = max_over_ranks(a.elapsed_time(b) / 1e3, dist, dev)
    return {"value": weak_scaling_value(w.B * w.T, steps, world, total_s), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "pipelined": "2 deep: upload, forward and download of consecutive steps overlap"}


def run_step(args, rank, world, dist):
    """One decode step per timed iteration on the decode workload: every step reads and
    rewrites the whole fp32 state, so the bound is HBM bandwidth."""
    import torch
    from chunkwise_recurrent_prefill_gb300 import gla
    from chunkwise_recurrent_prefill_gb300.workloads import STEP_WORKLOAD, make_step_inputs
    sw = STEP_WORKLOAD
    B, H, D = sw["B"], sw["H"], sw["D"]
    gla.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    x = make_step_inputs(B, H, D, sw["io"], sw["seed"], dev)
    o = torch.empty_like(x["v"])
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        gla.gla_step(x["q"], x["k"], x["v"], x["g"], x["scale"], x["S"], o=o, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert gla.last_device_status() == 0
    gid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gid if gid.startswith("GPU-") else "GPU-" + gid)
    sampler.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = gla.launch_counter()
    t_lo = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_hi = time.time()
    launches = gla.launch_counter() - launches0
    time.sleep(0.1)
    clock_source = "timed region"
    if sampler.count_in(t_lo, t_hi) < 3:
        # the timed region was shorter than a few sampling periods: run the same step (flush
        # included) back to back for ~0.6 s right after it and read the clocks there
        t_lo = time.time()
        while time.time() - t_lo < 0.6:
            for _ in range(20):
                flush.zero_()
                step()
            torch.cuda.synchronize()
        t_hi = time.time()
        clock_source = ("the same step run back to back for 0.6 s right after the timed "
                        "region (which was shorter than the 20 ms sampling period allows)")
        time.sleep(0.1)
    sampler.mark(t_lo, t_hi)
    sampler.stop()
    ms = sorted(a.elapsed_time(b) for a, b in evs)
    total_s = max_over_ranks(sum(ms) / 1e3, dist, dev)
    per = total_s / args.steps
    es = 2
    nbytes = B * H * (2 * D * D * 4 + 2 * D * es + 2 * D * es + D * 4)
    hbm_gbs, _, peak_src = load_peaks()
    achieved = nbytes / per / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": f"GLA decode step tokens/s (one token for each of B={B} sequences, "
                      f"H={H}, D={D}, bf16 q/k/v/o, fp32 state)",
            "value": weak_scaling_value(B, args.steps, world, total_s), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * per, "ms_p50": ms[len(ms) // 2],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0,1) q/k/v, logsigmoid(N(0,1))/16 gates, 0.02 N(0,1) state)",
            "config": {"workload": sw["name"], "B": B, "H": H, "Dk": D, "Dv": D, "io": sw["io"],
                       "l2": "flushed by a 256 MiB device write before every timed step"},
            "clocks": sampler.summary(clock_source), "gpu_launches": launches,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "traffic": None,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)",
                         "algorithmic_bytes_per_launch": nbytes, "kernel": "step"},
            "e2e": None, "cpu_baseline": None,
        }), flush=True)


def gdn_flops_per_token_head(Dk: int, Dv: int, C: int = 64) -> int:
    """Flops of the gated-delta-rule chunk algebra per token and head (causal halves
    of the in-chunk products): K K^T and Q K^T 2*C*Dk, the triangular solves C*(Dk+Dv),
    W S, Qh S and Kh^T U 6*Dk*Dv, P U C*Dv."""
    return 2 * C * Dk + C * (Dk + Dv) + 6 * Dk * Dv + C * Dv


TF32_PER_BF16 = 1.1 / 2.25   # nominal dense tensor rates of the part (PFLOP/s)


def fp32_alu_peak_tflops(sm_mhz: float | None) -> tuple[float, str]:
    """CUDA-core fp32 FMA peak: 152 SMs x 128 fp32 lanes x 2 flops x SM clock (the median
    clock sampled in the timed region, else the 2070 MHz maximum)."""
    mhz = sm_mhz or 2070.0
    return 152 * 128 * 2 * mhz * 1e6 / 1e12, f"152 SMs x 128 fp32 lanes x 2 x {mhz:.0f} MHz"


def run_gdn(args, rank, world, dist):
    """The gated delta rule forward on its bench workload (B=1, H=16, T=16384, D=128, bf16)."""
    import torch
    from chunkwise_recurrent_prefill_gb300 import gla
    from chunkwise_recurrent_prefill_gb300.workloads import (GDN_BENCH_WORKLOAD, GDN_WORKLOADS,
                                                             make_gdn_inputs)
    w = GDN_WORKLOADS[args.workload or GDN_BENCH_WORKLOAD]
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    x_cpu = make_gdn_inputs(w)
    x = {k_: (v_.to(dev) if hasattr(v_, "to") else v_) for k_, v_ in x_cpu.items()}
    o = torch.empty((w.B, w.T, w.H, w.Dv), dtype=x["q"].dtype, device=dev)
    hT = torch.empty((w.B, w.H, w.Dk, w.Dv), dtype=torch.float32, device=dev) \
        if w.want_hT else None
    ws = torch.empty(gla.gdn_workspace_size(w.B, w.T, w.H, w.Dk, w.Dv), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        gla.gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], o=o, hT=hT,
                    workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert gla.last_device_status() == 0
    gid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gid if gid.startswith("GPU-") else "GPU-" + gid)
    sampler.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = gla.launch_counter()
    t_lo = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_hi = time.time()
    if dist:
        dist.barrier()
    launches = gla.launch_counter() - launches0
    time.sleep(0.1)
    clock_source = "timed region"
    if sampler.count_in(t_lo, t_hi) < 3:
        # the timed region was shorter than a few sampling periods: run the same step (flush
        # included) back to back for ~0.6 s right after it and read the clocks there
        t_lo = time.time()
        while time.time() - t_lo < 0.6:
            for _ in range(20):
                flush.zero_()
                step()
            torch.cuda.synchronize()
        t_hi = time.time()
        clock_source = ("the same step run back to back for 0.6 s right after the timed "
                        "region (which was shorter than the 20 ms sampling period allows)")
        time.sleep(0.1)
    sampler.mark(t_lo, t_hi)
    sampler.stop()
    assert gla.last_device_status() == 0
    ms = sorted(a.elapsed_time(b) for a, b in evs)
    total_s = max_over_ranks(sum(ms) / 1e3, dist, dev)
    per = total_s / args.steps
    clocks = sampler.summary(clock_source)
    flops = w.B * w.T * w.H * gdn_flops_per_token_head(w.Dk, w.Dv)
    achieved = flops / per / 1e12
    es = 2 if w.io == "bf16" else 4
    nbytes = w.B * w.T * w.H * ((2 * w.Dk + 2 * w.Dv) * es + 8)
    hbm_gbs, bf16_tflops, peaks_src = load_peaks()
    tensor_path = w.io == "bf16" and w.Dk == 128 and w.Dv == 128
    if tensor_path:
        # tcgen05 kernels: bf16 products in the prep, tf32 products in the serial scan (the
        # larger share of the call); the tf32 peak is the measured bf16 peak x the nominal
        # dense tf32 / bf16 ratio (1.1 / 2.25 PFLOP/s)
        bound, peak = "tensor", bf16_tflops * TF32_PER_BF16
        peak_desc = (f"{peaks_src}: MEASURED_PEAKS.json bf16_tflops (burst) x {TF32_PER_BF16:.3f} "
                     "(nominal dense tf32 / bf16)")
        path = "gdn (tcgen05: bf16 prep, tf32 state scan)"
    else:
        peak, peak_desc = fp32_alu_peak_tflops(clocks.get("sm_mhz"))
        bound, peak_desc, path = "alu", "derived: " + peak_desc, "gdn (fp32 CUDA cores)"
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = gdn_cpu_oracle_sample(w, x_cpu, args.cpu_seconds)
    if rank == 0:
        print(json.dumps({
            "metric": GDN_METRIC,
            "value": weak_scaling_value(w.B * w.T, args.steps, world, total_s),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * per, "ms_p50": ms[len(ms) // 2],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "tf32" if tensor_path else "f32",
            "data": "synthetic (seeded unit-norm q/k, N(0,1) v, logsigmoid(N(0,1))/16 gates, "
                    "sigmoid(N(0,1)) write strengths)",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Dk": w.Dk, "Dv": w.Dv,
                       "io": w.io, "h0": w.with_h0, "hT": w.want_hT, "path": path,
                       "l2": "flushed by a 256 MiB device write before every timed step"},
            "clocks": clocks, "gpu_launches": launches,
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": committed_traffic("gdn", w.name),
                         "peak_source": peak_desc,
                         "algorithmic_flops_per_launch": flops,
                         "algorithmic_bytes_per_launch": nbytes,
                         "hbm_frac": nbytes / per / 1e9 / hbm_gbs,
                         "kernel": "gdn_prep + gdn_scan (one call)"},
            "e2e": None, "cpu_baseline": cpu,
        }), flush=True)


GDN_METRIC = "gated delta rule prefill fwd tokens/s (B·T, H=16 D=128 bf16)"


def run_reference_gdn(args, rank, world):
    """--impl reference --op gdn: the fp64 numpy token loop of the gated delta rule, each
    step a bounded sample (the first T_s tokens of every (batch, head) pair), rank 0 only."""
    if rank != 0:
        return
    import oracle
    from oracle import gdn_ref
    from chunkwise_recurrent_prefill_gb300.workloads import (GDN_BENCH_WORKLOAD, GDN_WORKLOADS,
                                                             make_gdn_inputs)
    oracle.build()
    w = GDN_WORKLOADS[args.workload or GDN_BENCH_WORKLOAD]
    x = make_gdn_inputs(w)
    cut = lambda t, n: None if t is None else t[:, :n].contiguous()   # noqa: E731
    args_ = lambda n: [cut(x[k_], n) for k_ in ("q", "k", "v", "g", "beta")]   # noqa: E731
    cal = min(w.T, 256)
    t0 = time.perf_counter()
    gdn_ref.recurrent_c(*args_(cal), x["scale"], x["h0"])
    rate = w.B * cal / max(time.perf_counter() - t0, 1e-6)
    per_step_s = 150.0 / max(1, args.steps + args.warmup)
    T_s = int(min(w.T, max(1, per_step_s * rate / w.B)))
    sl = args_(T_s)
    for _ in range(args.warmup):
        gdn_ref.recurrent_c(*sl, x["scale"], x["h0"])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        gdn_ref.recurrent_c(*sl, x["scale"], x["h0"])
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * w.B * T_s / total
    sample = (f"each step: first {T_s} of {w.T} tokens of all {w.B}x{w.H} (batch, head) pairs, "
              f"fp64 C token loop on the host cores")
    print(json.dumps({
        "impl": "reference", "metric": GDN_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Dk": w.Dk, "Dv": w.Dv,
                   "io": w.io, "path": "oracle", "l2": "n/a (host CPU)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def gdn_cpu_oracle_sample(w, x_cpu, target_s: float):
    """The fp64 C token loop of the gated delta rule (OpenMP over the (batch, head) pairs) on
    the first T_s tokens of every pair, T_s sized for about target_s of host time."""
    import oracle
    from oracle import gdn_ref
    oracle.build()
    cut = lambda t, n: None if t is None else t[:, :n].contiguous()   # noqa: E731
    args_ = lambda n: [cut(x_cpu[k_], n) for k_ in ("q", "k", "v", "g", "beta")]   # noqa: E731
    cal = min(w.T, 256)
    t0 = time.perf_counter()
    gdn_ref.recurrent_c(*args_(cal), x_cpu["scale"], x_cpu["h0"])
    rate = w.B * cal / max(time.perf_counter() - t0, 1e-6)
    T_s = int(min(w.T, max(64, target_s * rate / w.B)))
    sl = args_(T_s)
    t0 = time.perf_counter()
    gdn_ref.recurrent_c(*sl, x_cpu["scale"], x_cpu["h0"])
    dt = time.perf_counter() - t0
    return {"value": w.B * T_s / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"first {T_s} of {w.T} tokens of all {w.B}x{w.H} (batch, head) pairs, "
                      f"fp64 C token loop, {dt:.2f} s"}


def main():
    args = parse_args()
    from chunkwise_recurrent_prefill_gb300.workloads import BENCH_WORKLOAD, WORKLOADS
    w = WORKLOADS[args.workload or BENCH_WORKLOAD] if args.op != "gdn" else None
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if args.op == "gdn":
            run_reference_gdn(args, rank, world)
        else:
            run_reference(args, w or WORKLOADS[BENCH_WORKLOAD], rank, world)
        return
    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    else:
        torch.cuda.set_device(0)
    try:
        if args.op == "step":
            run_step(args, rank, world, dist)
        elif args.op == "gdn":
            run_gdn(args, rank, world, dist)
        else:
            run_ours(args, w, rank, world, dist)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
