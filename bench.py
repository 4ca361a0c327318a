#!/usr/bin/env python3
"""Benchmark of the mHC site program on GB300.

A step is one pass of the whole site program -- hc_pre_fused (RMS-rescaled
mixes contraction, gates, Sinkhorn, collapse) then hc_post -- over one batch of
synthetic tokens already resident in HBM.  The default workload is the prefill
chunk (T = 4096 tokens, s = 4 streams, hidden 4096, 20 Sinkhorn iterations,
eps 1e-6): its 256 MiB stream state is larger than L2, so every step streams
from HBM without a flush.  The JSON line also carries the T = 1 and T = 8 per-site
latencies (CUDA-graph replay, eager and Prepared calls).  At s > 4 (the wide-stream
workload) the roofline is the pre-chain's against the FP32 peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

With --gpus N > 1 the script expects torchrun: each rank runs its own batch on
its own GPU (weak scaling, no collective on the data path); value is the tokens
of all ranks over the slowest rank's time.  --impl reference times the float64
CPU oracle on the host cores instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mhc_hyper_connection_hc_gb300 import synth  # noqa: E402

METRIC = "mHC site tokens/s + achieved HBM GB/s (fraction of roofline); T=1 µs/site"
NOMINAL_HBM_GBS = 8000.0         # the ~8 TB/s HBM3e figure the targets are stated against
FALLBACK_HBM_GBS = 6800.0        # used only when MEASURED_PEAKS.json is absent
FALLBACK_NOTE = "of fallback (6.8 TB/s, one earlier GB300 measurement)"
GB300_SMS, GB300_MAX_MHZ, FP32_LANES = 152, 2070, 128
WORKLOAD_IDS = {"decode": 1, "verify": 2, "prefill": 3, "sweep": 4, "wide": 5}


# ----------------------------------------------------------------------------- host helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def aggregate(elapsed_s: float, units: float, group=None):
    """Max elapsed and summed units over ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    t = torch.tensor([elapsed_s], dtype=torch.float64)
    u = torch.tensor([units], dtype=torch.float64)
    if dist.get_backend(group) == "nccl":
        t, u = t.cuda(), u.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(p):
        return None
    try:
        return json.load(open(p))
    except (OSError, ValueError):
        return None


def hbm_peak(kind: str):
    """(GB/s, note): the measured copy bandwidth, else the fallback."""
    mp = measured_peaks()
    if mp:
        for key in (f"hbm_gbs_{kind}", "hbm_gbs"):
            if isinstance(mp.get(key), (int, float)):
                return float(mp[key]), f"of measured ({key})"
    return FALLBACK_HBM_GBS, FALLBACK_NOTE


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mhc_hyper_connection_hc_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, only if taken on the
    current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and parts[0] == kernel and parts[1] == workload and parts[3] == want:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms in the background, each
    sample with its timestamp.  mark() brackets the timed region ("start", "end") and the
    end of the measurement region ("region_end": the per-kernel rounds that run the same
    kernels back to back right after the timed steps).  The summary is taken over the
    samples inside the measurement region; sm_mhz is null when none falls inside it."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    STAMP = "%Y/%m/%d %H:%M:%S.%f"
    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = self.t2 = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.25)
        return self

    def mark(self, which: str):
        """Host wall time at "start" / "end" of the timed region, or "region_end"."""
        import datetime
        now = datetime.datetime.now()
        if which == "start":
            self.t0 = now
        elif which == "end":
            self.t1 = now
        else:
            self.t2 = now

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)   # one more sample after the region
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        import datetime
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((datetime.datetime.strptime(parts[0], self.STAMP), float(parts[2]), float(parts[3]),
                             parts[6:10]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        end = self.t2 or self.t1
        timed = [r for r in rows if self.t0 and self.t1 and self.t0 <= r[0] <= self.t1]
        region = [r for r in rows if self.t0 and end and self.t0 <= r[0] <= end]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {n for r in region for n, v in zip(names, r[3]) if v.lower() == "active"}
        return {"sm_mhz": statistics.median(r[1] for r in region) if region else None,
                "sm_max_mhz": max(r[2] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_in_timed_region": len(timed),
                "samples_in_measurement_region": len(region),
                "period_ms": self.PERIOD_MS,
                "region": "the timed steps and the per-kernel rounds right after them (same kernels, "
                          "back to back)"}


# ----------------------------------------------------------------------------- CPU oracle timing

def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo "model name", else the Arm part fields)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model Name", "Hardware"):
        for line in info.splitlines():
            if line.split(":")[0].strip() == key and ":" in line:
                return line.split(":", 1)[1].strip()
    parts = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = (t.strip() for t in line.split(":", 1))
            if k in ("CPU implementer", "CPU part") and k not in parts:
                parts[k] = v
    if parts:
        return "Arm " + ", ".join(f"{k} {v}" for k, v in sorted(parts.items()))
    import platform
    return platform.processor() or platform.machine()


def time_oracle(w: synth.Workload, max_tokens: int, budget_s: float, max_reps: int):
    """Time the float64 oracle (pre + post) on a bounded sample of the workload: on all
    host cores (the reported baseline) and on one thread over a smaller sample."""
    import oracle
    n = min(w.T, max_tokens)
    inp = synth.workload_inputs(w, T=n)
    x = inp["x"].astype(np.float64)
    f = inp["f"].astype(np.float64)
    threads = oracle.default_threads()
    eps = float(np.float32(w.eps))

    def best_of(m, nthreads):
        times = []
        t_start = time.perf_counter()
        while len(times) < max_reps and (not times or time.perf_counter() - t_start < budget_s):
            t0 = time.perf_counter()
            oracle.site(x[:m], inp["fn_w"], inp["scale"], inp["base"], f[:m], w.iters, eps, threads=nthreads)
            times.append(time.perf_counter() - t0)
        return min(times), len(times)

    best, reps = best_of(n, threads)
    n1 = max(1, min(n, max(threads, 1) * 16 if w.K * w.R <= 1 << 21 else 16))
    best1, reps1 = best_of(n1, 1)
    return {"value": n / best, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {w.T} tokens of the {w.name} workload (s={w.s}, d={w.d}, "
                      f"iters={w.iters}), pre-chain + hc_post in float64, best of {reps} "
                      f"runs, inputs pre-widened to float64 outside the timed call",
            "seconds_per_run": best,
            "single_thread": {"value": n1 / best1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{n1} tokens, best of {reps1} runs"},
            "cpu_model": cpu_model(), "host_cores": os.cpu_count()}


def run_reference(args):
    """The oracle as it stands, on the host cores: each step is one float64 pre-chain +
    hc_post over a fixed sample of the workload's tokens (inputs made and widened once,
    outside the timed loop)."""
    import oracle
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = selected_workload(args)
    sample = min(w.T, args.ref_tokens)
    inp = synth.workload_inputs(w, T=sample)
    x = inp["x"].astype(np.float64)
    f = inp["f"].astype(np.float64)
    threads = oracle.default_threads()
    eps = float(np.float32(w.eps))

    def step():
        oracle.site(x, inp["fn_w"], inp["scale"], inp["base"], f, w.iters, eps, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    elapsed = time.perf_counter() - t0
    value = sample * args.steps / elapsed
    cb = {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
          "sample": f"{sample} of {w.T} tokens of the {w.name} workload (s={w.s}, d={w.d}, "
                    f"iters={w.iters}) per step, pre-chain + hc_post in float64, {args.steps} steps",
          "cpu_model": cpu_model(), "host_cores": os.cpu_count()}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, sample_tokens=sample),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def selected_workload(args) -> synth.Workload:
    """The workload named on the command line, with --iters overriding its Sinkhorn
    iterations and --tokens its token count (a smaller case of the same shape, for
    profiler captures; the line then names the workload with that T)."""
    w = synth.WORKLOADS[WORKLOAD_IDS[args.workload]]
    if args.iters is not None:
        if args.iters < 1:
            raise SystemExit("--iters must be >= 1")
        w = dataclasses.replace(w, iters=args.iters)
    if getattr(args, "tokens", None) is not None:
        if args.tokens < 1:
            raise SystemExit("--tokens must be >= 1")
        w = dataclasses.replace(w, T=args.tokens)
    return w


def workload_config(w: synth.Workload, sample_tokens=None):
    cfg = {"workload": f"{w.name}: T={w.T} tokens, streams={w.s}, hidden={w.d}, "
                       f"{w.iters} Sinkhorn iters, eps={w.eps:g}",
           "T": w.T, "streams": w.s, "hidden": w.d, "rows": w.R, "iters": w.iters, "eps": w.eps,
           "x_dist": "U[-1,1)" if w.x_dist == "uniform" else "N(0,1)",
           "l2": f"inputs larger than L2: x is {w.T * w.K * 4 / 2**20:.0f} MiB per step, no flush"
                 if w.T * w.K * 4 > 129e6 else "inputs fit in L2 (latency workload)"}
    if sample_tokens is not None:
        cfg["tokens_per_step_sampled"] = sample_tokens
    return cfg


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch
    from mhc_hyper_connection_hc_gb300 import hc

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    w = selected_workload(args)
    T, s, d, iters = w.T, w.s, w.d, w.iters
    stream = torch.cuda.Stream(device=dev)

    inp = synth.workload_inputs(w)
    with torch.cuda.stream(stream):
        dv = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
        ws = hc.new_workspace(T, s, d, dev, stream)
        out = hc.new_pre_outputs(T, s, d, dev)
        x_out = torch.empty(T, s, d, dtype=torch.float32, device=dev)
    stream.synchronize()
    path = hc.hc_pre_auto_path(T, s, d)
    pre_launches = 1 if path in (hc.HC_PATH_CLUSTER, hc.HC_PATH_WIDE) else 2
    path_name = {hc.HC_PATH_CLUSTER: "cluster", hc.HC_PATH_WIDE: "wide"}.get(path, "generic")
    fused = args.pipeline == "fused"
    fused_cluster = path == hc.HC_PATH_CLUSTER and d // 16 <= 256   # else hc_post + generic pre
    # On the cluster path at prefill sizes a helper kernel runs behind the cluster kernel on
    # the SMs its clusters leave free, for the batch's last tokens (one more launch per call).
    help_pre = max(0, hc.hc_pre_helper_tokens(T, s, d, False, ws.numel()))
    help_fused = max(0, hc.hc_pre_helper_tokens(T, s, d, True, ws.numel())) if fused_cluster else 0
    pre_launches += 1 if help_pre else 0
    fused_launches = (1 + (1 if help_fused else 0)) if fused_cluster else 1 + pre_launches
    if fused:
        # The previous site's gates (this trio on this state, computed once) and the
        # new state: a step is site i's hc_post fused with site i+1's pre-chain.
        with torch.cuda.stream(stream):
            hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], iters, w.eps, out["pre"],
                            out["post"], out["comb"], out["y"], ws, stream)
            post_prev, comb_prev = out["post"].clone(), out["comb"].clone()
        stream.synchronize()

    def boundary():
        hc.hc_post_pre_fused(dv["x"], dv["f"], post_prev, comb_prev, dv["fn_w"], dv["scale"], dv["base"],
                             iters, w.eps, x_out, out["pre"], out["post"], out["comb"], out["y"], ws,
                             stream)

    def pre():
        hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], iters, w.eps, out["pre"],
                        out["post"], out["comb"], out["y"], ws, stream)

    def post():
        hc.hc_post(dv["x"], dv["f"], out["post"], out["comb"], x_out, stream)

    for _ in range(args.warmup):
        pre()
        post()
    stream.synchronize()
    if hc.hc_workspace_status(ws, stream) != 0:
        raise RuntimeError("a kernel flagged an error during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if fused:
        for _ in range(args.warmup):
            boundary()
        stream.synchronize()
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        clk.mark("start")
        for k in range(K):
            ev[k][0].record(stream)
            if fused:
                boundary()
                ev[k][1].record(stream)
            else:
                pre()
                ev[k][1].record(stream)
                post()
            ev[k][2].record(stream)
        stream.synchronize()
        clk.mark("end")
        # The pages' kernel-only timing, right after the timed steps: 20 warm-up then
        # back-to-back launches, in rounds; the median of the rounds' per-launch means.
        rounds = {"hc_pre_fused": timed_rounds(stream, pre, args.rounds, args.round_launches),
                  "hc_post": timed_rounds(stream, post, args.rounds, args.round_launches)}
        if fused:
            rounds["hc_post_pre_fused"] = timed_rounds(stream, boundary, args.rounds, args.round_launches)
        clk.mark("region_end")
    torch.cuda.synchronize(dev)
    barrier()
    clocks = clk.summary()
    total_s = ev[0][0].elapsed_time(ev[-1][2]) / 1e3
    if fused:
        fused_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
        # the two separate launches, timed after the step loop for context
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for k in range(K):
            ev2[k][0].record(stream)
            pre()
            ev2[k][1].record(stream)
            post()
            ev2[k][2].record(stream)
        stream.synchronize()
        pre_ms = [ev2[k][0].elapsed_time(ev2[k][1]) for k in range(K)]
        post_ms = [ev2[k][1].elapsed_time(ev2[k][2]) for k in range(K)]
    else:
        pre_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
        post_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    if hc.hc_workspace_status(ws, stream) != 0:
        raise RuntimeError("a kernel flagged an error in the timed region")
    max_s, all_tokens = aggregate(total_s, float(T * K))

    # Roofline of the dominant kernel (algorithmic bytes per launch / mean launch time).
    pre_bytes = T * s * d * 4 + T * d * 4                 # x read once, y written
    post_bytes = T * s * d * 4 * 2 + T * d * 4            # x and f read, x' written
    pre_flops = 2 * w.R * w.K * T + 2 * w.K * T + 2 * w.K * T
    pre_avg, post_avg = statistics.mean(pre_ms) / 1e3, statistics.mean(post_ms) / 1e3
    peak, note = hbm_peak("burst")
    fp32_peak = GB300_SMS * FP32_LANES * 2 * (clocks.get("sm_mhz") or GB300_MAX_MHZ) * 1e6 / 1e12
    src_hash = kernel_source_hash()
    wl_tag = f"T{T}_s{s}_d{d}"
    kernels = {
        "hc_pre_fused": {"us": pre_avg * 1e6, "algorithmic_bytes": pre_bytes,
                         "GB/s": pre_bytes / pre_avg / 1e9, "frac_hbm": pre_bytes / pre_avg / 1e9 / peak,
                         "TFLOP/s": pre_flops / pre_avg / 1e12,
                         "frac_fp32": pre_flops / pre_avg / 1e12 / fp32_peak,
                         "launches_per_step": pre_launches,
                         "path": path_name, "helper_tokens": help_pre},
        "hc_post": {"us": post_avg * 1e6, "algorithmic_bytes": post_bytes,
                    "GB/s": post_bytes / post_avg / 1e9, "frac_hbm": post_bytes / post_avg / 1e9 / peak,
                    "launches_per_step": 1},
    }
    if fused:
        fz_avg = statistics.mean(fused_ms) / 1e3
        fz_bytes = T * s * d * 4 * 2 + T * d * 4 * 2   # x_prev and f read; x_new and y written
        kernels["hc_post_pre_fused"] = {
            "us": fz_avg * 1e6, "algorithmic_bytes": fz_bytes, "GB/s": fz_bytes / fz_avg / 1e9,
            "frac_hbm": fz_bytes / fz_avg / 1e9 / peak,
            "TFLOP/s": (pre_flops + 2 * (s + 1) * s * d * T) / fz_avg / 1e12,
            "frac_fp32": (pre_flops + 2 * (s + 1) * s * d * T) / fz_avg / 1e12 / fp32_peak,
            "launches_per_step": fused_launches,
            "path": "cluster" if fused_cluster else f"{path_name} (hc_post, then the {path_name} pre-chain)",
            "helper_tokens": help_fused}
        kernels["hc_pre_fused"]["launches_per_step"] = 0
        kernels["hc_post"]["launches_per_step"] = 0
        dom = "hc_post_pre_fused"
    else:
        dom = max(kernels, key=lambda k: kernels[k]["us"])
    for name, r in rounds.items():
        kr = kernels[name]
        kr["us_median_of_rounds"] = r["us_median"]
        kr["rounds"] = r["desc"]
        kr["frac_hbm_median_of_rounds"] = kr["algorithmic_bytes"] / (r["us_median"] * 1e3) / peak
    for kr in kernels.values():
        kr["frac_nominal_8tbs"] = kr["GB/s"] / NOMINAL_HBM_GBS
    kernels["hc_pre_fused"]["l2_cold"] = measure_cold(stream, pre, pre_bytes, peak)
    kd = kernels[dom]
    roofline = {"bound": "hbm", "kernel": dom, "achieved": kd["GB/s"], "peak": peak, "unit": "GB/s",
                "frac": kd["GB/s"] / peak, "peak_note": note,
                "frac_nominal_8tbs": kd["GB/s"] / NOMINAL_HBM_GBS,
                "traffic": profiled_traffic(dom, wl_tag),
                "algorithmic_bytes_per_launch": kd["algorithmic_bytes"]}
    if path == hc.HC_PATH_WIDE:
        # At s > 4 the pre-chain is float32-FMA bound (~36 FLOP per byte at s = 8) and it is
        # the step's dominant kernel: report it against the FP32 peak of the sampled clock.
        kp = kernels["hc_pre_fused"]
        roofline = {"bound": "alu", "kernel": "hc_pre_fused", "achieved": kp["TFLOP/s"], "peak": fp32_peak,
                    "unit": "TFLOP/s", "frac": kp["TFLOP/s"] / fp32_peak,
                    "peak_note": (f"FP32 FMA peak: {GB300_SMS} SMs x {FP32_LANES} lanes x 2 FLOP x "
                                  f"{clocks.get('sm_mhz') or GB300_MAX_MHZ:.0f} MHz (the sampled median clock)"),
                    "traffic": profiled_traffic("hc_pre_fused", wl_tag),
                    "algorithmic_flop_per_launch": pre_flops,
                    "step_hbm": {"kernel": dom, "GB/s": kd["GB/s"], "frac": kd["GB/s"] / peak}}

    line = {"metric": METRIC, "value": all_tokens / max_s, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": 1e3 * max_s / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": dict(workload_config(w), pipeline=args.pipeline, step=(
                "site boundary: the previous site's hc_post fused with this site's pre-chain "
                "(hc_post_pre_fused, one call: the cluster kernel and, on the SMs its clusters leave "
                "free, the helper kernel for the batch's last tokens; the same work as hc_pre_fused + hc_post)"
                if fused else "hc_pre_fused then hc_post")), "roofline": roofline,
            "kernels": kernels,
            "gpu_launches": (fused_launches if fused else pre_launches + 1) * K,
            "clocks": clocks,
            "kernel_sources": src_hash}

    if not args.no_head:
        line["exit_head"] = measure_head(w, dv, ws, stream, peak)
        line["branch_norm"] = measure_norm(w, out["y"], stream, peak, pre_inputs=(dv, ws))
    if not args.no_e2e:
        if fused:
            def boundary_on(bi, bo):
                hc.hc_post_pre_fused(bi["x"], bi["f"], bi["post_prev"], bi["comb_prev"], dv["fn_w"],
                                     dv["scale"], dv["base"], iters, w.eps, bo["x_new"], bo["pre"], bo["post"],
                                     bo["comb"], bo["y"], ws, stream)
            line["e2e"] = measure_e2e(w, {"x": dv["x"], "f": dv["f"], "post_prev": post_prev,
                                          "comb_prev": comb_prev}, dict(out, x_new=x_out), stream, K, boundary_on)
        else:
            def site_on(bi, bo):
                hc.hc_pre_fused(bi["x"], dv["fn_w"], dv["scale"], dv["base"], iters, w.eps, bo["pre"],
                                bo["post"], bo["comb"], bo["y"], ws, stream)
                hc.hc_post(bi["x"], bi["f"], bo["post"], bo["comb"], bo["x_out"], stream)
            line["e2e"] = measure_e2e(w, {"x": dv["x"], "f": dv["f"]}, dict(out, x_out=x_out), stream, K, site_on)
    if not args.no_decode:
        line["decode_t1"] = measure_decode(dev, args.iters)
        line["verify_t8"] = measure_decode(dev, args.iters, cid=2)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = time_oracle(w, max_tokens=args.cpu_tokens, budget_s=10.0, max_reps=3)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def timed_rounds(stream, fn, n_rounds: int, n_launches: int, warmup: int = 20):
    """The pages' kernel-only timing (hc_fused_gate.rs, timing section): `warmup` launches,
    then `n_rounds` rounds of `n_launches` back-to-back launches on `stream`, CUDA events
    around each round; per-launch means of the rounds and their median."""
    import torch
    for _ in range(warmup):
        fn()
    means = []
    for _ in range(n_rounds):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_launches):
            fn()
        e1.record(stream)
        stream.synchronize()
        means.append(e0.elapsed_time(e1) * 1e3 / n_launches)
    return {"us_median": statistics.median(means), "us_rounds": means,
            "desc": f"{warmup} warm-up, then {n_rounds} rounds of {n_launches} back-to-back launches; "
                    f"median of the rounds' per-launch means"}


def measure_cold(stream, fn, nbytes, peak, reps: int = 10):
    """One launch of `fn` with L2 flushed before it (a 256 MiB write, larger than the
    129 MB L2), so fn_w and everything else start in HBM: mean of `reps` event-timed
    launches, each after its own flush."""
    import torch
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    times = []
    for _ in range(reps + 1):
        with torch.cuda.stream(stream):
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        stream.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    us = statistics.mean(times[1:])
    del flush
    return {"us": us, "GB/s": nbytes / us / 1e3, "frac_hbm": nbytes / us / 1e3 / peak,
            "note": "L2 flushed (256 MiB write) before each launch: fn_w read from HBM"}


def measure_e2e(w, dev_in, dev_out, stream, K, run):
    """The same step through the C ABI with HOST buffers: pinned host -> device
    copies of the step's inputs (dev_in), the step (run(inputs, outputs) on
    `stream`), and the device -> host read of every output (dev_out), every step
    inside the timed region.  Steps are pipelined over two device buffer sets and
    three streams, as a serving loop would run them: step k+1's inputs are copied
    in and step k-1's outputs copied out while step k runs (host -> device and
    device -> host use separate copy engines)."""
    import torch
    dev = next(iter(dev_in.values())).device
    host_in = {k: v.cpu().pin_memory() for k, v in dev_in.items()}
    host_out = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in dev_out.items()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    sets = [(dev_in, dev_out),
            ({k: torch.empty_like(v) for k, v in dev_in.items()},
             {k: torch.empty_like(v) for k, v in dev_out.items()})]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in, ev_run, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def issue(k):
        b = k % 2
        d_in, d_out = sets[b]
        if k >= 2:   # this set's inputs are free once step k-2 has run
            s_in.wait_event(ev_run[b])
        with torch.cuda.stream(s_in):
            for key, v in d_in.items():
                v.copy_(host_in[key], non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if k >= 2:   # and its outputs once step k-2's have been copied out
            stream.wait_event(ev_out[b])
        run(d_in, d_out)
        ev_run[b].record(stream)
        s_out.wait_event(ev_run[b])
        with torch.cuda.stream(s_out):
            for key, v in d_out.items():
                host_out[key].copy_(v, non_blocking=True)
        ev_out[b].record(s_out)

    for k in range(2):
        issue(k)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for k in range(K):
        issue(k)
    e1.record(s_out)   # after the last copy-out, which follows every earlier step's work
    torch.cuda.synchronize(dev)
    sec = e0.elapsed_time(e1) / 1e3
    return {"value": w.T * K / sec, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * sec / K,
            "pipelining": "2 device buffer sets; copy-in, compute and copy-out streams"}


def measure_norm(w, y, stream, peak, reps: int = 20, pre_inputs=None):
    """The branch-input norm with its Q8_0 pair on the step's y, outside the timed step:
    mean of `reps` event-timed launches after 3 warm-up launches, of hc_rms_norm_q8 alone
    (algorithmic bytes: y read; z, q and the block scales written), and, with
    pre_inputs = (dv, ws), of the pre-chain with the norm (hc_pre_fused_norm, one launch
    on the cluster path) beside the pre-chain alone: their difference is what the norm
    adds to the site."""
    import torch
    from mhc_hyper_connection_hc_gb300 import hc
    T, d = y.shape
    if d % 32:
        return {"note": "d is not a multiple of 32: no Q8_0 pair"}
    with torch.cuda.stream(stream):
        norm_w = torch.from_numpy((1.0 + 0.25 * synth.branch_output(w.cid, 7, 1, d)[0]).astype(np.float32))
        norm_w = norm_w.to(y.device)   # 1 + 0.25 U[-1, 1), as the norm's parity tests
        z = torch.empty_like(y)
        q = torch.empty(T, d, dtype=torch.int8, device=y.device)
        qs = torch.empty(T, d // 32, dtype=torch.float32, device=y.device)

    def timed(fn):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in ev:
            e0.record(stream)
            fn()
            e1.record(stream)
        stream.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3

    us = timed(lambda: hc.hc_rms_norm_q8(y, norm_w, 1e-5, z, q, qs, stream=stream))
    nbytes = T * d * 4 + T * d * 4 + T * d + T * (d // 32) * 4
    gbs = nbytes / us / 1e3
    res = {"us": us, "algorithmic_bytes": nbytes, "GB/s": gbs, "frac_hbm": gbs / peak,
           "note": "rms_norm of y (eps 1e-5) and its Q8_0 pair, timed separately from the step"}
    if pre_inputs is not None:
        dv, ws = pre_inputs
        with torch.cuda.stream(stream):
            o = hc.new_pre_outputs(T, w.s, d, y.device)
        pre_us = timed(lambda: hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], w.iters, w.eps,
                                               o["pre"], o["post"], o["comb"], o["y"], ws, stream))
        def fused(path=None):
            hc.hc_pre_fused_norm(dv["x"], dv["fn_w"], dv["scale"], dv["base"], w.iters, w.eps, norm_w, 1e-5,
                                 o["pre"], o["post"], o["comb"], o["y"], z, ws, q=q, q_scale=qs, stream=stream,
                                 path=path)
        fz_us = timed(fused)
        fz_bytes = T * w.s * d * 4 + T * d * 4 * 2 + T * d + T * (d // 32) * 4   # x read; y, z, q, scales written
        res["pre_fused_norm"] = {
            "us": fz_us, "pre_alone_us": pre_us, "norm_adds_us": fz_us - pre_us,
            "separate_calls_us": pre_us + us, "algorithmic_bytes": fz_bytes,
            "GB/s": fz_bytes / fz_us / 1e3, "frac_hbm": fz_bytes / fz_us / 1e3 / peak,
            "note": ("hc_pre_fused_norm as called (HC_PATH_AUTO: one launch while the cluster path runs its "
                     "decode variant, else the pre-chain then the norm kernel)")}
        if hc.hc_pre_auto_path(T, w.s, d) == hc.HC_PATH_CLUSTER and (d // 16) % 32 == 0:
            res["pre_fused_norm"]["one_launch_us"] = timed(lambda: fused(hc.HC_PATH_CLUSTER))
    return res


def measure_head(w, dv, ws, stream, peak, reps: int = 20):
    """The gated-head trunk exit (hc_head) on the step's stream state, outside the
    timed step: mean of `reps` event-timed launches after 3 warm-up launches."""
    import torch
    from mhc_hyper_connection_hc_gb300 import hc
    T, s, d = w.T, w.s, w.d
    hw, hs, hb = synth.head_params(w.cid, s, d)
    with torch.cuda.stream(stream):
        hw, hs, hb = (torch.from_numpy(a).to(dv["x"].device) for a in (hw, hs, hb))
        gates = torch.empty(T, s, device=dv["x"].device)
        y = torch.empty(T, d, device=dv["x"].device)

    def head():
        hc.hc_head(dv["x"], hw, hs, hb, w.eps, y, ws, gates=gates, stream=stream)

    for _ in range(3):
        head()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in ev:
        e0.record(stream)
        head()
        e1.record(stream)
    stream.synchronize()
    if hc.hc_workspace_status(ws, stream) != 0:
        raise RuntimeError("the head kernel flagged an error")
    us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3
    nbytes = T * s * d * 4 + T * d * 4   # x read once, y written
    gbs = nbytes / us / 1e3
    # the head has no wide kernel: HC_PATH_AUTO runs the generic one for s > 4
    path = hc.HC_PATH_CLUSTER if hc.hc_pre_auto_path(T, s, d) == hc.HC_PATH_CLUSTER else hc.HC_PATH_GENERIC
    return {"us": us, "algorithmic_bytes": nbytes, "GB/s": gbs, "frac_hbm": gbs / peak,
            "path": "cluster" if path == hc.HC_PATH_CLUSTER else "generic",
            "note": "gated-head trunk exit on the same state, timed separately from the step"}


def measure_decode(dev, iters=None, n_sites: int = 300, cid: int = 1):
    """Latency of the site program at a small token count (the single-decode workload by
    default; cid=2 the verify batch, its two sites chained, each with its own fn_w): per
    site, pre-chain + hc_post, from a CUDA graph, and the same launches issued eagerly on a
    stream, both through the checked per-call binding and through Prepared calls (the
    arguments checked once), plus the pre-chain alone (iters: Sinkhorn iterations,
    default the workload's)."""
    import torch
    from mhc_hyper_connection_hc_gb300 import hc
    w = synth.WORKLOADS[cid]
    if iters is not None:
        w = dataclasses.replace(w, iters=iters)
    T, S, D = w.T, w.s, w.d
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        sites = []
        for k in range(w.sites):
            inp = synth.site_inputs(w.cid, T, S, D, w.x_dist, site=k)
            sites.append({n: torch.from_numpy(v).to(dev) for n, v in inp.items()})
        ws = hc.new_workspace(T, S, D, dev, stream)
        out = hc.new_pre_outputs(T, S, D, dev)
        xs = [sites[0]["x"]] + [torch.empty(T, S, D, device=dev) for _ in range(w.sites)]
    stream.synchronize()

    def site_calls(k, prepare=False):
        sk = sites[k]
        pre = hc.hc_pre_fused(xs[k], sk["fn_w"], sk["scale"], sk["base"], w.iters, w.eps, out["pre"],
                              out["post"], out["comb"], out["y"], ws, stream, prepare=prepare)
        post = hc.hc_post(xs[k], sk["f"], out["post"], out["comb"], xs[k + 1], stream, prepare=prepare)
        return pre, post

    def chain():
        for k in range(w.sites):
            site_calls(k)

    def pre_only():
        hc.hc_pre_fused(xs[0], sites[0]["fn_w"], sites[0]["scale"], sites[0]["base"], w.iters, w.eps, out["pre"],
                        out["post"], out["comb"], out["y"], ws, stream)

    prepared = [site_calls(k, prepare=True) for k in range(w.sites)]
    pre_p = prepared[0][0]
    with torch.cuda.stream(stream):
        norm_w = torch.ones(D, device=dev)
        z = torch.empty(T, D, device=dev)
        qn = torch.empty(T, D, dtype=torch.int8, device=dev)
        qsn = torch.empty(T, D // 32, device=dev)

    def pre_norm():
        hc.hc_pre_fused_norm(xs[0], sites[0]["fn_w"], sites[0]["scale"], sites[0]["base"], w.iters, w.eps, norm_w,
                             1e-5, out["pre"], out["post"], out["comb"], out["y"], z, ws, q=qn, q_scale=qsn,
                             stream=stream)

    def pre_then_norm():
        pre_only()
        hc.hc_rms_norm_q8(out["y"], norm_w, 1e-5, z, qn, qsn, stream=stream)

    def chain_prepared():
        for pre, post in prepared:
            pre()
            post()

    res = {"workload": workload_config(w)["workload"]}
    n_rep = max(1, n_sites // w.sites)
    for name, fn, per in (("site", chain, w.sites), ("pre", pre_only, 1),
                          ("site_prepared", chain_prepared, w.sites), ("pre_prepared", pre_p, 1),
                          ("pre_norm", pre_norm, 1), ("pre_then_norm", pre_then_norm, 1)):
        with torch.cuda.stream(stream):
            for _ in range(20):
                fn()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n_rep):
                fn()
            e1.record(stream)
            stream.synchronize()
            res[f"us_per_{name}_stream"] = e0.elapsed_time(e1) * 1e3 / (n_rep * per)
            if name.endswith("prepared"):
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(n_rep):
                    fn()
            g.replay()
            stream.synchronize()
            e0.record(stream)
            g.replay()
            e1.record(stream)
            stream.synchronize()
            res[f"us_per_{name}_graph"] = e0.elapsed_time(e1) * 1e3 / (n_rep * per)
    # single launch + synchronize wall (the pages' gate measured this way, with allocations)
    walls = []
    for _ in range(20):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        site_calls(0)
        stream.synchronize()
        walls.append((time.perf_counter() - t0) * 1e6)
    res["us_per_site_wall_sync"] = statistics.median(walls)
    cold = measure_cold(stream, pre_only, T * S * D * 4 + T * D * 4, 1.0)
    res["us_per_pre_l2_cold"] = cold["us"]
    res["l2_cold_note"] = "one pre-chain launch after a 256 MiB L2 flush: fn_w and x from HBM"
    res["stream_note"] = ("_stream: back-to-back eager calls, CUDA events around them (host cost per call "
                          "included when it exceeds the kernel's); _prepared: the same through Prepared calls; "
                          "pre_norm: hc_pre_fused_norm with the Q8_0 pair (one launch at this size), "
                          "pre_then_norm: hc_pre_fused then hc_rms_norm_q8")
    if hc.hc_workspace_status(ws, stream) != 0:
        raise RuntimeError("a kernel flagged an error in the latency measurement")
    res["iters"] = w.iters
    res["path"] = "cluster" if hc.hc_pre_auto_path(T, S, D) == hc.HC_PATH_CLUSTER else "generic"
    return res


STAMP_EVENTS = ("stage_ready", "dots_done", "shipped", "partials", "gates_sent", "pre_arrived", "collapsed",
                "refilled", "xf_start", "xf_landed", "xf_done", "sink_done", "kernel_start")
STAMP_TILES, STAMP_EV, STAMP_CTAS = 512, 16, 2


def run_stamps(args):
    """Per-phase timing of the pre kernel from its phase-stamp build (HC_STAMPS):
    %globaltimer stamps at every tile's phase boundaries (cluster kernel: CTAs 0 and 8 of
    cluster 0; wide kernel: CTA 0, and the reductions and finishes wherever they ran),
    for the pre-chain and the fused site boundary of the selected workload; medians over
    the tiles (the first two skipped) of each phase, in microseconds."""
    import torch
    from mhc_hyper_connection_hc_gb300 import build as lib_build, hc
    hc.load(lib_build.build(stamps=True))
    dev = torch.device("cuda", 0)
    w = selected_workload(args)
    T, s, d = w.T, w.s, w.d
    inp = synth.workload_inputs(w)
    dv = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    ws = hc.new_workspace(T, s, d, dev)
    out = hc.new_pre_outputs(T, s, d, dev)
    x_new = torch.empty(T, s, d, device=dev)
    hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], w.iters, w.eps, out["pre"], out["post"],
                    out["comb"], out["y"], ws)
    post_prev, comb_prev = out["post"].clone(), out["comb"].clone()
    base = 256   # stamps follow the 256-byte status block

    def read(fn):
        for _ in range(3):
            fn()
        hc.hc_workspace_init(ws)
        fn()
        torch.cuda.synchronize()
        if hc.hc_workspace_status(ws) != 0:
            raise RuntimeError("a kernel flagged an error")
        raw = ws[base:base + STAMP_CTAS * STAMP_TILES * STAMP_EV * 8].view(torch.int64)
        return raw.view(STAMP_CTAS, STAMP_TILES, STAMP_EV).cpu().numpy().astype(np.float64) / 1e3   # µs

    def med(vals):
        vals = [v for v in vals if np.isfinite(v)]
        return round(float(np.median(vals)), 3) if vals else None

    def analyse(st):
        E = {n: i for i, n in enumerate(STAMP_EVENTS)}
        t0 = st[0, 0, E["kernel_start"]]
        ntile = int(np.max(np.nonzero(st[0, :, E["stage_ready"]])[0])) + 1 if np.any(st[0, :, E["stage_ready"]]) else 0

        def ev(c, it, name):
            v = st[c, it, E[name]] if 0 <= it < STAMP_TILES else 0.0
            return v if v > 0 else np.nan

        rng = range(2, ntile) if ntile > 4 else range(0, ntile)
        res = {"tiles_stamped": ntile, "cta": "cluster 0, CTA 0 (owner of token 0 of every tile); "
                                              "compute phases are warpgroup 0's",
               "kernel_us": round(float(np.nanmax(st[0, :ntile, :12]) - t0), 3) if ntile else None,
               "first_stage_ready_us": round(float(ev(0, 0, "stage_ready") - t0), 3) if ntile else None}
        res["dots"] = med(ev(0, i, "dots_done") - ev(0, i, "stage_ready") for i in rng)
        res["reduce_and_ship"] = med(ev(0, i, "shipped") - ev(0, i, "dots_done") for i in rng)
        res["tile_period"] = med(ev(0, i, "stage_ready") - ev(0, i - 1, "stage_ready") for i in rng)
        res["wait_for_stage"] = med(ev(0, i, "stage_ready") - ev(0, i - 1, "shipped") for i in rng)
        res["shipped_to_owner_partials"] = med(ev(0, i, "partials") - ev(0, i, "shipped") for i in rng)
        res["owner_gates"] = med(ev(0, i, "gates_sent") - ev(0, i, "partials") for i in rng)
        res["shipped_to_pre_arrived"] = med(ev(0, i, "pre_arrived") - ev(0, i, "shipped") for i in rng)
        res["collapse"] = med(ev(0, i, "collapsed") - ev(0, i, "pre_arrived") for i in rng)
        res["collapse_period"] = med(ev(0, i, "collapsed") - ev(0, i - 1, "collapsed") for i in rng)
        res["refill_to_stage_ready"] = med(ev(0, i + 3, "stage_ready") - ev(0, i, "refilled") for i in rng)
        res["sinkhorn_after_gates"] = med(ev(0, i, "sink_done") - ev(0, i, "gates_sent") for i in rng)
        if np.any(st[0, :ntile, E["xf_done"]] > 0):
            res["transform_wait"] = med(ev(0, i, "xf_landed") - ev(0, i, "xf_start") for i in rng)
            res["transform"] = med(ev(0, i, "xf_done") - ev(0, i, "xf_landed") for i in rng)
            res["transform_done_to_stage_ready"] = med(ev(0, i, "stage_ready") - ev(0, i, "xf_done") for i in rng)
        return res

    def pre():
        hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], w.iters, w.eps, out["pre"], out["post"],
                        out["comb"], out["y"], ws)

    def boundary():
        hc.hc_post_pre_fused(dv["x"], dv["f"], post_prev, comb_prev, dv["fn_w"], dv["scale"], dv["base"], w.iters,
                             w.eps, x_new, out["pre"], out["post"], out["comb"], out["y"], ws)

    def analyse_wide(st):
        """The wide-stream kernel's stamps: slot 0 CTA 0 (compute warp 0, publisher, collapse
        warp); slot 1 the reduction of column 0 and the finish of every tile, whichever CTA
        did them."""
        E = {n: i for i, n in enumerate(STAMP_EVENTS)}
        t0 = st[0, 0, E["kernel_start"]]
        ntile = int(np.max(np.nonzero(st[0, :, E["stage_ready"]])[0])) + 1 if np.any(st[0, :, E["stage_ready"]]) else 0

        def ev(c, it, name):
            v = st[c, it, E[name]] if 0 <= it < STAMP_TILES else 0.0
            return v if v > 0 else np.nan

        rng = range(2, ntile) if ntile > 4 else range(0, ntile)
        ready = np.sort(st[0, :ntile, E["stage_ready"]])
        res = {"tiles_stamped": ntile,
               "kernel_us": round(float(np.nanmax(st[:, :ntile, :]) - t0), 3) if ntile else None,
               "first_stage_ready_us": round(float(ev(0, 0, "stage_ready") - t0), 3) if ntile else None}
        res["dots"] = med(ev(0, i, "dots_done") - ev(0, i, "stage_ready") for i in rng)
        res["reduce_and_ship"] = med(ev(0, i, "shipped") - ev(0, i, "dots_done") for i in rng)
        res["tile_period"] = med(ev(0, i, "stage_ready") - ev(0, i - 1, "stage_ready") for i in rng)
        res["wait_for_stage"] = med(ev(0, i, "stage_ready") - ev(0, i - 1, "shipped") for i in rng)
        res["shipped_to_published"] = med(ev(0, i, "partials") - ev(0, i, "shipped") for i in rng)
        res["shipped_to_refill_issued"] = med(ev(0, i, "refilled") - ev(0, i, "shipped") for i in rng)
        res["published_to_all_ctas_in"] = med(ev(1, i, "xf_start") - ev(0, i, "partials") for i in rng)
        res["column0_sum"] = med(ev(1, i, "xf_done") - ev(1, i, "xf_start") for i in rng)
        res["column0_sum_to_all_columns_in"] = med(ev(1, i, "xf_landed") - ev(1, i, "xf_done") for i in rng)
        res["all_columns_in_to_flag_set"] = med(ev(1, i, "gates_sent") - ev(1, i, "xf_landed") for i in rng)
        res["flag_set_to_seen_by_cta0"] = med(ev(0, i, "pre_arrived") - ev(1, i, "gates_sent") for i in rng)
        res["shipped_to_flag_seen"] = med(ev(0, i, "pre_arrived") - ev(0, i, "shipped") for i in rng)
        res["sinkhorn"] = med(ev(1, i, "sink_done") - ev(1, i, "gates_sent") for i in rng)
        res["collapse"] = med(ev(0, i, "collapsed") - ev(0, i, "pre_arrived") for i in rng)
        res["collapse_period"] = med(ev(0, i, "collapsed") - ev(0, i - 1, "collapsed") for i in rng)
        # how many tiles CTA 0's dot loop is ahead of its collapse
        res["collapse_lag_tiles"] = med(float(np.searchsorted(ready, ev(0, i, "collapsed")) - i)
                                        for i in rng if not np.isnan(ev(0, i, "collapsed")))
        res["last_collapse_after_last_ship_us"] = (
            round(float(np.nanmax(st[0, :ntile, E["collapsed"]]) - np.nanmax(st[0, :ntile, E["shipped"]])), 3)
            if ntile else None)
        return res

    wide = hc.hc_pre_auto_path(T, s, d) == hc.HC_PATH_WIDE
    an = analyse_wide if wide else analyse
    line = {"stamps": {"workload": workload_config(w)["workload"],
                       "unit": "µs, median over tiles", "path": "wide" if wide else "cluster",
                       "pre_chain": an(read(pre)), "fused_boundary": an(read(boundary))}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", choices=tuple(WORKLOAD_IDS), default="prefill")
    ap.add_argument("--iters", type=int, default=None, help="override the workload's Sinkhorn iterations")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (smaller cases for profiler captures)")
    ap.add_argument("--pipeline", choices=("fused", "separate"), default="fused",
                    help="a step is one site boundary: hc_post_pre_fused (fused) or hc_pre_fused + hc_post")
    ap.add_argument("--cpu-tokens", type=int, default=4096, help="tokens of the CPU-oracle sample")
    ap.add_argument("--ref-tokens", type=int, default=256, help="tokens per reference-arm step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-head", action="store_true", help="skip the gated-head exit measurement")
    ap.add_argument("--rounds", type=int, default=5, help="rounds of the per-kernel timing")
    ap.add_argument("--stamps", action="store_true",
                    help="per-phase timing from the phase-stamp build of the fused pre kernel (not a bench line)")
    ap.add_argument("--round-launches", type=int, default=300, help="back-to-back launches per round")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, _ = dist_env()
    if args.gpus != world and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        return run_reference(args)
    if args.stamps:
        return run_stamps(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
