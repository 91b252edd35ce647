"""Benchmark of batched draft verification on GB300.

Default workload: greedy MTP chain verification, B=64 requests, depth K=3,
V=128000, bf16 target logits [64, 4, 128000], T=0 (argmax matching with the
bonus token from the target argmax).  One step = one spec_verify_chain call
(one kernel launch: the row kernel with the fused cut) over one batch.

Timing: W warm-up steps, then exactly K steps replayed from CUDA graphs of
back-to-back calls, bracketed by a barrier and a device synchronise, timed
with CUDA events on the launching stream; max over ranks.  Inputs rotate over
enough device copies that the bytes touched between two uses of a copy exceed
4x the L2.  `e2e` repeats the metric through the Python API with pinned host
buffers: each step copies its inputs host->device, verifies, and reads the
result back.

`--impl reference` times the float64 CPU oracle on host cores instead (a
bounded sample of the same workload per step).

Multi-GPU (torchrun): replicas only -- every rank verifies its own batch, no
collective on the data path (weak scaling); value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/sec and achieved HBM GB/s vs 8 TB/s at V=128000, 1 GB300"
UNIT = "verified draft tokens/s"
# The kernel that dominates each kind of step, the sources that define it (and its launch), and
# the committed file with its ncu DRAM traffic, valid only while those sources are unchanged.
KERNELS = {
    "greedy": {"name": "sv::argmax_kernel<bf16> (argmax + fused cut, one launch)",
               "sources": ["argmax_kernel.cuh", "spec_device.cuh", "spec_internal.h", "budget_cut.cu", "api.cu"],
               "traffic": os.path.join(ROOT, "profiles", "argmax_kernel_traffic.txt")},
    "sampling": {"name": "sv::sample_kernel<bf16> (+ sv::cut_kernel / budget_cut_kernel, PDL-chained)",
                 "sources": ["sample_kernel.cuh", "spec_async.cuh", "spec_device.cuh", "spec_internal.h", "row_bf16.cu", "api.cu"],
                 "traffic": os.path.join(ROOT, "profiles", "stream_kernel_traffic.txt")},
}


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a host float over ranks (identity at world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index, self.period = index, period_ms
        self.samples = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line.strip()))

    def mark(self, on: bool):
        if on:
            self.t_on = time.perf_counter()
        else:
            self.t_off = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for t, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            rows.append((t, parts))
        inside = [p for t, p in rows if self.t_on is not None and self.t_on <= t <= (self.t_off or t)]
        used = inside if inside else [p for _, p in rows]
        sm = sorted(float(p[0]) for p in used if _isnum(p[0]))
        smax = [float(p[1]) for p in used if _isnum(p[1])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in used for i in range(4) if p[3 + i].lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "samples_total": len(rows)}


def _isnum(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


# ---------------------------------------------------------------- workloads

def make_workload(name: str, rank: int):
    import workloads as W
    if name == "greedy_mtp":
        return W.greedy_mtp(seed=1 + 100 * rank)
    if name == "stochastic_mtp":
        return W.stochastic_mtp(seed=2 + 100 * rank)
    if name == "dfly_block":
        return W.dfly_block(seed=3 + 100 * rank)
    if name.startswith("budget_sweep"):
        B = int(name.split("_B")[-1]) if "_B" in name else 64
        return W.budget_sweep(B, seed=4 + 100 * rank)
    if name == "tiny_chain":
        return W.tiny_chain(seed=0 + 100 * rank)
    raise ValueError(name)


def call_kind(w, name):
    """(entry point, reads draft?) for a workload, matching its configuration."""
    if name == "greedy_mtp":
        return "chain", False
    if name in ("stochastic_mtp", "tiny_chain"):
        return "chain", True
    return "block", True


def algorithmic_bytes(w, reads_draft: bool) -> int:
    """Bytes the outputs depend on: logits read once + ids/uniforms read + outputs written."""
    e = w.target.element_size()
    B, K, V = w.B, w.K, w.V
    b = B * (K + 1) * V * e + (B * K * V * e if reads_draft else 0)
    b += B * K * 4 + (B * (K + 1) * 4 if w.temperature > 0 else 0)
    b += B * (K + 1) * 4 + B * 4
    return b


def kernel_source_hash(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNELS[kind]["sources"]:
        with open(os.path.join(ROOT, "draft_verification_spec_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind: str, config_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel."""
    path = KERNELS[kind]["traffic"]
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if "=" in line and not line.lstrip().startswith("#"):
            k, v = line.split("=", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash(kind):
        return None
    key = f"{config_name}.dram_bytes_per_launch"
    return int(float(vals[key])) if key in vals else None


# ---------------------------------------------------------------- GPU arm

class DeviceRunner:
    """Device-resident copies of one workload and a CUDA graph of back-to-back calls."""

    def __init__(self, w, name, device, min_bytes):
        import torch
        import draft_verification_spec_gb300 as sv
        self.sv, self.torch, self.w, self.name, self.dev = sv, torch, w, name, device
        self.kind, self.reads_draft = call_kind(w, name)
        per = w.target.numel() * w.target.element_size() + (
            w.draft.numel() * w.draft.element_size() if self.reads_draft else 0)
        self.nsets = max(1, math.ceil(min_bytes / per))
        self.sets = []
        for _ in range(self.nsets):
            t = w.target.to(device)
            d = w.draft.to(device) if self.reads_draft else None
            self.sets.append((t, d, w.tokens.to(device), w.uniforms.to(device)))
        B, K = w.B, w.K
        f = lambda *s: torch.empty(*s, dtype=torch.float32, device=device)  # noqa: E731
        i = lambda *s: torch.empty(*s, dtype=torch.int32, device=device)  # noqa: E731
        block = self.kind == "block"
        self.out = sv.VerifyOutput(i(B, K + 1), i(B), f(B, K) if block else None, f(B, K) if block else None,
                                   f(B) if block else None, i(B) if w.budget is not None else None)
        self.stream = torch.cuda.Stream(device)
        self.ws = sv.Workspace(device)
        self.bytes_per_step = algorithmic_bytes(w, self.reads_draft)
        self.greedy_fused = w.temperature == 0 and w.budget is None
        self.kernel_kind = "greedy" if w.temperature == 0 else "sampling"
        self.graphs = {}

    def step(self, i, tuning=None):
        t, d, x, u = self.sets[i % self.nsets]
        w, sv = self.w, self.sv
        if self.kind == "chain":
            sv.verify_chain(t, d, x, u, w.temperature, want_alpha=False, stream=self.stream,
                            workspace=self.ws, out=self.out, tuning=tuning)
        else:
            sv.verify_block(t, d, x, u, w.temperature, budget=w.budget, want_stats=True,
                            stream=self.stream, workspace=self.ws, out=self.out, tuning=tuning)

    def launches_per_step(self):
        # greedy without a budget: one argmax kernel with the cut fused in; otherwise the row
        # kernel, then the cut (or budget + cut) kernel chained to it
        return 1 if self.greedy_fused else 2

    def graph(self, n):
        torch = self.torch
        if n not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                self.step(0)                       # populate the library's per-kernel caches
            self.stream.synchronize()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    self.step(i)
            self.graphs[n] = g
        return self.graphs[n]

    def run(self, steps, chunk=500):
        """Replay exactly `steps` calls; returns elapsed ms from CUDA events on the stream."""
        torch = self.torch
        full, rem = divmod(steps, chunk)
        g_full = self.graph(chunk) if full else None
        g_rem = self.graph(rem) if rem else None
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            start.record(self.stream)
            for _ in range(full):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            stop.record(self.stream)
        stop.synchronize()
        return start.elapsed_time(stop)


def run_gpu(args, rank, local_rank, world):
    import torch
    import draft_verification_spec_gb300 as sv
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    sv.lib()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 * 2 ** 20)
    min_bytes = 4 * l2 + 1

    w = make_workload(args.config, rank)
    r = DeviceRunner(w, args.config, dev, min_bytes)
    # warm-up (untimed)
    r.run(args.warmup, chunk=max(1, min(args.warmup, 500)))
    torch.cuda.synchronize()
    tuning = sv.Tuning()
    with torch.cuda.stream(r.stream):
        r.step(0, tuning=tuning)
    torch.cuda.synchronize()
    plan = tuning.plan
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    ms = r.run(args.steps)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    ms_max = max_over_ranks(ms, world, dev)
    per_step_ms = ms_max / args.steps
    tokens_per_step = w.B * w.K
    value = sum_over_ranks(tokens_per_step * args.steps, world, dev) / (ms_max / 1e3)

    # roofline of the (only) kernel of the step: algorithmic bytes / average duration
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else None
    peak_gbs, peak_src = (peaks["hbm_gbs"], "measured") if peaks else (6800.0, "fallback")
    # the dominant kernel's average duration: with one launch per step it is the step time on
    # the launching stream; with two, the step time is an upper bound (the chained cut kernel is
    # a few microseconds and overlaps the row kernel's tail), so `achieved` is a lower bound
    launch_ms = ms / args.steps
    achieved = r.bytes_per_step / (launch_ms / 1e3) / 1e9

    # end to end: pinned host inputs -> device, verify, result -> host, every step
    e2e = run_e2e(w, args, dev, world) if not args.no_e2e else None

    extra = {}
    if rank == 0 and not args.no_extra and world == 1:
        for name in args.extra:
            try:
                wx = make_workload(name, 0)
                rx = DeviceRunner(wx, name, dev, min_bytes)
                rx.run(5, chunk=5)
                nsteps = args.extra_steps
                msx = rx.run(nsteps)
                t = msx / nsteps / 1e3
                bx = rx.bytes_per_step
                extra[name] = {"tokens_per_s": wx.B * wx.K / t, "rows_per_s": wx.B * (2 * wx.K + 1) / t,
                               "us_per_step": t * 1e6, "logit_bytes": wx.logits_bytes(rx.reads_draft),
                               "achieved_gbs": bx / t / 1e9, "frac_of_measured_hbm": bx / t / 1e9 / peak_gbs,
                               "launches_per_step": rx.launches_per_step(), "kernel": KERNELS[rx.kernel_kind]["name"],
                               "traffic": profiled_traffic(rx.kernel_kind, name)}
                del rx
                torch.cuda.empty_cache()
            except Exception as ex:  # a secondary measurement never hides the main line
                extra[name] = {"error": repr(ex)[:200]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = run_cpu_baseline(w, args.cpu_seconds)

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.target.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded; shapes and distributions of the verification configurations)",
        "config": {"workload": f"{args.config} B={w.B} K={w.K} V={w.V} "
                               f"{'bf16' if w.target.dtype == torch.bfloat16 else 'fp32'} T={w.temperature}",
                   "B": w.B, "K": w.K, "V": w.V, "temperature": w.temperature, "entry": f"spec_verify_{r.kind}",
                   "reads_draft": r.reads_draft, "parallelism": f"replicas x{world}",
                   "l2": f"inputs rotate over {r.nsets} device copies ({r.nsets * w.logits_bytes(r.reads_draft) / 1e6:.0f} MB > 4x L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA graphs of back-to-back calls, CUDA events on the launching stream",
                   "plan": plan},
        "rows_per_s": value / max(w.K, 1) * (2 * w.K + 1) if r.reads_draft else value / max(w.K, 1) * (w.K + 1),
        "achieved_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
                     "frac": achieved / peak_gbs, "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
                     "traffic": profiled_traffic(r.kernel_kind, args.config),
                     "algorithmic_bytes_per_launch": r.bytes_per_step,
                     "launch_ms": launch_ms, "kernel": KERNELS[r.kernel_kind]["name"],
                     "launches_per_step": r.launches_per_step(),
                     "note": ("one launch per step: launch_ms is the step time on the launching stream"
                              if r.launches_per_step() == 1 else
                              "two launches per step: launch_ms is the whole step, so achieved is a lower bound")},
        "gpu_launches": args.steps * r.launches_per_step(),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "configs": extra,
    }
    return line


def run_e2e(w, args, dev, world):
    """Same metric through the public API with host buffers; copies inside the timed region."""
    import torch
    import draft_verification_spec_gb300 as sv
    kind, reads_draft = call_kind(w, args.config)
    h_t = w.target.pin_memory()
    h_d = w.draft.pin_memory() if reads_draft else None
    h_x = w.tokens.pin_memory()
    h_u = w.uniforms.pin_memory() if w.temperature > 0 else None
    d_t = torch.empty_like(w.target, device=dev)
    d_d = torch.empty_like(w.draft, device=dev) if reads_draft else None
    d_x = torch.empty_like(w.tokens, device=dev)
    d_u = torch.empty_like(w.uniforms, device=dev) if h_u is not None else None
    h_tok = torch.empty(w.B, w.K + 1, dtype=torch.int32).pin_memory()
    h_acc = torch.empty(w.B, dtype=torch.int32).pin_memory()
    s = torch.cuda.Stream(dev)
    ws = sv.Workspace(dev)
    steps = max(1, min(args.steps, args.e2e_steps))

    def one():
        d_t.copy_(h_t, non_blocking=True)
        if d_d is not None:
            d_d.copy_(h_d, non_blocking=True)
        d_x.copy_(h_x, non_blocking=True)
        if d_u is not None:
            d_u.copy_(h_u, non_blocking=True)
        if kind == "chain":
            out = sv.verify_chain(d_t, d_d, d_x, d_u, w.temperature, stream=s, workspace=ws)
        else:
            out = sv.verify_block(d_t, d_d, d_x, d_u, w.temperature, budget=w.budget, stream=s, workspace=ws)
        h_tok.copy_(out.tokens, non_blocking=True)
        h_acc.copy_(out.accepted, non_blocking=True)

    with torch.cuda.stream(s):
        for _ in range(3):
            one()
    s.synchronize()
    barrier(world)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        start.record(s)
        for _ in range(steps):
            one()
        stop.record(s)
    stop.synchronize()
    ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    tokens = sum_over_ranks(w.B * w.K * steps, world, dev)
    h2d = h_t.numel() * h_t.element_size() + (h_d.numel() * h_d.element_size() if h_d is not None else 0) + \
        h_x.numel() * 4 + (h_u.numel() * 4 if h_u is not None else 0)
    d2h = h_tok.numel() * 4 + h_acc.numel() * 4
    return {"value": tokens / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": ms / steps,
            "path": "pinned host -> device copy, verify_chain/verify_block (Python API), result -> host"}


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

def oracle_step(w, reqs):
    import numpy as np
    from oracle import spec_oracle as O
    zt = w.target[reqs].to(dtype=__import__("torch").float64).numpy()
    zd = None if (w.temperature == 0 and w.budget is None) else w.draft[reqs].to(
        dtype=__import__("torch").float64).numpy()
    d = None
    if w.budget is not None:
        a, _, _ = O.overlap_stats(zt, zd, w.temperature)
        d = O.alloc_budget(a, max(1, w.budget * len(range(*reqs.indices(w.B))) // w.B)).depth
    return O.verify(zt, zd, w.tokens[reqs].numpy(), w.uniforms[reqs].double().numpy(), w.temperature,
                    depth=d, need_alpha=w.temperature > 0)


def run_cpu_baseline(w, seconds: float):
    """The oracle as it stands, single process, on a bounded sample: whole passes over the batch."""
    n_req = w.B
    t0 = time.perf_counter()
    passes = 0
    while True:
        for s in range(0, w.B, 8):
            oracle_step(w, slice(s, min(w.B, s + 8)))
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    cores = _threads_used()
    return {"value": passes * n_req * w.K / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{passes} full pass(es) over the {w.B}-request batch in {dt:.1f} s (numpy float64)",
            "cpu": _cpu_model()}


def _threads_used() -> int:
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return 1   # the oracle's vocabulary reductions (max, exp, sum, cumsum, argmax) are single-threaded numpy


def _cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = make_workload(args.config, 0)
    # size the per-step sample so the whole run stays within a few minutes
    t0 = time.perf_counter()
    oracle_step(w, slice(0, 1))
    per_req = time.perf_counter() - t0
    budget_s = 150.0
    n_req = int(max(1, min(w.B, budget_s / max(1, args.steps + args.warmup) / max(per_req, 1e-6))))
    for i in range(args.warmup):
        oracle_step(w, slice(i % w.B, i % w.B + 1))
    t0 = time.perf_counter()
    for i in range(args.steps):
        s = (i * n_req) % w.B
        oracle_step(w, slice(s, min(w.B, s + n_req)))
    dt = time.perf_counter() - t0
    done = sum(min(w.B, (i * n_req) % w.B + n_req) - (i * n_req) % w.B for i in range(args.steps))
    value = done * w.K / dt
    cores = _threads_used()
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": f"{args.config} B={w.B} K={w.K} V={w.V} T={w.temperature}"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{n_req} request(s) of the {w.B}-request batch per step",
                             "cpu": _cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- main

def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="greedy_mtp")
    ap.add_argument("--extra", nargs="*", default=["stochastic_mtp", "dfly_block", "budget_sweep_B4",
                                                   "budget_sweep_B16", "budget_sweep_B64"])
    ap.add_argument("--extra-steps", type=int, default=3000)
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    return a


def main(argv=None):
    args = parse(argv)
    rank, local_rank, world = dist_env()
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    if args.impl == "reference":
        if world > 1:
            init_dist(world, "gloo")
        line = run_reference(args, rank, world)
    else:
        init_dist(world, "nccl")
        line = run_gpu(args, rank, local_rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
