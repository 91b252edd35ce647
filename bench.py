"""Benchmark of batched draft verification on GB300.

Default workload: the batch-level budgeted verification sweep at its largest
concurrency, B=64 requests, DFly blocks of K=16, V=128000, bf16 logits
[64, 17, 128000] (target) and [64, 16, 128000] (draft), T=0.9, budget N=8B:
every position's alpha, the global top-N prefix choice, then verification to
the chosen depths (540.7 MB of logits per call).  One step = one
spec_verify_block call (the streaming row kernel, then the budget-and-cut
kernel chained to it) over one batch.  The verified draft tokens of a step are
the N positions the budget spends.  The other verification configurations
(greedy and stochastic MTP chains, DFly block, smaller budget sweeps) are
measured as secondary lines under "configs".

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
    "draft": {"name": "sv::draft_stats_kernel<bf16> (then sv::budget_cut_kernel, PDL-chained)",
              "sources": ["draft_conf.cu", "packed_math.cuh", "spec_device.cuh", "spec_internal.h", "api.cu"],
              "traffic": os.path.join(ROOT, "profiles", "draft_stats_kernel_traffic.txt")},
    "sampling": {"name": "sv::sample_kernel<bf16> (then sv::cut_kernel / sv::budget_cut_kernel, PDL-chained)",
                 "sources": ["sample_kernel.cuh", "spec_async.cuh", "spec_device.cuh", "spec_internal.h", "row_bf16.cu", "api.cu"],
                 "traffic": os.path.join(ROOT, "profiles", "sample_kernel_traffic.txt")},
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
    if name.startswith("budget_sweep") or name.startswith("draft_budget"):
        # draft_budget*: the budget sweep's draft rows, the budget chosen before the target runs
        B = int(name.split("_B")[-1]) if "_B" in name else 64
        return W.budget_sweep(B, seed=4 + 100 * rank)
    if name == "tiny_chain":
        return W.tiny_chain(seed=0 + 100 * rank)
    raise ValueError(name)


def call_kind(w, name):
    """(entry point, reads draft?) for a workload, matching its configuration."""
    if name.startswith("draft_budget_adaptive"):
        return "draft_adaptive", True
    if name.startswith("draft_budget"):
        return "draft", True
    if name == "greedy_mtp":
        return "chain", False
    if name in ("stochastic_mtp", "tiny_chain"):
        return "chain", True
    return "block", True


def verified_tokens(w) -> int:
    """Draft positions a step verifies: the budget's N, else every drafted position."""
    return min(w.budget, w.B * w.K) if w.budget is not None else w.B * w.K


def algorithmic_bytes(w, reads_draft: bool, kind: str = "") -> int:
    """Bytes the outputs depend on: logits read once + ids/uniforms read + outputs written."""
    if kind.startswith("draft"):
        # the draft rows once, the drafted tokens, depth, prefix confidences and N
        return w.B * w.K * w.V * w.draft.element_size() + w.B * w.K * 4 + w.B * 4 + w.B * w.K * 4 + 4
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
        import workloads as W
        self.kind, self.reads_draft = call_kind(w, name)
        self.draft_only = self.kind.startswith("draft")
        per = (0 if self.draft_only else w.target.numel() * w.target.element_size()) + (
            w.draft.numel() * w.draft.element_size() if self.reads_draft else 0)
        self.logit_bytes = per
        self.nsets = max(1, math.ceil(min_bytes / per))
        self.sets = []
        for _ in range(self.nsets):
            t = None if self.draft_only else w.target.to(device)
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
        self.bytes_per_step = algorithmic_bytes(w, self.reads_draft, self.kind)
        self.greedy_fused = w.temperature == 0 and w.budget is None
        self.kernel_kind = "draft" if self.draft_only else ("greedy" if w.temperature == 0 else "sampling")
        if self.draft_only:
            self.dout = (torch.zeros(1, dtype=torch.int32, device=device), i(B), f(B, K))
            cn, ct = W.verify_cost_table(B, K)
            self.cost = (torch.tensor(cn, dtype=torch.float32, device=device),
                         torch.tensor(ct, dtype=torch.float32, device=device)) if self.kind == "draft_adaptive" else None
        self.graphs = {}

    def step(self, i, tuning=None):
        t, d, x, u = self.sets[i % self.nsets]
        w, sv = self.w, self.sv
        if self.draft_only:
            sv.draft_budget(d, x, w.temperature, budget=None if self.cost else w.budget, cost=self.cost,
                            stream=self.stream, workspace=self.ws, out=self.dout)
        elif self.kind == "chain":
            sv.verify_chain(t, d, x, u, w.temperature, want_alpha=False, stream=self.stream,
                            workspace=self.ws, out=self.out, tuning=tuning)
        else:
            sv.verify_block(t, d, x, u, w.temperature, budget=w.budget, want_stats=True,
                            stream=self.stream, workspace=self.ws, out=self.out, tuning=tuning)

    def split(self, n=200):
        """Average device time (us) of the row kernel and of the kernel chained after it, from CUDA
        events on the launching stream: start, the library's split event between the two launches,
        stop (the chained kernel then runs without programmatic dependent launch)."""
        torch = self.torch
        if self.greedy_fused or self.draft_only:
            return None
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(self.stream):
            for a, m, b in ev:
                m.record(self.stream)               # creates the event before its handle is passed
        self.stream.synchronize()
        with torch.cuda.stream(self.stream):
            for i, (a, m, b) in enumerate(ev):
                a.record(self.stream)
                self.step(i, tuning=self.sv.Tuning(split_event=m))
                b.record(self.stream)
        self.stream.synchronize()
        row = sum(a.elapsed_time(m) for a, m, _ in ev) / n * 1e3
        cut = sum(m.elapsed_time(b) for _, m, b in ev) / n * 1e3
        return {"row_kernel_us": row, "chained_kernel_us": cut, "calls": n,
                "how": "per-call CUDA events around a plain (ungraphed) loop, split event recorded by the "
                       "library between the two launches"}

    def decisions(self):
        """One call with every statistic requested: realised mean alpha and accepted length."""
        torch, sv, w = self.torch, self.sv, self.w
        t, d, x, u = self.sets[0]
        if self.draft_only:
            return None
        with torch.cuda.stream(self.stream):
            if self.kind == "chain":
                out = sv.verify_chain(t, w.draft.to(self.dev) if d is None and w.K > 0 else d, x, u, w.temperature,
                                      want_alpha=True, stream=self.stream, workspace=self.ws)
            else:
                out = sv.verify_block(t, d, x, u, w.temperature, budget=w.budget, want_stats=True,
                                      stream=self.stream, workspace=self.ws)
        self.stream.synchronize()
        return out

    def tokens_per_step(self):
        """Positions a step selects for verification: the N of the last call for the adaptive
        draft-side budget, else verified_tokens."""
        if self.kind == "draft_adaptive":
            self.stream.synchronize()
            return int(self.dout[0].item())
        return verified_tokens(self.w)

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
    tokens_per_step = verified_tokens(w)
    value = sum_over_ranks(tokens_per_step * args.steps, world, dev) / (ms_max / 1e3)

    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else None
    peak_gbs, peak_src = (peaks["hbm_gbs"], "measured") if peaks else (6800.0, "fallback")
    step_ms = ms / args.steps
    # roofline of the dominant kernel: algorithmic bytes / its average duration.  With one launch
    # per step that is the step time; with two, the row kernel's own time from the split loop.
    split = r.split() if rank == 0 else None
    launch_ms = step_ms if split is None else split["row_kernel_us"] / 1e3
    achieved = r.bytes_per_step / (launch_ms / 1e3) / 1e9
    step_gbs = r.bytes_per_step / (step_ms / 1e3) / 1e9
    dec_out = r.decisions() if rank == 0 else None
    decisions = decision_stats(w, dec_out, step_ms / 1e3) if rank == 0 else None

    # end to end: pinned host inputs -> device, verify, result -> host, every step
    e2e = run_e2e(w, args, dev, world) if not args.no_e2e else None

    extra = {}
    if rank == 0 and not args.no_extra and world == 1:
        for name in args.extra:
            if name == args.config:
                continue
            try:
                wx = make_workload(name, 0)
                rx = DeviceRunner(wx, name, dev, min_bytes)
                rx.run(5, chunk=5)
                nsteps = args.extra_steps
                msx = rx.run(nsteps)
                t = msx / nsteps / 1e3
                bx = rx.bytes_per_step
                sx = rx.split(100)
                tk = sx["row_kernel_us"] / 1e6 if sx else t
                extra[name] = {"verified_tokens_per_s": rx.tokens_per_step() / t,
                               "drafted_tokens_per_s": wx.B * wx.K / t,
                               "rows_per_s": wx.B * (wx.K if rx.draft_only else 2 * wx.K + 1) / t,
                               "us_per_step": t * 1e6, "tokens_per_step": rx.tokens_per_step(),
                               "logit_bytes": rx.logit_bytes,
                               "algorithmic_bytes": bx,
                               "achieved_gbs_step": bx / t / 1e9, "frac_of_measured_hbm_step": bx / t / 1e9 / peak_gbs,
                               "achieved_gbs_kernel": bx / tk / 1e9, "frac_of_measured_hbm_kernel": bx / tk / 1e9 / peak_gbs,
                               "split": sx, "launches_per_step": rx.launches_per_step(),
                               "kernel": KERNELS[rx.kernel_kind]["name"],
                               "traffic": profiled_traffic(rx.kernel_kind, name),
                               "decisions": decision_stats(wx, rx.decisions(), t)}
                del rx
                torch.cuda.empty_cache()
            except Exception as ex:  # a secondary measurement never hides the main line
                extra[name] = {"error": repr(ex)[:200]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = run_cpu_baseline(w, args.cpu_seconds, dec_out)
        if decisions is not None and cpu is not None:
            decisions["oracle_agreement"] = cpu.pop("agreement", None)

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.target.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded; shapes and distributions of the verification configurations)",
        "config": {"workload": f"{args.config} B={w.B} K={w.K} V={w.V} "
                               f"{'bf16' if w.target.dtype == torch.bfloat16 else 'fp32'} T={w.temperature}"
                               + (f" N={w.budget}" if w.budget is not None else ""),
                   "B": w.B, "K": w.K, "V": w.V, "temperature": w.temperature, "budget_N": w.budget,
                   "entry": f"spec_verify_{r.kind}", "reads_draft": r.reads_draft,
                   "verified_tokens_per_step": tokens_per_step, "parallelism": f"replicas x{world}",
                   "l2": f"inputs rotate over {r.nsets} device copies ({r.nsets * w.logits_bytes(r.reads_draft) / 1e6:.0f} MB > 4x L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA graphs of back-to-back calls, CUDA events on the launching stream",
                   "plan": plan},
        "rows_per_s": w.B * (2 * w.K + 1 if r.reads_draft else w.K + 1) / (per_step_ms / 1e3),
        "achieved_gbs": step_gbs,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
                     "frac": achieved / peak_gbs, "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
                     "traffic": profiled_traffic(r.kernel_kind, args.config),
                     "algorithmic_bytes_per_launch": r.bytes_per_step,
                     "launch_ms": launch_ms, "kernel": KERNELS[r.kernel_kind]["name"],
                     "launches_per_step": r.launches_per_step(),
                     "step_ms": step_ms, "step_achieved": step_gbs, "step_frac": step_gbs / peak_gbs,
                     "split": split,
                     "note": ("one launch per step: launch_ms is the step time on the launching stream"
                              if split is None else
                              "launch_ms is the row kernel's average device time from the split loop; "
                              "step_* divide by the whole step (row kernel + chained kernel)")},
        "decisions": decisions,
        "gpu_launches": args.steps * r.launches_per_step(),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "configs": extra,
    }
    return line


def decision_stats(w, out, step_s):
    """Realised statistics of one call's decisions (GPU outputs only)."""
    if out is None:
        return None
    acc = out.accepted.double().cpu()
    st = {"mean_accepted": float(acc.mean()), "mean_emitted": float(acc.mean()) + 1.0,
          "acceptance_rate": float(acc.sum()) / max(1, (int(out.depth.sum()) if out.depth is not None
                                                        else w.B * w.K)),
          "accepted_tokens_per_s": float(acc.sum()) / step_s}
    if out.alpha is not None and w.K > 0:
        st["mean_alpha"] = float(out.alpha.double().mean())
    if out.expected_len is not None:
        st["mean_expected_accepted"] = float(out.expected_len.double().mean())
    if out.depth is not None:
        st["mean_depth"] = float(out.depth.double().mean())
    return st


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

def oracle_pass(w, depth=None, chunk=8):
    """The float64 oracle over the whole batch (requests in chunks): alpha and the global budget
    when the workload has one, then the decisions at depth (the budget's, or the one given)."""
    import numpy as np
    import torch
    from oracle import spec_oracle as O
    up = lambda t: t.to(dtype=torch.float64).numpy()  # noqa: E731
    need_draft = not (w.temperature == 0 and w.budget is None)
    if w.budget is not None and depth is None:
        a = np.concatenate([O.overlap_stats(up(w.target[s:s + chunk]), up(w.draft[s:s + chunk]), w.temperature)[0]
                            for s in range(0, w.B, chunk)])
        depth = O.alloc_budget(a, w.budget).depth
    parts = []
    for s in range(0, w.B, chunk):
        e = min(w.B, s + chunk)
        parts.append(O.verify(up(w.target[s:e]), up(w.draft[s:e]) if need_draft else None, w.tokens[s:e].numpy(),
                              w.uniforms[s:e].double().numpy(), w.temperature,
                              depth=None if depth is None else np.asarray(depth)[s:e],
                              need_alpha=w.temperature > 0))
    return parts


def agreement(w, parts, gpu_out):
    """Requests whose oracle decision margin is below 1e-5 (ambiguous), and disagreements among the
    others (bit-exact expected)."""
    import numpy as np
    tok = np.concatenate([p.tokens for p in parts])
    acc = np.concatenate([p.accepted for p in parts])
    margin = np.concatenate([p.margin for p in parts])
    g_tok = gpu_out.tokens.cpu().numpy()
    g_acc = gpu_out.accepted.cpu().numpy()
    amb = margin < 1e-5
    differ = (g_acc != acc) | np.any(g_tok != tok, axis=1)
    return {"requests": int(w.B), "ambiguous": int(amb.sum()), "unambiguous_mismatches": int((differ & ~amb).sum()),
            "ambiguous_mismatches": int((differ & amb).sum()), "margin_threshold": 1e-5}


def run_cpu_baseline(w, seconds: float, gpu_out=None):
    """The oracle as it stands, single process, on a bounded sample: whole passes over the batch.
    The first pass runs at the GPU's chosen depths and is compared with the GPU's decisions."""
    t0 = time.perf_counter()
    agree = None
    if gpu_out is not None:
        depth = gpu_out.depth.cpu().numpy() if gpu_out.depth is not None else None
        agree = agreement(w, oracle_pass(w, depth=depth), gpu_out)
    passes = 1 if gpu_out is not None else 0
    while passes == 0 or time.perf_counter() - t0 < seconds:
        oracle_pass(w)
        passes += 1
    dt = time.perf_counter() - t0
    cores = _threads_used()
    line = {"value": passes * verified_tokens(w) / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{passes} full pass(es) over the {w.B}-request batch in {dt:.1f} s (numpy float64)",
            "cpu": _cpu_model()}
    if agree is not None:
        line["agreement"] = agree
    return line


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
    # size the per-step sample so the whole run (warm-up included) stays within a few minutes:
    # whole requests while they fit, else the first m drafted positions of one request (down to
    # one (target, draft) row pair); a pair stands for its share of the batch's verified tokens
    budget_s = 150.0
    per_step = budget_s / max(1, args.steps + args.warmup)
    pairs_total = max(1, w.B * w.K)
    tokens_per_pair = verified_tokens(w) / pairs_total
    t0 = time.perf_counter()
    oracle_pass(_subset(w, 1))
    per_req = time.perf_counter() - t0
    if per_req <= per_step or w.K == 0:
        n_req = int(max(1, min(w.B, per_step / max(per_req, 1e-6))))
        sub, pairs, what = _subset(w, n_req), n_req * max(1, w.K), f"{n_req} request(s) of the {w.B}-request batch"
    else:
        t0 = time.perf_counter()
        oracle_pass(_prefix(w, 1))
        per_pair = time.perf_counter() - t0
        m = int(max(1, min(w.K, per_step / max(per_pair, 1e-6))))
        sub, pairs, what = _prefix(w, m), m, f"the first {m} of {w.K} drafted position(s) of one request"
    for _ in range(args.warmup):
        oracle_pass(sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(sub)
    dt = time.perf_counter() - t0
    value = args.steps * pairs * tokens_per_pair / dt
    cores = _threads_used()
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": f"{args.config} B={w.B} K={w.K} V={w.V} T={w.temperature}"
                                   + (f" N={w.budget}" if w.budget is not None else "")},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{what} per step ({tokens_per_pair:g} verified token(s) per "
                                       f"drafted position, the batch's share)",
                             "cpu": _cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _prefix(w, m):
    """Request 0 of a workload cut to its first m drafted positions (its budget scaled to them)."""
    import workloads as W
    b = None if w.budget is None else max(1, w.budget * m // max(1, w.B * w.K))
    return W.Workload(w.name, w.target[:1, :m + 1], w.draft[:1, :m], w.tokens[:1, :m], w.uniforms[:1, :m + 1],
                      w.temperature, b, w.meta)


def _subset(w, n):
    """The first n requests of a workload (the budget scaled with the batch)."""
    import workloads as W
    b = None if w.budget is None else max(1, w.budget * n // w.B)
    return W.Workload(w.name, w.target[:n], w.draft[:n], w.tokens[:n], w.uniforms[:n], w.temperature, b, w.meta)


# ---------------------------------------------------------------- main

def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="budget_sweep_B64")
    ap.add_argument("--extra", nargs="*", default=["greedy_mtp", "stochastic_mtp", "dfly_block", "budget_sweep_B4",
                                                   "budget_sweep_B16", "budget_sweep_B64", "draft_budget_B64",
                                                   "draft_budget_adaptive_B64"])
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
