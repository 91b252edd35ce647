"""CPU checks of the benchmark's host logic: the reference arm's JSON line, the algorithmic byte
count behind the roofline, and the guard that drops a profiled DRAM traffic figure once the
kernel's sources no longer match the capture."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--config", "tiny_chain", "--steps", "3", "--warmup", "3"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_algorithmic_bytes_count_each_logit_once():
    w = W.greedy_mtp(B=2, V=1000)
    e = w.target.element_size()
    target_only = 2 * 4 * 1000 * e
    small = 2 * 3 * 4 + 2 * 4 * 4 + 2 * 4          # ids, emitted tokens, accepted counts
    assert bench.algorithmic_bytes(w, False) == target_only + small
    w2 = W.random_case(seed=1, B=2, K=3, V=1000, T=0.9, dtype=torch.bfloat16)
    with_draft = target_only + 2 * 3 * 1000 * e
    assert bench.algorithmic_bytes(w2, True) == with_draft + small + 2 * 4 * 4   # + uniforms


def test_profiled_traffic_needs_matching_sources(tmp_path, monkeypatch):
    path = tmp_path / "traffic.txt"
    good = bench.kernel_source_hash("greedy")
    path.write_text(f"# comment\nkernel_source_hash = {good}\ngreedy_mtp.dram_bytes_per_launch = 123456\n")
    monkeypatch.setitem(bench.KERNELS["greedy"], "traffic", str(path))
    assert bench.profiled_traffic("greedy", "greedy_mtp") == 123456
    assert bench.profiled_traffic("greedy", "stochastic_mtp") is None       # no figure for that workload
    path.write_text("kernel_source_hash = 0000000000000000\ngreedy_mtp.dram_bytes_per_launch = 123456\n")
    assert bench.profiled_traffic("greedy", "greedy_mtp") is None           # the kernel changed since



def test_oracle_agreement_counts_a_planted_disagreement():
    """The bench's decision check: GPU decisions equal the oracle's except where the oracle's margin
    is below 1e-5; a planted disagreement on an unambiguous request is reported."""
    import draft_verification_spec_gb300 as sv_mod  # noqa: F401  (only VerifyOutput is used; no GPU)
    from draft_verification_spec_gb300 import VerifyOutput
    w = W.random_case(seed=3, B=5, K=3, V=300, T=0.9, dtype=torch.float32)
    parts = bench.oracle_pass(w)
    import numpy as np
    tok = torch.tensor(np.concatenate([p.tokens for p in parts]), dtype=torch.int32)
    acc = torch.tensor(np.concatenate([p.accepted for p in parts]), dtype=torch.int32)
    margin = np.concatenate([p.margin for p in parts])
    out = VerifyOutput(tok.clone(), acc.clone())
    a = bench.agreement(w, parts, out)
    assert a["requests"] == 5 and a["unambiguous_mismatches"] == 0 and a["ambiguous_mismatches"] == 0
    assert a["ambiguous"] == int((margin < 1e-5).sum())
    b = int(np.argmax(margin))                       # the least ambiguous request
    out.tokens[b, int(out.accepted[b])] += 1
    assert bench.agreement(w, parts, out)["unambiguous_mismatches"] == 1


def test_reference_arm_budgeted_config_scales_the_budget():
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--config", "budget_sweep_B4", "--steps", "3", "--warmup", "3"])
    d = json.loads([ln for ln in buf.getvalue().splitlines() if ln.startswith("{")][0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert "N=32" in d["config"]["workload"] and "the batch's share" in d["cpu_baseline"]["sample"]
    assert "0.5 verified token(s) per drafted position" in d["cpu_baseline"]["sample"]   # N / (B K) = 32 / 64


def test_reference_arm_prefix_sample():
    """A request cut to its first m drafted positions keeps the rows those positions need, and its
    budget is the batch's scaled to them."""
    w = W.budget_sweep(4, V=1000)
    p = bench._prefix(w, 3)
    assert (p.B, p.K, p.V) == (1, 3, 1000)
    assert tuple(p.target.shape) == (1, 4, 1000) and tuple(p.uniforms.shape) == (1, 4)
    assert p.budget == max(1, w.budget * 3 // (w.B * w.K))
    assert bool((p.target[0] == w.target[0, :4]).all()) and bool((p.tokens[0] == w.tokens[0, :3]).all())


def test_verified_tokens_is_the_budget_when_there_is_one():
    w = W.budget_sweep(4, V=1000)
    assert bench.verified_tokens(w) == 32
    assert bench.verified_tokens(W.greedy_mtp(B=2, V=1000)) == 6


def test_draft_budget_configs_read_only_the_draft_rows():
    """The draft-side budget configurations run on the budget sweep's draft rows alone: the entry
    point, the algorithmic bytes (draft rows once, tokens, depth, confidences, N) and the cost
    table (n from B to B(K+1), increasing cost)."""
    w = W.budget_sweep(4, V=1000)
    assert bench.call_kind(w, "draft_budget_B4") == ("draft", True)
    assert bench.call_kind(w, "draft_budget_adaptive_B4") == ("draft_adaptive", True)
    B, K, V = w.B, w.K, w.V
    want = B * K * V * w.draft.element_size() + B * K * 4 + B * 4 + B * K * 4 + 4
    assert bench.algorithmic_bytes(w, True, "draft") == want
    assert bench.algorithmic_bytes(w, True, "draft_adaptive") == want
    n, t = W.verify_cost_table(B, K)
    assert n[0] == B and n[-1] == B * (K + 1) and all(a < b for a, b in zip(n, n[1:]))
    assert all(a <= b for a, b in zip(t, t[1:]))
