"""CUDA draft-side confidence budget and utility / cost choice of N vs the float64 oracle (C ABI).

The draft statistics kernel reads only the draft rows; the budget kernel merges its partials into
q_k(x_k), builds the prefix confidences and selects the keys (fixed N, or the N that maximises
(B + S(N)) / cost(B + N)).  Confidences agree with the oracle to a relative 1e-4; depths and N
are bit-exact where the oracle's decision margin is >= 1e-5 and otherwise a valid choice within
that margin.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import spec_oracle as O
from tests.parity_utils import MARGIN, check_budget_choice, to_np
import workloads as W

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sv():
    import draft_verification_spec_gb300 as m
    m.lib()
    return m


def _np(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def _check_n(n_gpu, ref):
    """N: the oracle's when its relative utility margin is >= 1e-5, else within that of the best."""
    if ref.margin >= MARGIN:
        assert n_gpu == ref.N
    else:
        assert ref.utility[n_gpu] >= ref.utility[ref.N] * (1.0 - MARGIN)


def _run_draft(sv, draft, tokens, T, budget=None, cost=None):
    d = torch.device("cuda")
    n_out, depth, conf = sv.draft_budget(draft.to(d), tokens.to(d), T, budget=budget, cost=cost)
    torch.cuda.synchronize()
    assert sv.default_workspace().status() == 0
    return int(n_out.item()), depth.cpu().numpy(), to_np(conf)


def _check_draft(sv, w, budget=None, cost=None):
    qx = O.draft_confidence(_np(w.draft), w.tokens.numpy(), w.temperature)
    n, depth, conf = _run_draft(sv, w.draft, w.tokens, w.temperature, budget=budget, cost=cost)
    c_ref, _ = O.cumulative_alpha(qx)
    np.testing.assert_allclose(conf, c_ref, rtol=1e-4, atol=1e-9)
    if cost is None:
        br = O.alloc_budget(qx, budget)
        assert n == 0                       # N is reported only when it is chosen
    else:
        ref = O.adaptive_budget(qx, *cost)
        _check_n(n, ref)
        br = O.alloc_budget(qx, n)
    if not check_budget_choice(depth, br.conf, min(n if cost is not None else budget, qx.size), br.margin):
        np.testing.assert_array_equal(depth, br.depth)
    return n, depth


def test_draft_budget_golden(sv):
    """The hand-worked confidences and depths of tests/golden/draft_confidence.json, on the GPU."""
    with open(os.path.join(GOLD, "draft_confidence.json")) as f:
        g = json.load(f)
    with np.errstate(divide="ignore"):
        zd = torch.tensor(np.log(np.array(g["probs_T1"])), dtype=torch.float32)
    x = torch.tensor(g["tokens"], dtype=torch.int32)
    for T, key_q, key_d in ((g["T"], "conf", "depth_by_N"), (0.0, None, "T0_depth_by_N")):
        for N, want in g[key_d].items():
            n, depth, conf = _run_draft(sv, zd, x, T, budget=int(N))
            assert depth.tolist() == want
            if key_q:
                np.testing.assert_allclose(conf, g[key_q], rtol=1e-6, atol=1e-7)
    xo = torch.tensor(g["out_of_range_tokens"], dtype=torch.int32)
    _, _, conf = _run_draft(sv, zd, xo, g["T"], budget=2)
    np.testing.assert_allclose(conf[:, 0], [0.0, g["out_of_range_qx"][1][0]], rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("V,dtype", [(3001, torch.bfloat16), (4096, torch.float32), (50008, torch.bfloat16),
                                     (131072, torch.float32)])
@pytest.mark.parametrize("T", [0.0, 0.9])
def test_draft_budget_shapes(sv, V, dtype, T):
    """Aligned and unaligned rows, one and several parts per row, both element types, T = 0 and T > 0."""
    w = W.random_case(seed=V + int(10 * T), B=5, K=6, V=V, T=T, dtype=dtype)
    for N in (0, 7, 30):
        _check_draft(sv, w, budget=N)
    _check_draft(sv, w, cost=W.verify_cost_table(5, 6))


def test_draft_budget_greedy_ties(sv):
    """T = 0 with planted three-way ties across the parts of a row: the lowest index is the argmax."""
    B, K, V = 3, 4, 70000
    g = torch.Generator().manual_seed(12)
    zd = torch.randn(B, K, V, generator=g).to(torch.bfloat16)
    x = torch.empty(B, K, dtype=torch.int32)
    for b in range(B):
        for k in range(K):
            idx = torch.randperm(V, generator=g)[:3].sort().values
            zd[b, k, idx] = 40.0
            x[b, k] = int(idx[(b + k) % 3])          # the tie's first, second or third index
    w = W.Workload("ties", torch.zeros(B, K + 1, V), zd, x, torch.zeros(B, K + 1), 0.0)
    qx = O.draft_confidence(_np(zd), x.numpy(), 0.0)
    assert set(np.unique(qx)) <= {0.0, 1.0} and qx.sum() > 0
    for N in (1, 5, 12):
        _check_draft(sv, w, budget=N)


@pytest.mark.parametrize("B", [16, 64])
def test_draft_budget_full_size(sv, B):
    """The budget sweep's draft rows (V = 128000 bf16, K = 16): fixed N = 8B and the adaptive N."""
    w = W.budget_sweep(B)
    _check_draft(sv, w, budget=w.budget)
    _check_draft(sv, w, cost=W.verify_cost_table(B, w.K))


def test_alloc_budget_adaptive_matches_oracle(sv):
    """The utility / cost choice of N on the target-side alpha of a batch, and on the golden tables."""
    w = W.budget_sweep(16, V=20000)
    alpha, _, _ = O.overlap_stats(_np(w.target), _np(w.draft), w.temperature)
    alpha = alpha.astype(np.float32).astype(np.float64)          # what the GPU is given
    d = torch.device("cuda")
    a32 = torch.tensor(alpha, dtype=torch.float32, device=d)
    for cost in (W.verify_cost_table(16, w.K), ([16.0, 272.0], [1.0, 1.0]), ([16.0, 272.0], [16.0, 272.0])):
        n, depth, conf = sv.alloc_budget_adaptive(a32, cost)
        torch.cuda.synchronize()
        ref = O.adaptive_budget(alpha, *cost)
        _check_n(int(n.item()), ref)
        br = O.alloc_budget(alpha, int(n.item()))
        if not check_budget_choice(depth.cpu().numpy(), br.conf, int(n.item()), br.margin):
            np.testing.assert_array_equal(depth.cpu().numpy(), br.depth)
    with open(os.path.join(GOLD, "adaptive_budget.json")) as f:
        g = json.load(f)
    ga = torch.tensor(g["alpha"], dtype=torch.float32, device=d)
    for t in g["tables"].values():
        n, depth, _ = sv.alloc_budget_adaptive(ga, (t["cost_n"], t["cost_t"]))
        torch.cuda.synchronize()
        assert int(n.item()) == t["N"] and depth.cpu().tolist() == t["depth"]


def test_draft_budget_degenerate_and_invalid(sv):
    d = torch.device("cuda")
    # K = 0: nothing to select; N = 0 whatever the table
    zd = torch.zeros(3, 0, 10, device=d)
    x = torch.zeros(3, 0, dtype=torch.int32, device=d)
    n, depth, _ = sv.draft_budget(zd, x, 0.7, cost=([3.0, 6.0], [1.0, 2.0]))
    torch.cuda.synchronize()
    assert int(n.item()) == 0 and depth.cpu().tolist() == [0, 0, 0]
    # a cost table longer than 64 points is refused; so is a call with neither N nor a table
    zd = torch.zeros(2, 2, 10, device=d)
    x = torch.zeros(2, 2, dtype=torch.int32, device=d)
    with pytest.raises(sv.SpecError):
        sv.draft_budget(zd, x, 0.7, cost=(list(range(65)), [1.0] * 65))
    with pytest.raises(ValueError):
        sv.draft_budget(zd, x, 0.7)


@pytest.mark.parametrize("B,K", [(100, 21), (256, 16), (512, 16), (273, 30)])
def test_budget_large_batches(sv, B, K):
    """Up to the documented B K <= 8192 keys (the sort's 8 and 16 values per thread, padding to a
    power of two, shared memory past 48 KB): the utility / cost N and a given N against the
    oracle, on dyadic alphas whose products are exact in float32 and tie often."""
    rng = np.random.default_rng(B * 100 + K)
    alpha = rng.choice([0.5, 0.75, 1.0, 0.875, 0.25], size=(B, K)).astype(np.float32)
    d = torch.device("cuda")
    a32 = torch.tensor(alpha, device=d)
    a64 = alpha.astype(np.float64)
    for cost in (W.verify_cost_table(B, K), ([float(B), float(B * (K + 1))], [1.0, 3.0])):
        n, depth, conf = sv.alloc_budget_adaptive(a32, cost)
        torch.cuda.synchronize()
        ref = O.adaptive_budget(a64, *cost)
        _check_n(int(n.item()), ref)
        br = O.alloc_budget(a64, int(n.item()))
        if not check_budget_choice(depth.cpu().numpy(), br.conf, int(n.item()), br.margin):
            np.testing.assert_array_equal(depth.cpu().numpy(), br.depth)
    for N in (1, B * K // 3, B * K - 1):
        depth, _ = sv.alloc_budget(a32, N)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(depth.cpu().numpy(), O.alloc_budget(a64, N).depth)
