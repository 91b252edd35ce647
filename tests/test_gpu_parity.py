"""CUDA path vs the float64 oracle, through the C ABI (ctypes binding), on seeded inputs.

Full-size configurations (V = 128000, bf16) run in the launch configuration
the benchmark times; small and ragged shapes cover the tails (unaligned rows,
partial chunks, empty CTA slices, a single vocabulary entry) and the
degenerate cases of the method (K = 0, alpha = 1, disjoint supports, ties).
"""
import math

import numpy as np
import pytest
import torch

from oracle import spec_oracle as O
from tests.parity_utils import (check_budget_choice, check_guards, compare, guarded_output, oracle_alpha,
                                oracle_verify, to_np)
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import draft_verification_spec_gb300 as m
    m.lib()
    return m


def _dev(w):
    d = torch.device("cuda")
    return (w.target.to(d), w.draft.to(d), w.tokens.to(d), w.uniforms.to(d))


def _run_chain(sv, w, want_alpha=True, depth=None, tuning=None):
    t, d, x, u = _dev(w)
    draft = d if (w.K > 0 and (w.temperature > 0 or want_alpha)) else None
    # every output carries a canary tail, checked after the call
    out, guards = guarded_output(w.B, w.K, stats=want_alpha)
    out.cum_alpha = out.expected_len = None
    out = sv.verify_chain(t, draft, x, u, w.temperature, want_alpha=want_alpha, out=out, tuning=tuning,
                          depth=None if depth is None else torch.as_tensor(depth, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    check_guards(guards)
    return out


def _run_block(sv, w, budget=None, want_stats=True, tuning=None):
    t, d, x, u = _dev(w)
    out, guards = guarded_output(w.B, w.K, stats=want_stats, depth=budget is not None)
    out = sv.verify_block(t, d, x, u, w.temperature, budget=budget, want_stats=want_stats, out=out,
                          tuning=tuning)
    torch.cuda.synchronize()
    check_guards(guards)
    return out


# ---------------------------------------------------------------- the five configurations

def test_tiny_chain(sv):
    w = W.tiny_chain()
    out = _run_chain(sv, w)
    ref = oracle_verify(w)
    assert compare(out, ref, w) == 0
    assert sv.default_workspace().status() == 0


def test_greedy_mtp_full(sv):
    w = W.greedy_mtp()
    out = _run_chain(sv, w, want_alpha=False)            # the benchmark's call: target only
    ref = oracle_verify(w, need_alpha=False)
    compare(out, ref, w, check_alpha=False)
    out2 = _run_chain(sv, w, want_alpha=True)            # with the one-hot alpha (reads the draft)
    compare(out2, oracle_verify(w), w)


def test_stochastic_mtp_full(sv):
    w = W.stochastic_mtp()
    out = _run_chain(sv, w)
    ref = oracle_verify(w)
    amb = compare(out, ref, w)
    print(f"stochastic_mtp: {amb} of {w.B} requests ambiguous (margin < 1e-5), checked for consistency")
    mean_alpha = float(to_np(out.alpha).mean())
    assert 0.3 < mean_alpha < 0.9


def test_dfly_block_full(sv):
    w = W.dfly_block()
    out = _run_block(sv, w)
    ref = oracle_verify(w)
    amb = compare(out, ref, w)
    print(f"dfly_block: {amb} of {w.B} requests ambiguous (margin < 1e-5), checked for consistency")
    a = to_np(out.alpha).mean(axis=0)
    assert a[0] > a[-1]                                   # the noise ramp makes alpha decay


@pytest.mark.parametrize("B", [4, 8, 16, 32, 64])
def test_budget_sweep_full(sv, B):
    w = W.budget_sweep(B)
    out = _run_block(sv, w, budget=w.budget)
    a_ref = oracle_alpha(w)
    np.testing.assert_allclose(to_np(out.alpha), a_ref, atol=1e-5, rtol=0)
    br = O.alloc_budget(a_ref, w.budget)
    gdepth = out.depth.cpu().numpy()
    if not check_budget_choice(gdepth, br.conf, w.budget, br.margin):
        np.testing.assert_array_equal(gdepth, br.depth)
    # decisions at the depth the GPU chose
    ref = oracle_verify(w, depth=gdepth)
    compare(out, ref, w)


# ---------------------------------------------------------------- shapes, tails, dtypes

CASES = [
    # (B, K, V, T, dtype)
    (1, 0, 1, 0.0, torch.float32),
    (2, 1, 1, 1.0, torch.float32),
    (3, 2, 2, 0.7, torch.float32),
    (2, 3, 17, 1.0, torch.bfloat16),       # unaligned rows: element-wise path
    (3, 5, 1000, 0.9, torch.float32),
    (2, 4, 1004, 1.3, torch.float32),      # fp32 16-byte copies; the last item is mostly past the row end
    (3, 3, 1023, 0.9, torch.bfloat16),     # unaligned bf16
    (2, 2, 8191, 0.0, torch.bfloat16),
    (2, 7, 8200, 0.5, torch.bfloat16),     # two CTAs per row, ragged second slice
    (1, 31, 3000, 1.0, torch.float32),     # K at its limit
    (2, 3, 40000, 0.9, torch.bfloat16),
    (2, 2, 131080, 0.9, torch.bfloat16),   # above 128K: a ragged item in every CTA slice
    (1, 2, 262144, 1.1, torch.bfloat16),   # largest V
    (1, 1, 262144, 0.0, torch.float32),
]


@pytest.mark.parametrize("B,K,V,T,dtype", CASES)
def test_shapes_chain_and_block(sv, B, K, V, T, dtype):
    w = W.random_case(seed=B * 1000 + K * 10 + V, B=B, K=K, V=V, T=T, dtype=dtype)
    ref = oracle_verify(w)
    out = _run_chain(sv, w, want_alpha=K > 0)
    compare(out, ref, w)
    if K > 0:
        outb = _run_block(sv, w)
        compare(outb, ref, w)


def test_alpha_one_accepts_everything(sv):
    w = W.random_case(seed=5, B=4, K=6, V=5000, T=0.8, dtype=torch.bfloat16)
    w.draft = w.target[:, :w.K].clone()
    out = _run_block(sv, w)
    assert np.all(out.accepted.cpu().numpy() == w.K)
    np.testing.assert_allclose(to_np(out.alpha), 1.0, atol=1e-5)
    compare(out, oracle_verify(w), w)


def test_disjoint_supports_reject_at_zero(sv):
    B, K, V = 3, 2, 2000
    t = torch.full((B, K + 1, V), float("-inf"))
    d = torch.full((B, K, V), float("-inf"))
    g = torch.Generator().manual_seed(3)
    t[:, :, : V // 2] = torch.randn(B, K + 1, V // 2, generator=g)
    d[:, :, V // 2:] = torch.randn(B, K, V - V // 2, generator=g)
    x = torch.randint(V // 2, V, (B, K), generator=g, dtype=torch.int32)
    u = torch.rand(B, K + 1, generator=g)
    w = W.Workload("disjoint", t, d, x, u, 1.0)
    out = _run_block(sv, w)
    assert np.all(out.accepted.cpu().numpy() == 0)
    np.testing.assert_allclose(to_np(out.alpha), 0.0, atol=1e-6)   # alpha = sum p - R carries fp32 rounding
    compare(out, oracle_verify(w), w)


def test_greedy_planted_ties_lowest_index(sv):
    B, K, V = 4, 3, 70000
    g = torch.Generator().manual_seed(9)
    t = torch.randn(B, K + 1, V, generator=g).to(torch.bfloat16)
    for b in range(B):
        for k in range(K + 1):
            idx = torch.randperm(V, generator=g)[:3].sort().values
            t[b, k, idx] = 50.0                           # three-way tie, spread over CTA slices
    d = t[:, :K].clone()
    x = torch.argmax(t[:, :K].float(), dim=-1).to(torch.int32)
    x[1, 1] = int(torch.nonzero(t[1, 1].float() == 50.0)[-1])   # a tied but not-lowest index
    w = W.Workload("ties", t, d, x, torch.rand(B, K + 1, generator=g), 0.0)
    out = _run_chain(sv, w, want_alpha=True)
    ref = oracle_verify(w)
    compare(out, ref, w)
    assert out.accepted.cpu()[1].item() == 1


# ---------------------------------------------------------------- greedy kernels

GREEDY_CASES = [
    # (B, K, V, dtype)
    (3, 2, 8, torch.bfloat16),        # one partial tile: most lanes read -inf
    (2, 3, 1000, torch.float32),      # fp32 partial tile
    (2, 4, 2048, torch.bfloat16),     # exactly one tile per row
    (3, 1, 20008, torch.bfloat16),    # ragged last tile
    (2, 5, 12300, torch.float32),     # fp32 ragged
    (5, 3, 128000, torch.bfloat16),   # warp runs that span rows and requests
    (1, 0, 65536, torch.bfloat16),    # K = 0
    (2, 3, 1023, torch.bfloat16),     # unaligned rows: element-wise loads
]


@pytest.mark.parametrize("B,K,V,dtype", GREEDY_CASES)
def test_greedy_fused_and_separate_cut_agree(sv, B, K, V, dtype):
    w = W.random_case(seed=7 * B + 13 * K + V, B=B, K=K, V=V, T=0.0, dtype=dtype)
    ref = oracle_verify(w)
    outs = []
    for variant in (0, 2):   # the cut fused into the argmax kernel, then in its own kernel
        t, d, x, u = _dev(w)
        out = sv.verify_chain(t, d if K > 0 else None, x, u, 0.0, want_alpha=K > 0,
                              tuning=sv.Tuning(greedy_variant=variant))
        torch.cuda.synchronize()
        compare(out, ref, w)
        outs.append(out)
    assert torch.equal(outs[1].tokens, outs[0].tokens) and torch.equal(outs[1].accepted, outs[0].accepted)
    if K > 0:
        assert torch.equal(outs[1].alpha, outs[0].alpha)
    assert sv.default_workspace().status() == 0


# ---------------------------------------------------------------- other entry points

def test_overlap_alpha_matches_oracle(sv):
    for w in (W.stochastic_mtp(B=8), W.random_case(seed=4, B=3, K=5, V=1023, T=0.6, dtype=torch.bfloat16),
              W.greedy_mtp(B=8)):
        t, d, _, _ = _dev(w)
        a, c, E = sv.overlap_alpha(t, d, w.temperature)
        torch.cuda.synchronize()
        ra, rc, rE = O.overlap_stats(w.target.double().numpy(), w.draft.double().numpy(), w.temperature)
        np.testing.assert_allclose(to_np(a), ra, atol=1e-5, rtol=0)
        np.testing.assert_allclose(to_np(c), rc, atol=1e-5, rtol=0)
        np.testing.assert_allclose(to_np(E), rE, atol=1e-4, rtol=0)


def test_alloc_budget_exact_dyadic(sv):
    rng = np.random.default_rng(0)
    for B, K in [(3, 3), (7, 5), (64, 16), (128, 16), (1, 1), (5, 0)]:
        a = rng.choice([0.0, 0.25, 0.5, 0.75, 1.0], size=(B, K)).astype(np.float32)
        for N in sorted({0, 1, B, (B * K) // 2, B * K - 1, B * K, B * K + 3}):
            if N < 0:
                continue
            depth, conf = sv.alloc_budget(torch.tensor(a, device="cuda"), N)
            torch.cuda.synchronize()
            ref = O.alloc_budget(a.astype(np.float64), N)
            np.testing.assert_array_equal(depth.cpu().numpy(), ref.depth)
            np.testing.assert_array_equal(conf.cpu().numpy().astype(np.float64), ref.conf)


def test_alloc_budget_golden_ties(sv):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "budget_ties.json")))
    a = torch.tensor(g["alpha"], dtype=torch.float32, device="cuda")
    for N, want in g["depth_by_N"].items():
        depth, _ = sv.alloc_budget(a, int(N))
        assert depth.cpu().tolist() == want


def test_chain_with_depth_from_budget(sv):
    w = W.stochastic_mtp(B=16)
    t, d, x, u = _dev(w)
    a, _, _ = sv.overlap_alpha(t, d, w.temperature)
    depth, _ = sv.alloc_budget(a, 20)
    out = sv.verify_chain(t, d, x, u, w.temperature, depth=depth, want_alpha=True)
    torch.cuda.synchronize()
    dd = depth.cpu().numpy()
    assert np.all(out.accepted.cpu().numpy() <= dd)
    compare(out, oracle_verify(w, depth=dd), w)


# ---------------------------------------------------------------- errors and status

def test_invalid_arguments_rejected_synchronously(sv):
    w = W.tiny_chain()
    t, d, x, u = _dev(w)
    with pytest.raises(sv.SpecError) as e:
        sv.verify_chain(t, d, x, u, -1.0)
    assert e.value.code == 1
    with pytest.raises(sv.SpecError) as e:
        sv.verify_chain(t, d, x, u, float("nan"))
    assert e.value.code == 1
    lib = sv.lib()
    import ctypes
    code = lib.spec_verify_chain(ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(d.data_ptr()), 0,
                                 ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(u.data_ptr()), 1, 3, 1024, 1.0,
                                 None, None, None, None, None, 0, None)
    assert code == 1
    assert lib.spec_verify_chain(ctypes.c_void_p(t.data_ptr()), None, 0, None, None, 1, 40, 1024, 0.0,
                                 None, None, None, None, None, 0, None) == 2


def test_token_out_of_range_sets_status(sv):
    w = W.tiny_chain()
    t, d, x, u = _dev(w)
    ws = sv.Workspace()
    x = x.clone()
    x[0, 0] = w.V + 5
    out = sv.verify_chain(t, d, x, u, 1.0, workspace=ws)
    assert ws.status() == 5
    assert out.accepted.item() == 0
    assert ws.status() == 0                                 # read-and-clear


def test_bounded_wait_timeout_reports_and_recovers(sv):
    w = W.stochastic_mtp(B=4)
    t, d, x, u = _dev(w)
    ws = sv.Workspace()
    # every bounded wait gives up at once: the timeout is reported, and the kernel still completes
    # its copies and exchanges before it returns
    sv.verify_chain(t, d, x, u, w.temperature, workspace=ws, tuning=sv.Tuning(wait_limit_us=-1))
    assert ws.status() == 4
    ws.reset()
    out = sv.verify_chain(t, d, x, u, w.temperature, workspace=ws, want_alpha=True)
    assert ws.status() == 0
    compare(out, oracle_verify(w), w)


def test_workspace_reuse_across_shapes(sv):
    ws = sv.Workspace()
    for w in (W.random_case(1, 3, 4, 5000, 0.9, torch.bfloat16), W.tiny_chain(),
              W.random_case(2, 5, 2, 9000, 0.0, torch.bfloat16), W.random_case(3, 2, 16, 3000, 1.2)):
        t, d, x, u = _dev(w)
        for _ in range(3):
            out = sv.verify_block(t, d, x, u, w.temperature, workspace=ws)
            torch.cuda.synchronize()
            compare(out, oracle_verify(w), w)
    assert ws.status() == 0


def test_repeated_calls_deterministic(sv):
    w = W.stochastic_mtp(B=32)
    t, d, x, u = _dev(w)
    o1 = sv.verify_chain(t, d, x, u, w.temperature, want_alpha=True)
    o2 = sv.verify_chain(t, d, x, u, w.temperature, want_alpha=True)
    torch.cuda.synchronize()
    assert torch.equal(o1.tokens, o2.tokens) and torch.equal(o1.alpha, o2.alpha)


# ---------------------------------------------------------------- paths not covered above

def test_greedy_block_with_budget(sv):
    # T = 0 with a budget: one-hot alpha from the argmax keys, the budget, then the cut
    w = W.random_case(seed=21, B=6, K=5, V=9000, T=0.0, dtype=torch.bfloat16)
    N = 13
    out = _run_block(sv, w, budget=N)
    a_ref = oracle_alpha(w)
    np.testing.assert_array_equal(to_np(out.alpha), a_ref)
    br = O.alloc_budget(a_ref, N)
    np.testing.assert_array_equal(out.depth.cpu().numpy(), br.depth)     # dyadic keys: exact
    compare(out, oracle_verify(w, depth=br.depth), w)
    assert sv.default_workspace().status() == 0


def test_greedy_chain_with_depth(sv):
    w = W.random_case(seed=22, B=5, K=4, V=7000, T=0.0, dtype=torch.bfloat16)
    depth = np.array([0, 1, 4, 2, 3], dtype=np.int32)
    out = _run_chain(sv, w, want_alpha=True, depth=depth)
    compare(out, oracle_verify(w, depth=depth), w)
    assert np.all(out.accepted.cpu().numpy() <= depth)


def test_overlap_alpha_fp32(sv):
    w = W.random_case(seed=23, B=3, K=4, V=5000, T=0.7, dtype=torch.float32)
    t, d, _, _ = _dev(w)
    a, c, E = sv.overlap_alpha(t, d, w.temperature)
    torch.cuda.synchronize()
    ra, rc, rE = O.overlap_stats(w.target.double().numpy(), w.draft.double().numpy(), w.temperature)
    np.testing.assert_allclose(to_np(a), ra, atol=1e-5, rtol=0)
    np.testing.assert_allclose(to_np(c), rc, atol=1e-5, rtol=0)
    np.testing.assert_allclose(to_np(E), rE, atol=1e-4, rtol=0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_k0_sampling_is_plain_decoding(sv, dtype):
    # K = 0 at T > 0: no draft, the emitted token is the draw from p_0
    w = W.random_case(seed=24, B=4, K=0, V=3000, T=0.8, dtype=dtype)
    out = _run_chain(sv, w, want_alpha=False)
    compare(out, oracle_verify(w), w)
    assert np.all(out.accepted.cpu().numpy() == 0)


def test_fp32_block_with_budget(sv):
    w = W.random_case(seed=25, B=5, K=6, V=6000, T=1.1, dtype=torch.float32)
    N = 11
    out = _run_block(sv, w, budget=N)
    a_ref = oracle_alpha(w)
    np.testing.assert_allclose(to_np(out.alpha), a_ref, atol=1e-5, rtol=0)
    gdepth = out.depth.cpu().numpy()
    br = O.alloc_budget(a_ref, N)
    if not check_budget_choice(gdepth, br.conf, N, br.margin):
        np.testing.assert_array_equal(gdepth, br.depth)
    compare(out, oracle_verify(w, depth=gdepth), w)


# ---------------------------------------------------------------- fp32 rows split over several CTAs

@pytest.mark.parametrize("V,cluster", [(65536, 0), (65536, 4), (131072, 0), (131072, 8)])
def test_fp32_multi_cta_chain_block_budget(sv, V, cluster):
    """fp32 logits at T > 0 with the row split over a cluster (the DSMEM exchange of fp32 partials)."""
    w = W.random_case(seed=31 + V // 1024 + cluster, B=3, K=3, V=V, T=0.9, dtype=torch.float32)
    tun = sv.Tuning(cluster=cluster)
    ref = oracle_verify(w)
    compare(_run_chain(sv, w, want_alpha=True, tuning=tun), ref, w)
    if cluster:
        assert tun.plan["cluster"] == cluster
    compare(_run_block(sv, w, tuning=sv.Tuning(cluster=cluster)), ref, w)
    N = 5
    out = _run_block(sv, w, budget=N, tuning=sv.Tuning(cluster=cluster))
    a_ref = oracle_alpha(w)
    np.testing.assert_allclose(to_np(out.alpha), a_ref, atol=1e-5, rtol=0)
    br = O.alloc_budget(a_ref, N)
    gdepth = out.depth.cpu().numpy()
    if not check_budget_choice(gdepth, br.conf, N, br.margin):
        np.testing.assert_array_equal(gdepth, br.depth)
    compare(out, oracle_verify(w, depth=gdepth), w)
    assert sv.default_workspace().status() == 0


def _slab_fits(V, esz, cluster):
    """Whether a CTA slice fits the sampling kernel's shared-memory slab (96 KB per row; the shapes
    tested here stay far below the limit of 80 (CTA, item) segments per row)."""
    slice_ = math.ceil(math.ceil(V / cluster) / 8) * 8
    return slice_ * esz <= 96 * 1024


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,cluster", [(24, 16), (4104, 1), (4099, 2), (50008, 4), (128000, 4), (128000, 8),
                                       (128000, 16)])
def test_slab_sizes(sv, dtype, V, cluster):
    """Every slab size the planner can pick gives the oracle's results: chain, block with a budget,
    and alpha alone (empty CTA slices at V = 24 over 16 CTAs, unaligned rows at V = 4099, ragged
    last items elsewhere); a forced cluster size whose slice does not fit is refused."""
    esz = 2 if dtype == torch.bfloat16 else 4
    w = W.random_case(seed=V + cluster + esz, B=3, K=4, V=V, T=0.9, dtype=dtype)
    if not _slab_fits(V, esz, cluster):
        with pytest.raises(sv.SpecError):
            _run_chain(sv, w, tuning=sv.Tuning(cluster=cluster))
        return
    ref = oracle_verify(w)
    tun = sv.Tuning(cluster=cluster)
    compare(_run_chain(sv, w, want_alpha=True, tuning=tun), ref, w)
    assert tun.plan["cluster"] == cluster
    slice_bytes = tun.plan["slice"] * esz
    assert 2 * slice_bytes <= tun.plan["smem_bytes"] <= 192 * 1024                # both rows of the slice fit
    assert tun.plan["smem_bytes"] % (2 * tun.plan["items"]) == 0
    N = 7
    out = _run_block(sv, w, budget=N, tuning=sv.Tuning(cluster=cluster))
    a_ref = oracle_alpha(w)
    np.testing.assert_allclose(to_np(out.alpha), a_ref, atol=1e-5, rtol=0)
    br = O.alloc_budget(a_ref, N)
    gdepth = out.depth.cpu().numpy()
    if not check_budget_choice(gdepth, br.conf, N, br.margin):
        np.testing.assert_array_equal(gdepth, br.depth)
    compare(out, oracle_verify(w, depth=gdepth), w)
    t, d, _, _ = _dev(w)
    a, _, _ = sv.overlap_alpha(t, d, w.temperature, tuning=sv.Tuning(cluster=cluster))
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_np(a), a_ref, atol=1e-5, rtol=0)
    assert sv.default_workspace().status() == 0


@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
def test_every_cluster_size_bf16(sv, cluster):
    """The same bf16 batch at every cluster size gives the oracle's decisions."""
    w = W.stochastic_mtp(B=6, V=128000)
    ref = oracle_verify(w)
    tun = sv.Tuning(cluster=cluster)
    if not _slab_fits(128000, 2, cluster):
        with pytest.raises(sv.SpecError):
            _run_chain(sv, w, want_alpha=True, tuning=tun)
        return
    compare(_run_chain(sv, w, want_alpha=True, tuning=tun), ref, w)
    assert tun.plan["cluster"] == cluster
