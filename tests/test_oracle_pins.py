"""Pins for the float64 oracle, checked against what the pages and the mathematics fix.

None of these re-types an oracle formula: they use hand-computed golden cases
(tests/golden/), identities (alpha = 1 - TV), library routines for special
cases (scipy softmax), brute-force histograms over 10^6 seeded trials, the
closed-form expected length, and exhaustive search for the budget.
"""
import json
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

from oracle import spec_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _logits(p):
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p)


# ---------------------------------------------------------------- golden cases

def test_hand_example_alpha_and_decisions():
    g = _load("hand_example.json")
    zt = _logits(g["p"])[None]          # [1, K+1, V]
    zd = _logits(g["q"])[None]          # [1, K, V]
    for case in g["cases"]:
        r = O.verify(zt, zd, np.array([case["tokens"]]), np.array([case["uniforms"]]), g["T"])
        assert r.tokens[0].tolist() == case["out"]
        assert int(r.accepted[0]) == case["accepted"]
        np.testing.assert_allclose(r.alpha[0], g["alpha"], atol=1e-15)
        np.testing.assert_allclose(r.cum_alpha[0], g["cum_alpha"], atol=1e-15)
        assert abs(r.expected_len[0] - g["expected_len"]) < 1e-15


def test_hand_example_decision_margins():
    """The two margins the match rule uses, worked by hand for the three cases (derivation in the JSON)."""
    g = _load("hand_example.json")
    zt = _logits(g["p"])[None]
    zd = _logits(g["q"])[None]
    for case in g["cases"]:
        r = O.verify(zt, zd, np.array([case["tokens"]]), np.array([case["uniforms"]]), g["T"])
        assert abs(r.margin_accept[0] - case["margin_accept"]) < 1e-12
        assert abs(r.margin_cdf[0] - case["margin_cdf"]) < 1e-12
        assert abs(r.margin[0] - min(case["margin_accept"], case["margin_cdf"])) < 1e-12


def test_budget_margin_golden():
    g = _load("budget_ties.json")
    a = np.array(g["alpha"])
    for N, want in g["margin_by_N"].items():
        assert O.alloc_budget(a, int(N)).margin == want, N
    assert O.alloc_budget(a, 0).margin == np.inf and O.alloc_budget(a, 9).margin == np.inf


def test_greedy_onehot_alpha_golden():
    """T = 0: alpha is [argmax target == argmax draft], ties in either row going to the lowest index."""
    g = _load("greedy_onehot_alpha.json")
    zt = np.array(g["target"], dtype=np.float64)[None]
    zd = np.array(g["draft"], dtype=np.float64)[None]
    r = O.verify(zt, zd, np.zeros((1, 2), dtype=int), np.zeros((1, 3)), 0.0)
    assert r.alpha[0].tolist() == g["alpha"]
    assert r.cum_alpha[0].tolist() == g["cum_alpha"] and r.expected_len[0] == g["expected_len"]
    a, c, E = O.overlap_stats(zt, zd, 0.0)
    assert a[0].tolist() == g["alpha"] and c[0].tolist() == g["cum_alpha"] and E[0] == g["expected_len"]


def test_alpha_handbuilt_equals_one_minus_tv():
    for c in _load("alpha_handbuilt.json")["cases"]:
        p, q = np.array(c["p"]), np.array(c["q"])
        a = O.overlap_alpha(p, q)
        assert abs(a - c["alpha"]) < 1e-15
        assert abs(a - (1.0 - c["tv"])) < 1e-15
        assert abs(O.overlap_alpha(q, p) - a) < 1e-15     # symmetric


def test_alpha_through_softmax_of_log_probs():
    c = _load("alpha_handbuilt.json")["cases"][0]
    p = O.softmax(_logits(c["p"]), 1.0)
    q = O.softmax(_logits(c["q"]), 1.0)
    assert abs(O.overlap_alpha(p, q) - c["alpha"]) < 1e-15


def test_mal_convention_from_pages():
    g = _load("mal_convention.json")
    for pair in g["pairs"]:
        assert round(1 + g["depth"] * pair["acceptance_rate"], 2) == pair["mal"]


def test_budget_hand_ties():
    g = _load("budget_ties.json")
    a = np.array(g["alpha"])
    for N, want in g["depth_by_N"].items():
        assert O.alloc_budget(a, int(N)).depth.tolist() == want, N


# ---------------------------------------------------------------- identities

def test_alpha_is_one_minus_tv_random():
    rng = np.random.default_rng(7)
    for V in (1, 2, 3, 17, 1000):
        z1, z2 = rng.normal(0, 2, (50, V)), rng.normal(0, 2, (50, V))
        p, q = O.softmax(z1, 0.9), O.softmax(z2, 0.9)
        tv = 0.5 * np.abs(p - q).sum(-1)
        np.testing.assert_allclose(O.overlap_alpha(p, q), 1 - tv, atol=1e-13)
        np.testing.assert_allclose(O.overlap_alpha(p, p), 1.0, atol=1e-13)


def test_alpha_disjoint_support_is_zero():
    z1 = np.array([0.0, 1.0, -np.inf, -np.inf])
    z2 = np.array([-np.inf, -np.inf, 3.0, 0.0])
    assert O.overlap_alpha(O.softmax(z1, 1.0), O.softmax(z2, 1.0)) == 0.0


def test_softmax_matches_scipy_and_invariances():
    rng = np.random.default_rng(3)
    z = rng.normal(0, 3, (7, 129))
    for T in (0.25, 0.9, 1.0, 2.5):
        p = O.softmax(z, T)
        np.testing.assert_allclose(p, scipy.special.softmax(z / T, axis=-1), rtol=1e-12, atol=1e-300)
        np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-13)
        np.testing.assert_allclose(O.softmax(z + 123.0, T), p, rtol=1e-11)
        np.testing.assert_allclose(O.softmax(z / T, 1.0), p, rtol=1e-12)
    zz = z.copy()
    zz[:, :5] = -np.inf
    assert np.all(O.softmax(zz, 0.9)[:, :5] == 0.0)


def test_cumulative_alpha_closed_form_by_hand():
    c, E = O.cumulative_alpha(np.array([[0.5, 0.5, 1.0, 0.0]]))
    assert c[0].tolist() == [0.5, 0.25, 0.25, 0.0]
    assert E[0] == 1.0


def test_inverse_cdf_against_linear_scan():
    rng = np.random.default_rng(11)
    for V in (1, 2, 5, 16):
        mass = rng.random(V) * (rng.random(V) > 0.3)
        if mass.sum() == 0:
            mass[0] = 1.0
        for u in np.linspace(0, 1, 257, endpoint=False):
            v, _ = O.inverse_cdf(mass, u)
            # linear scan written independently: walk until the running sum passes u*total
            total = 0.0
            for m in mass:
                total += m
            run, want = 0.0, None
            for i, m in enumerate(mass):
                run += m
                if run > u * total:
                    want = i
                    break
            assert int(v) == want
            assert mass[int(v)] > 0          # zero-mass bins are never drawn


# ---------------------------------------------------------------- brute force

def _chain(seed, K, V, spread=1.5, noise=0.8):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, spread, (K + 1, V))
    zd = zt[:K] + rng.normal(0, noise, (K, V))
    return zt, zd


def _run_trials(zt, zd, T, n_trials, seed, depth=None, chunk=100_000):
    """n_trials identical requests with fresh draft tokens x ~ q and fresh uniforms."""
    K, V = zd.shape
    q = scipy.special.softmax(zd / T, axis=-1)
    qc = np.cumsum(q, axis=-1)
    rng = np.random.default_rng(seed)
    toks, accs = [], []
    for s in range(0, n_trials, chunk):
        n = min(chunk, n_trials - s)
        x = np.stack([np.minimum(np.searchsorted(qc[k], rng.random(n) * qc[k, -1], side="right"), V - 1)
                      for k in range(K)], axis=1)
        u = rng.random((n, K + 1))
        r = O.verify(np.broadcast_to(zt, (n, K + 1, V)), np.broadcast_to(zd, (n, K, V)), x, u, T,
                     depth=None if depth is None else np.full(n, depth))
        toks.append(r.tokens)
        accs.append(r.accepted)
    return np.concatenate(toks), np.concatenate(accs)


def _chi2_ok(samples, p, min_pvalue=1e-3):
    V = p.shape[0]
    obs = np.bincount(samples, minlength=V).astype(np.float64)
    zero = p == 0
    assert obs[zero].sum() == 0
    exp = p[~zero] * obs.sum()
    stat = scipy.stats.chisquare(obs[~zero], exp * obs[~zero].sum() / exp.sum())
    return stat.pvalue > min_pvalue


N_TRIALS = 1_000_000


@pytest.fixture(scope="module")
def chain_trials():
    zt, zd = _chain(5, K=3, V=12)
    T = 0.9
    toks, acc = _run_trials(zt, zd, T, N_TRIALS, seed=123)
    return zt, zd, T, toks, acc


def test_target_distribution_unchanged_first_token(chain_trials):
    zt, zd, T, toks, acc = chain_trials
    p = scipy.special.softmax(zt / T, axis=-1)
    assert _chi2_ok(toks[:, 0], p[0])


def test_target_distribution_unchanged_every_position(chain_trials):
    zt, zd, T, toks, acc = chain_trials
    p = scipy.special.softmax(zt / T, axis=-1)
    K = zd.shape[0]
    for m in range(1, K + 1):
        reached = acc >= m
        assert reached.sum() > 10_000
        assert _chi2_ok(toks[reached, m], p[m]), m


def test_expected_length_closed_form(chain_trials):
    zt, zd, T, toks, acc = chain_trials
    p = scipy.special.softmax(zt / T, axis=-1)
    q = scipy.special.softmax(zd / T, axis=-1)
    a = np.minimum(p[:3], q).sum(-1)
    closed = sum(np.prod(a[: m + 1]) for m in range(3))
    sigma = acc.std() / np.sqrt(acc.size)
    assert abs(acc.mean() - closed) < 4 * sigma
    # oracle's own cumulative form agrees with the closed form
    _, E = O.cumulative_alpha(O.overlap_alpha(O.softmax(zt[:3], T), O.softmax(zd, T)))
    assert abs(E - closed) < 1e-12


def test_depth_limited_bonus_distribution():
    zt, zd = _chain(9, K=4, V=10)
    T = 1.3
    toks, acc = _run_trials(zt, zd, T, 300_000, seed=5, depth=2)
    assert acc.max() <= 2
    p = scipy.special.softmax(zt / T, axis=-1)
    full = acc == 2
    assert _chi2_ok(toks[full, 2], p[2])
    assert np.all(toks[:, 3:] == -1)


def test_alpha_one_always_accepts():
    zt, _ = _chain(1, K=3, V=8)
    toks, acc = _run_trials(zt, zt[:3].copy(), 0.9, 20_000, seed=2)
    assert np.all(acc == 3)


def test_alpha_zero_always_rejects_at_zero():
    V = 6
    zt = np.full((3, V), -np.inf)
    zt[:, :3] = [0.0, 0.5, 1.0]
    zd = np.full((2, V), -np.inf)
    zd[:, 3:] = [1.0, 0.0, -1.0]
    toks, acc = _run_trials(zt, zd, 1.0, 50_000, seed=4)
    assert np.all(acc == 0)
    p0 = scipy.special.softmax(zt[0])
    assert _chi2_ok(toks[:, 0], p0)


def test_no_drafts_is_plain_decoding():
    """K = 0: one token per request, the target argmax at T = 0 and a draw from p_0 at T > 0."""
    zt = np.random.default_rng(12).normal(0, 1.5, (1, 9))
    r = O.verify(zt[None], None, np.zeros((1, 0), dtype=int), np.zeros((1, 1)), 0.0)
    assert r.accepted[0] == 0 and r.tokens[0, 0] == int(np.argmax(zt[0]))
    n = 200_000
    u = np.random.default_rng(13).random((n, 1))
    r = O.verify(np.broadcast_to(zt, (n, 1, 9)), np.zeros((n, 0, 9)), np.zeros((n, 0), dtype=int), u, 0.8)
    assert np.all(r.accepted == 0)
    assert _chi2_ok(r.tokens[:, 0], scipy.special.softmax(zt[0] / 0.8))


# ---------------------------------------------------------------- greedy

def test_greedy_acceptance_is_argmax_agreement():
    rng = np.random.default_rng(8)
    B, K, V = 200, 4, 33
    zt = rng.integers(-3, 4, (B, K + 1, V)).astype(np.float64)   # many ties
    x = rng.integers(0, V, (B, K))
    for b in range(0, B, 2):                                     # half the rows: draft = true argmax prefix
        for k in range(K):
            row = zt[b, k]
            x[b, k] = int(np.flatnonzero(row == row.max())[0])
    r = O.verify(zt, None, x, rng.random((B, K + 1)), 0.0)
    for b in range(B):
        n = 0
        while n < K:
            row = zt[b, n]
            first_max = int(np.flatnonzero(row == row.max())[0])
            if x[b, n] != first_max:
                break
            n += 1
        assert r.accepted[b] == n
        row = zt[b, n]
        assert r.tokens[b, n] == int(np.flatnonzero(row == row.max())[0])
        assert np.all(r.tokens[b, :n] == x[b, :n]) and np.all(r.tokens[b, n + 1:] == -1)


def test_greedy_planted_ties_lowest_index():
    zt = np.zeros((1, 2, 5))
    zt[0, 0, [1, 3]] = 2.0
    zt[0, 1, [0, 4]] = 1.0
    r = O.verify(zt, None, np.array([[3]]), np.zeros((1, 2)), 0.0)
    assert r.accepted[0] == 0 and r.tokens[0].tolist() == [1, -1]
    r = O.verify(zt, None, np.array([[1]]), np.zeros((1, 2)), 0.0)
    assert r.accepted[0] == 1 and r.tokens[0].tolist() == [1, 0]


# ---------------------------------------------------------------- budget

def _prefix_allocations(B, K, N):
    def rec(b, left):
        if b == B:
            if left == 0:
                yield []
            return
        for d in range(0, min(K, left) + 1):
            for rest in rec(b + 1, left - d):
                yield [d] + rest
    yield from rec(0, N)


def test_budget_maximises_expected_accepted_exhaustive():
    rng = np.random.default_rng(21)
    for trial in range(40):
        B, K = rng.integers(1, 5), rng.integers(1, 5)
        a = rng.random((B, K)) * (rng.random((B, K)) > 0.15)
        c = np.cumprod(a, axis=1)
        for N in range(0, B * K + 2):
            r = O.alloc_budget(a, N)
            d = r.depth
            assert d.sum() == min(N, B * K)
            assert np.all((0 <= d) & (d <= K))
            got = sum(c[b, :d[b]].sum() for b in range(B))
            best = max(sum(c[b, :dd[b]].sum() for b in range(B))
                       for dd in _prefix_allocations(B, K, min(N, B * K)))
            assert got >= best - 1e-12
        assert np.all(O.alloc_budget(a, B * K + 7).depth == K)
        assert np.all(O.alloc_budget(a, 0).depth == 0)


def test_budget_clamps_alpha():
    a = np.array([[1.5, np.nan, -0.2], [0.9, 0.9, 0.9]])
    r = O.alloc_budget(a, 4)
    assert r.conf[0].tolist() == [1.0, 0.0, 0.0]
    assert r.depth.tolist() == [1, 3]


# ---------------------------------------------------------------- planted mistakes

def _mutant(old, new):
    """Load a copy of the oracle with one plausible mistake planted in its source (CPU only)."""
    import importlib.util
    import types
    path = O.__file__
    text = open(path).read()
    assert text.count(old) == 1, old
    import sys
    name = "oracle_mutant_%d" % (abs(hash((old, new))) % 10**8)
    mod = types.ModuleType(name)
    mod.__file__ = path
    sys.modules[name] = mod
    try:
        exec(compile(text.replace(old, new), path, "exec"), mod.__dict__)
    finally:
        pass
    return mod


def _hist_pin(mod, n=200_000):
    zt, zd = _chain(5, K=3, V=12)
    T = 0.9
    p = scipy.special.softmax(zt / T, axis=-1)
    saved = O.verify
    try:
        globals()["O"].verify = mod.verify
        toks, acc = _run_trials(zt, zd, T, n, seed=3)
    finally:
        globals()["O"].verify = saved
    return _chi2_ok(toks[:, 0], p[0]) and all(_chi2_ok(toks[acc >= m, m], p[m]) for m in (1, 2, 3))


def _hand_pin(mod):
    g = _load("hand_example.json")
    ok = True
    for case in g["cases"]:
        r = mod.verify(_logits(g["p"])[None], _logits(g["q"])[None], np.array([case["tokens"]]),
                       np.array([case["uniforms"]]), 1.0)
        ok &= r.tokens[0].tolist() == case["out"]
        ok &= bool(np.allclose(r.alpha[0], g["alpha"])) and abs(r.expected_len[0] - g["expected_len"]) < 1e-12
    return ok


def _budget_pin(mod):
    g = _load("budget_ties.json")
    a = np.array(g["alpha"])
    return all(mod.alloc_budget(a, int(N)).depth.tolist() == w for N, w in g["depth_by_N"].items())


def _icdf_pin(mod):
    # boundary draws worked by hand: C = (0, .5, 1); u = 0 -> first C > 0 is index 1;
    # u = .5 -> first C > .5 is index 2 (zero-mass bin 0 is never drawn)
    mass = np.array([0.0, 0.5, 0.5])
    return int(mod.inverse_cdf(mass, 0.0)[0]) == 1 and int(mod.inverse_cdf(mass, 0.5)[0]) == 2


def _greedy_pin(mod):
    zt = np.zeros((1, 2, 5))
    zt[0, 0, [1, 3]] = 2.0
    zt[0, 1, [0, 4]] = 1.0
    r = mod.verify(zt, None, np.array([[1]]), np.zeros((1, 2)), 0.0)
    return r.tokens[0].tolist() == [1, 0]


def _margin_pin(mod):
    g = _load("hand_example.json")
    ok = True
    for case in g["cases"]:
        r = mod.verify(_logits(g["p"])[None], _logits(g["q"])[None], np.array([case["tokens"]]),
                       np.array([case["uniforms"]]), 1.0)
        ok &= abs(r.margin_accept[0] - case["margin_accept"]) < 1e-12
        ok &= abs(r.margin_cdf[0] - case["margin_cdf"]) < 1e-12
    return bool(ok)


def _budget_margin_pin(mod):
    g = _load("budget_ties.json")
    a = np.array(g["alpha"])
    return all(mod.alloc_budget(a, int(N)).margin == m for N, m in g["margin_by_N"].items())


def _onehot_pin(mod):
    g = _load("greedy_onehot_alpha.json")
    zt = np.array(g["target"], dtype=np.float64)[None]
    zd = np.array(g["draft"], dtype=np.float64)[None]
    r = mod.verify(zt, zd, np.zeros((1, 2), dtype=int), np.zeros((1, 3)), 0.0)
    a, _, _ = mod.overlap_stats(zt, zd, 0.0)
    return r.alpha[0].tolist() == g["alpha"] and a[0].tolist() == g["alpha"]


def _draft_logits(probs):
    with np.errstate(divide="ignore"):
        return np.log(np.array(probs, dtype=np.float64))     # ln 0 = -inf: probability 0


def _draftconf_pin(mod):
    """The hand-worked draft-side confidences and budgets (tests/golden/draft_confidence.json)."""
    g = _load("draft_confidence.json")
    zd, x = _draft_logits(g["probs_T1"]), np.array(g["tokens"])
    ok = bool(np.allclose(mod.draft_confidence(zd, x, g["T"]), g["qx"], rtol=0, atol=1e-12))
    ok &= mod.draft_confidence(zd, x, 0.0).tolist() == g["T0_qx"]
    ok &= bool(np.allclose(mod.draft_confidence(zd, np.array(g["out_of_range_tokens"]), g["T"]),
                           g["out_of_range_qx"], rtol=0, atol=1e-12))
    for N, want in g["depth_by_N"].items():
        r = mod.draft_budget(zd, x, g["T"], int(N))
        ok &= r.depth.tolist() == want and bool(np.allclose(r.conf, g["conf"], rtol=0, atol=1e-12))
    for N, want in g["T0_depth_by_N"].items():
        ok &= mod.draft_budget(zd, x, 0.0, int(N)).depth.tolist() == want
    return ok


def _adaptive_pin(mod):
    """The hand-worked utility/cost choices of N (tests/golden/adaptive_budget.json)."""
    g = _load("adaptive_budget.json")
    a = np.array(g["alpha"])
    ok = True
    for t in g["tables"].values():
        r = mod.adaptive_budget(a, t["cost_n"], t["cost_t"])
        ok &= r.N == t["N"] and r.budget.depth.tolist() == t["depth"]
        if "utility" in t:
            ok &= bool(np.allclose(r.utility, t["utility"], rtol=0, atol=1e-12))
            ok &= abs(r.margin - t["margin"]) < 1e-12
    return ok


def _adaptive_brute_pin(mod, seed=5):
    """N* against exhaustive search over every prefix-closed depth vector (tiny B, K)."""
    import itertools
    rng = np.random.default_rng(seed)
    for _ in range(20):
        B, K = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        a = rng.uniform(0, 1, (B, K)) ** 0.5
        cost_n = np.arange(B, B * (K + 1) + 1, dtype=np.float64)
        cost_t = np.cumsum(rng.uniform(0.1, 1.0, cost_n.size)) + rng.uniform(0, 3)   # increasing
        c = np.cumprod(a, axis=1)
        best = np.full(B * K + 1, -1.0)                  # the best expected tokens at each N
        for d in itertools.product(range(K + 1), repeat=B):
            n = sum(d)
            best[n] = max(best[n], sum(c[b, :d[b]].sum() for b in range(B)))
        U = (B + best) / np.interp(B + np.arange(B * K + 1), cost_n, cost_t)
        r = mod.adaptive_budget(a, cost_n, cost_t)
        if r.N != int(np.argmax(U)) or not np.allclose(r.utility, U, rtol=1e-12, atol=0):
            return False
    return True


def test_draft_confidence_golden():
    assert _draftconf_pin(O)


def test_draft_confidence_identities():
    rng = np.random.default_rng(3)
    zd = rng.normal(0, 2, (3, 4, 50))
    x = rng.integers(0, 50, (3, 4))
    q = O.draft_confidence(zd, x, 0.7)
    # a constant added to a row changes nothing; T scales the logits
    np.testing.assert_allclose(O.draft_confidence(zd + rng.normal(0, 5, (3, 4, 1)), x, 0.7), q, rtol=1e-12)
    np.testing.assert_allclose(O.draft_confidence(zd / 0.7, x, 1.0), q, rtol=1e-12)
    # one vocabulary entry: certainty; the greedy limit of a small temperature is the one-hot
    assert np.all(O.draft_confidence(zd[..., :1], np.zeros((3, 4), dtype=int), 0.9) == 1.0)
    zs = zd.copy()
    zs[np.arange(3)[:, None], np.arange(4)[None, :], x] += 10.0   # the drafted token leads by 10
    np.testing.assert_allclose(O.draft_confidence(zs, x, 1e-3), O.draft_confidence(zs, x, 0.0), atol=1e-12)


def test_draft_confidence_inverse_mean():
    """E_{x ~ q}[1 / q(x)] = V for a full-support q: the confidence is a normalised probability."""
    rng = np.random.default_rng(11)
    V, n = 6, 200000
    z = rng.normal(0, 1, V)
    q_true = np.exp(z) / np.exp(z).sum()       # only to draw x; the check uses the oracle's q(x)
    x = rng.choice(V, size=n, p=q_true)
    qx = O.draft_confidence(np.broadcast_to(z, (1, n, V)), x[None], 1.0)[0]
    inv = 1.0 / qx
    assert abs(inv.mean() - V) < 4 * inv.std() / np.sqrt(n)


def test_adaptive_budget_golden():
    assert _adaptive_pin(O)


def test_adaptive_budget_closed_forms():
    rng = np.random.default_rng(8)
    a = rng.uniform(0, 1, (5, 4))
    a[1, 2] = 0.0
    a[3, 0] = 0.0
    B, K = a.shape
    n = np.array([B, B * (K + 1)], dtype=np.float64)
    # constant cost: every key with positive confidence pays, a zero key adds nothing
    c = np.cumprod(a, axis=1)
    assert O.adaptive_budget(a, n, [2.0, 2.0]).N == int((c > 0).sum())
    # cost proportional to the positions verified: N = 0 is never beaten (confidences <= 1)
    assert O.adaptive_budget(a, n, n).N == 0


def test_adaptive_budget_exhaustive():
    assert _adaptive_brute_pin(O)


def test_pins_pass_on_the_real_oracle():
    assert _hist_pin(O) and _hand_pin(O) and _budget_pin(O) and _greedy_pin(O) and _icdf_pin(O)
    assert _margin_pin(O) and _budget_margin_pin(O) and _onehot_pin(O)
    assert _draftconf_pin(O) and _adaptive_pin(O) and _adaptive_brute_pin(O)


@pytest.mark.parametrize("old,new,pin", [
    ("ok = u[:, :K] * qx < px", "ok = u[:, :K] * px < qx", "hist"),                      # p/q swapped in the test
    ("resid = np.maximum(p_n - q_n, 0.0)", "resid = np.maximum(q_n - p_n, 0.0)", "hist"),  # residual sign
    ("resid = np.maximum(p_n - q_n, 0.0)", "resid = np.maximum(p_n - q_n, 0.0) * 0 + p_n", "hist"),  # no residual
    ("a = np.sum(np.minimum(p, q), axis=-1)", "a = np.sum(np.maximum(p, q), axis=-1)", "hand"),
    ("c = np.cumprod(alpha, axis=-1)", "c = np.cumsum(alpha, axis=-1)", "hand"),
    ("above = C > t[..., None]", "above = C >= t[..., None]", "icdf"),
    ("p_n = p[rows, n]", "p_n = p[rows, np.minimum(n + 1, K)]", "hand"),                 # off-by-one row
    ("order = np.lexsort((bf, mf, -cf))", "order = np.lexsort((mf, bf, -cf))", "budget"),  # tie order
    ("order = np.lexsort((bf, mf, -cf))", "order = np.lexsort((bf, mf, cf))", "budget"),   # ascending c
    ("return np.argmax(z, axis=-1)", "return z.shape[-1] - 1 - np.argmax(z[..., ::-1], axis=-1)", "greedy"),
    # decision margins: measured against u * R instead of u, one bin too early, the ratio inverted
    ("margin = np.minimum(np.abs(Cprev / R - u), np.abs(Cv / R - u))",
     "margin = np.minimum(np.abs(Cprev - u * R), np.abs(Cv - u * R))", "margin"),
    ("np.take_along_axis(C, np.maximum(v - 1, 0)[..., None], axis=-1)[..., 0], 0.0)",
     "np.take_along_axis(C, np.maximum(v - 2, 0)[..., None], axis=-1)[..., 0], 0.0)", "margin"),
    ("np.abs(u[:, :K] - px / qx)", "np.abs(u[:, :K] - qx / px)", "margin"),
    # budget margin between the wrong pair of ranked keys
    ("margin = abs(cf[order[n_sel - 1]] - cf[order[n_sel]])",
     "margin = abs(cf[order[max(n_sel - 2, 0)]] - cf[order[n_sel - 1]])", "budget_margin"),
    # T = 0 one-hot alpha comparing the target with itself
    ("alpha = (g[:, :K] == greedy_argmax(zd)).astype(np.float64)",
     "alpha = (g[:, :K] == greedy_argmax(zt[:, :K])).astype(np.float64)", "onehot"),
    ("alpha = (greedy_argmax(zt[:, :K]) == greedy_argmax(zd)).astype(np.float64)",
     "alpha = (greedy_argmax(zt[:, :K]) == greedy_argmax(zt[:, :K])).astype(np.float64)", "onehot"),
    # draft-side confidence: the draft's top probability instead of the drafted token's; T
    # ignored; the one-hot at the wrong index
    ("qx = np.take_along_axis(softmax(zd, T), xi[..., None], axis=-1)[..., 0]",
     "qx = softmax(zd, T).max(axis=-1)", "draftconf"),
    ("qx = np.take_along_axis(softmax(zd, T), xi[..., None], axis=-1)[..., 0]",
     "qx = np.take_along_axis(softmax(zd, 1.0), xi[..., None], axis=-1)[..., 0]", "draftconf"),
    ("qx = (greedy_argmax(zd) == xi).astype(np.float64)",
     "qx = (greedy_argmax(-zd) == xi).astype(np.float64)", "draftconf"),
    # utility: the B first positions forgotten in the yield or in the cost; ties to the largest N
    ("U = (B + S) / cost", "U = S / cost", "adaptive"),
    ("n_tok = B + np.arange(B * K + 1, dtype=np.float64)", "n_tok = np.arange(B * K + 1, dtype=np.float64)",
     "adaptive"),
    ("N = int(np.argmax(U))", "N = int(U.size - 1 - np.argmax(U[::-1]))", "adaptive"),
    ("S = np.concatenate([[0.0], np.cumsum(cf[ranked])])", "S = np.concatenate([[0.0], np.cumsum(cf)])",
     "adaptive_brute"),
])
def test_pins_catch_planted_mistakes(old, new, pin):
    mod = _mutant(old, new)
    check = {"hist": _hist_pin, "hand": _hand_pin, "budget": _budget_pin, "greedy": _greedy_pin,
             "icdf": _icdf_pin, "margin": _margin_pin, "budget_margin": _budget_margin_pin,
             "onehot": _onehot_pin, "draftconf": _draftconf_pin, "adaptive": _adaptive_pin,
             "adaptive_brute": _adaptive_brute_pin}[pin]
    assert not check(mod)
