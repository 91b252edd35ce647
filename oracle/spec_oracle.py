"""Float64 CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg do.  It shares no code, table or helper with the CUDA library.

It is written to be read against the AngelSpec pages (agifrontier tutorial,
section "KL to end-to-end TV loss", and section "runtime adaptation:
verification as a shared pool"):

* the acceptance probability of one drafted position is the overlap
  alpha(p, q) = sum_v min(p(v), q(v)) = 1 - TV(p, q)  (KL -> TV section,
  inline formula);
* acceptance is serial: the first rejected position voids every later draft
  (same paragraph);
* the expected number of accepted drafts of a depth-D chain is
  sum_{m<D} prod_{k<=m} alpha_k, the term inside L_e2e (display equation of
  that section);
* T = 0 is greedy decoding, T = 0.9 stochastic (same section, results);
* verification is a batch-level resource spent on high-confidence prefixes
  across requests (abstract; "shared pool" section).

The pages name rejection sampling that leaves the target distribution
unchanged but do not print its rule.  The oracle takes the standard
speculative-sampling rule, whose per-position acceptance probability is
exactly the alpha above: accept x ~ q iff u * q(x) < p(x); on the first
rejection emit a token from norm(max(0, p - q)); after full acceptance emit a
bonus token from p.  Inverse-CDF draws pick the smallest index whose
inclusive prefix mass is strictly above u * (computed total), in vocabulary
order.

Every input is float64 (bf16 / fp32 logits upcast exactly).  Requests are
handled as whole-array numpy operations; the vocabulary dimension uses numpy
reductions (max, exp, sum, minimum, cumsum, argmax) only, with no blocking
or reordering beyond what those library routines do.

Parity pins: every function here is pinned by tests that do not re-type its
formula (hand-computed golden cases, identities, brute-force histograms,
closed forms, exhaustive search); none is "parity unpinned".
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np


# --------------------------------------------------------------------------
# per-row building blocks
# --------------------------------------------------------------------------

def softmax(z: np.ndarray, T: float) -> np.ndarray:
    """Tempered softmax over the last axis: exp((z - max z) / T) / sum.

    The pages quote verification at a single temperature T for a run (T = 0
    and T = 0.9, KL -> TV section, results); the same T divides target and
    draft logits.  Logits of -inf get probability 0.
    """
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp((z - m) / T)
    return e / np.sum(e, axis=-1, keepdims=True)


def overlap_alpha(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """alpha(p, q) = sum_v min(p_v, q_v), clamped to [0, 1] (KL -> TV section, inline formula)."""
    a = np.sum(np.minimum(p, q), axis=-1)
    return np.clip(a, 0.0, 1.0)


def cumulative_alpha(alpha: np.ndarray):
    """Prefix confidences c_m = prod_{k<=m} alpha_k and E = sum_{m<K} c_m.

    E is the expected number of accepted drafts, the summand of L_e2e
    (KL -> TV section, display equation).  Works on [..., K] arrays.
    """
    c = np.cumprod(alpha, axis=-1)
    return c, np.sum(c, axis=-1)


def inverse_cdf(mass: np.ndarray, u):
    """Inverse-CDF draw, row by row: smallest v with C(v) > u * C(V-1).

    ``mass`` is [..., V] (non-negative, not necessarily normalised), ``u`` has
    the leading shape.  C is the inclusive prefix sum in vocabulary order.
    Returns (index, margin) where margin = min(|C(v-1)/R - u|, |C(v)/R - u|)
    with R = C(V-1) measures how close the draw was to a bin boundary.  If
    rounding leaves no index above the threshold, the last index with
    positive mass is taken (margin 0).
    """
    mass = np.asarray(mass, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    C = np.cumsum(mass, axis=-1)
    R = C[..., -1]
    t = u * R
    above = C > t[..., None]
    found = np.any(above, axis=-1)
    v = np.argmax(above, axis=-1)                       # first True
    V = mass.shape[-1]
    last_pos = V - 1 - np.argmax((mass > 0)[..., ::-1], axis=-1)
    v = np.where(found, v, last_pos)
    Cv = np.take_along_axis(C, v[..., None], axis=-1)[..., 0]
    Cprev = np.where(v > 0, np.take_along_axis(C, np.maximum(v - 1, 0)[..., None], axis=-1)[..., 0], 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        margin = np.minimum(np.abs(Cprev / R - u), np.abs(Cv / R - u))
    margin = np.where(found, margin, 0.0)
    return v, margin


def greedy_argmax(z: np.ndarray) -> np.ndarray:
    """argmax over the last axis, lowest index on ties (numpy's first occurrence)."""
    return np.argmax(z, axis=-1)


# --------------------------------------------------------------------------
# one batched verification call
# --------------------------------------------------------------------------

@dataclass
class VerifyResult:
    tokens: np.ndarray        # [B, K+1] int64, -1 after the emitted slot
    accepted: np.ndarray      # [B] int64, n_b accepted drafts (emitted = n_b + 1)
    alpha: np.ndarray         # [B, K] float64
    cum_alpha: np.ndarray     # [B, K] float64
    expected_len: np.ndarray  # [B] float64
    margin: np.ndarray        # [B] float64: smallest decision margin up to the cut
    depth: np.ndarray         # [B] int64 depth used
    margin_accept: Optional[np.ndarray] = None   # [B] smallest |u_k - p_k(x_k)/q_k(x_k)| over tested k
    margin_cdf: Optional[np.ndarray] = None      # [B] boundary distance of the final draw


def _first_false(ok: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Index of the first False among positions k < d[b] of ok[b, :], else d[b]."""
    B, K = ok.shape
    if K == 0:                      # nothing drafted: d is 0 and the chain ends at position 0
        return d.copy()
    k = np.arange(K)[None, :]
    stop = (~ok) & (k < d[:, None])
    return np.where(np.any(stop, axis=1), np.argmax(stop, axis=1), d)


def verify(target, draft, tokens, uniforms, T: float, depth=None, need_alpha: bool = True) -> VerifyResult:
    """Verify a batch of drafts against the target.

    target   [B, K+1, V] logits of the target at the K drafted positions and
             one more (the bonus position);
    draft    [B, K, V] draft logits (MTP chain or DFly block; the same rule
             applies to both, acceptance being serial in either case);
    tokens   [B, K] drafted token ids;
    uniforms [B, K+1]: u[b, k] tests position k, u[b, K] drives the one
             final draw (residual or bonus);
    depth    optional [B] verification depth d_b in [0, K] (from the budget);
             positions >= d_b are not verified and the bonus is drawn at d_b.

    T > 0: serial accept test u*q(x) < p(x); the first failing position n
    ends the chain and emits a draw from norm(max(0, p_n - q_n)); if all d_b
    positions pass, the bonus is drawn from p_{d_b}.  T = 0: accept iff
    x == argmax target, and the emitted token is the target argmax at the
    first mismatch (or at d_b).  At T = 0 alpha is the one-hot limit
    [argmax target == argmax draft].
    """
    zt = np.asarray(target, dtype=np.float64)
    zd = None if draft is None else np.asarray(draft, dtype=np.float64)
    x = np.asarray(tokens, dtype=np.int64)
    u = np.asarray(uniforms, dtype=np.float64)
    B, K1, V = zt.shape
    K = K1 - 1
    d = np.full(B, K, dtype=np.int64) if depth is None else np.clip(np.asarray(depth, dtype=np.int64), 0, K)
    rows = np.arange(B)
    alpha = np.zeros((B, K))
    margin = np.full(B, np.inf)
    m_acc = np.full(B, np.inf)
    m_cdf = np.full(B, np.inf)

    if T == 0.0:
        g = greedy_argmax(zt)                                   # [B, K+1]
        if zd is not None and need_alpha and K > 0:
            alpha = (g[:, :K] == greedy_argmax(zd)).astype(np.float64)
        n = _first_false(x == g[:, :K], d)
        final = g[rows, n]
    else:
        p = softmax(zt, T)                                      # [B, K+1, V]
        q = softmax(zd, T)                                      # [B, K, V]
        if K > 0:
            alpha = overlap_alpha(p[:, :K], q)
        xs = np.clip(x, 0, V - 1)
        px = np.take_along_axis(p[:, :K], xs[..., None], axis=-1)[..., 0]   # [B, K]
        qx = np.take_along_axis(q, xs[..., None], axis=-1)[..., 0]
        ok = u[:, :K] * qx < px
        n = _first_false(ok, d)
        kk = np.arange(K)[None, :]
        tested = (kk <= n[:, None]) & (kk < d[:, None])         # positions whose test ran
        with np.errstate(divide="ignore", invalid="ignore"):
            acc_margin = np.where(tested & (qx > 0), np.abs(u[:, :K] - px / qx), np.inf)
        if K > 0:
            m_acc = acc_margin.min(axis=1)
            margin = np.minimum(margin, m_acc)
        rejected = n < d
        # final-draw distribution per request: residual at n if rejected, else p at n (= d)
        p_n = p[rows, n]                                        # [B, V]
        q_n = q[rows, np.minimum(n, K - 1)] if K > 0 else np.zeros_like(p_n)
        resid = np.maximum(p_n - q_n, 0.0)
        use_resid = rejected & (np.sum(resid, axis=-1) > 0)     # residual mass 0 only if p == q
        mass = np.where(use_resid[:, None], resid, p_n)
        final, m_cdf = inverse_cdf(mass, u[:, K])
        margin = np.minimum(margin, m_cdf)

    out = np.full((B, K + 1), -1, dtype=np.int64)
    for b in range(B):
        out[b, :n[b]] = x[b, :n[b]]
        out[b, n[b]] = final[b]
    cum, E = cumulative_alpha(alpha)
    return VerifyResult(out, n.astype(np.int64), alpha, cum, E, margin, d, m_acc, m_cdf)


def overlap_stats(target, draft, T: float):
    """alpha, prefix confidences and expected length only (no decisions).

    Reads target rows 0..K-1 of [B, K+1, V] against draft rows [B, K, V].
    """
    zt = np.asarray(target, dtype=np.float64)
    zd = np.asarray(draft, dtype=np.float64)
    K = zd.shape[1]
    if T == 0.0:
        alpha = (greedy_argmax(zt[:, :K]) == greedy_argmax(zd)).astype(np.float64)
    else:
        alpha = overlap_alpha(softmax(zt[:, :K], T), softmax(zd, T))
    c, E = cumulative_alpha(alpha)
    return alpha, c, E


# --------------------------------------------------------------------------
# batch-level verification budget (D-cut selection)
# --------------------------------------------------------------------------

@dataclass
class BudgetResult:
    depth: np.ndarray    # [B] int64
    conf: np.ndarray     # [B, K] prefix confidences
    margin: float        # |c_(N) - c_(N+1)| between the last selected and first dropped key


def alloc_budget(alpha, N: int) -> BudgetResult:
    """Spend a global budget of N verified positions on the best prefixes.

    Keys are the prefix confidences c[b, m] = prod_{k<=m} alpha[b, k]
    (alpha clamped to [0, 1] first), ordered by c descending, then m
    ascending, then b ascending; the first min(N, B*K) keys are selected and
    d_b counts the selected keys of request b.  Because c is non-increasing
    in m and ties go to the smaller m, the selection is prefix-closed, so it
    is a valid per-request verification depth.
    """
    a = np.clip(np.nan_to_num(np.asarray(alpha, dtype=np.float64), nan=0.0), 0.0, 1.0)
    B, K = a.shape
    c, _ = cumulative_alpha(a)
    bb, mm = np.meshgrid(np.arange(B), np.arange(K), indexing="ij")
    cf, mf, bf = c.ravel(), mm.ravel(), bb.ravel()
    order = np.lexsort((bf, mf, -cf))        # primary key last: -c, then m, then b
    n_sel = int(min(max(N, 0), B * K))
    depth = np.zeros(B, dtype=np.int64)
    for i in order[:n_sel]:
        depth[bf[i]] += 1
    if 0 < n_sel < B * K:
        margin = abs(cf[order[n_sel - 1]] - cf[order[n_sel]])
    else:
        margin = np.inf
    return BudgetResult(depth, c, margin)


# --------------------------------------------------------------------------
# draft-side confidence: the budget chosen before the target forward
# --------------------------------------------------------------------------

def draft_confidence(draft, tokens, T: float) -> np.ndarray:
    """q_k(x_k): the probability the draft model gave the token it drafted, [B, K].

    The runtime section of the AngelSpec page selects what to verify from the draft model's
    output distribution, before the target runs; the per-position confidence read here is
    q_k(x_k) = softmax(z_D[b, k] / T)[x_k].  At T = 0 the draft distribution is the one-hot
    at its argmax (lowest index on ties), so q_k(x_k) = [x_k == argmax z_D[b, k]].  A token
    outside [0, V) has confidence 0.
    """
    zd = np.asarray(draft, dtype=np.float64)
    x = np.asarray(tokens, dtype=np.int64)
    V = zd.shape[-1]
    ok = (x >= 0) & (x < V)
    xi = np.where(ok, x, 0)
    if T == 0.0:
        qx = (greedy_argmax(zd) == xi).astype(np.float64)
    else:
        qx = np.take_along_axis(softmax(zd, T), xi[..., None], axis=-1)[..., 0]
    return np.where(ok, qx, 0.0)


def draft_budget(draft, tokens, T: float, N: int) -> BudgetResult:
    """The budget of alloc_budget spent on draft-side prefix confidences prod_{k<=m} q_k(x_k)."""
    return alloc_budget(draft_confidence(draft, tokens, T), N)


# --------------------------------------------------------------------------
# utility / cost choice of the budget N
# --------------------------------------------------------------------------

@dataclass
class AdaptiveResult:
    N: int                # the chosen budget
    utility: np.ndarray   # [B*K + 1]: U(N) for every N
    budget: BudgetResult  # the selection at the chosen N
    margin: float         # (U(N*) - best U(N), N != N*) / U(N*); inf when there is one candidate


def adaptive_budget(alpha, cost_n, cost_t) -> AdaptiveResult:
    """Choose N online: maximise the expected tokens per unit of verification cost.

    The runtime section of the AngelSpec page spends verification where it pays, against a
    profiled cost of verifying more positions.  With keys ordered as in alloc_budget and S(N)
    the sum of the first N prefix confidences (the expected accepted drafts of the selection),
    a batch of B requests that verifies B + N positions (every request verifies its first
    emitted position) yields B + S(N) tokens, so

        U(N) = (B + S(N)) / cost(B + N),   N = 0 .. B*K,

    where cost is the piecewise-linear interpolation of the table (cost_n ascending, cost_t),
    held constant beyond its ends (numpy.interp).  N* is the first N with the largest U.
    """
    a = np.clip(np.nan_to_num(np.asarray(alpha, dtype=np.float64), nan=0.0), 0.0, 1.0)
    B, K = a.shape
    c, _ = cumulative_alpha(a)
    bb, mm = np.meshgrid(np.arange(B), np.arange(K), indexing="ij")
    cf, mf, bf = c.ravel(), mm.ravel(), bb.ravel()
    ranked = np.lexsort((bf, mf, -cf))       # the key order of alloc_budget
    S = np.concatenate([[0.0], np.cumsum(cf[ranked])])
    n_tok = B + np.arange(B * K + 1, dtype=np.float64)
    cost = np.interp(n_tok, np.asarray(cost_n, dtype=np.float64), np.asarray(cost_t, dtype=np.float64))
    U = (B + S) / cost
    N = int(np.argmax(U))
    if U.size > 1:
        rest = np.delete(U, N)
        margin = float((U[N] - rest.max()) / U[N])
    else:
        margin = np.inf
    return AdaptiveResult(N, U, alloc_budget(a, N), margin)


def verify_budgeted(target, draft, tokens, uniforms, T: float, N: int):
    """alpha for every position, the budget selection, then verification to depth d_b."""
    alpha, _, _ = overlap_stats(target, draft, T)
    br = alloc_budget(alpha, N)
    vr = verify(target, draft, tokens, uniforms, T, depth=br.depth)
    return vr, br
