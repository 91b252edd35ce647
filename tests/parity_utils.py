"""Compare the CUDA path with the float64 oracle under the match rules.

* T = 0: tokens, accepted counts and depths bit-exact; alpha (one-hot) exact.
* T > 0: tokens and accepted counts bit-exact for every request whose
  smallest decision margin (accept test |u - p/q|, inverse-CDF boundary
  distance) is >= 1e-5; requests below are counted as ambiguous and only
  checked for validity.  alpha and prefix confidences within 1e-5 absolute,
  expected length within 1e-4 (a sum of up to K prefix products).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import spec_oracle as O

MARGIN = 1e-5
ALPHA_ATOL = 1e-5
CUM_ATOL = 1e-5
E_ATOL = 1e-4


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy() if t.is_floating_point() else t.detach().cpu().numpy()


def oracle_verify(w, depth=None, need_alpha=True, chunk=8):
    """Oracle over request chunks (requests are independent), upcasting exactly to float64."""
    parts = []
    for s in range(0, w.B, chunk):
        e = min(w.B, s + chunk)
        zt = w.target[s:e].to(torch.float64).numpy()
        zd = w.draft[s:e].to(torch.float64).numpy() if w.K > 0 else np.zeros((e - s, 0, w.V))
        d = None if depth is None else np.asarray(depth)[s:e]
        parts.append(O.verify(zt, zd, w.tokens[s:e].numpy(), w.uniforms[s:e].double().numpy(),
                              w.temperature, depth=d, need_alpha=need_alpha))
    cat = lambda f: np.concatenate([getattr(p, f) for p in parts])  # noqa: E731
    return O.VerifyResult(cat("tokens"), cat("accepted"), cat("alpha"), cat("cum_alpha"),
                          cat("expected_len"), cat("margin"), cat("depth"))


def oracle_alpha(w, chunk=8):
    al = []
    for s in range(0, w.B, chunk):
        e = min(w.B, s + chunk)
        a, _, _ = O.overlap_stats(w.target[s:e].to(torch.float64).numpy(),
                                  w.draft[s:e].to(torch.float64).numpy(), w.temperature)
        al.append(a)
    return np.concatenate(al)


def check_valid_tokens(tokens, accepted, x, V, K):
    B = tokens.shape[0]
    for b in range(B):
        n = int(accepted[b])
        assert 0 <= n <= K
        assert np.all(tokens[b, :n] == x[b, :n])
        assert 0 <= tokens[b, n] < V
        assert np.all(tokens[b, n + 1:] == -1)


def consistent_within(w, b, tokens_row, n, d, tol=MARGIN):
    """An ambiguous request's GPU decisions agree with the oracle's float64 probabilities up to tol.

    Accepted positions need u - p/q < tol, the rejecting one u - p/q > -tol, and the emitted
    token's inverse-CDF bin [C(v-1)/R, C(v)/R] (residual or p) must contain u[b, K] within tol.
    """
    T, K = w.temperature, w.K
    zt = w.target[b].to(torch.float64).numpy()
    zd = w.draft[b].to(torch.float64).numpy()
    u = w.uniforms[b].double().numpy()
    x = w.tokens[b].numpy()
    p, q = O.softmax(zt, T), O.softmax(zd, T)
    for k in range(min(n + 1, d)):
        px, qx = p[k, x[k]], q[k, x[k]]
        ratio = px / qx if qx > 0 else (np.inf if px > 0 else -np.inf)
        if k < n and not (u[k] - ratio < tol):
            return False
        if k == n and not (u[k] - ratio > -tol):
            return False
    if n < d:
        mass = np.maximum(p[n] - q[n], 0.0)
        if mass.sum() <= 0:
            mass = p[n]
    else:
        mass = p[n]
    v = int(tokens_row[n])
    if not (0 <= v < w.V) or mass[v] <= 0:
        return False
    C = np.cumsum(mass) / mass.sum()
    lo = C[v - 1] if v > 0 else 0.0
    return lo - tol <= u[K] <= C[v] + tol


def compare(gpu, ref, w, check_alpha=True):
    """Returns the number of ambiguous requests (T > 0); asserts everything else.

    Ambiguous requests (a decision margin below 1e-5 in the oracle) are not compared
    token by token; their GPU decisions must instead be consistent with the float64
    probabilities within that margin.
    """
    tok = gpu.tokens.cpu().numpy()
    acc = gpu.accepted.cpu().numpy()
    check_valid_tokens(tok, acc, w.tokens.numpy(), w.V, w.K)
    if w.temperature == 0.0:
        np.testing.assert_array_equal(tok, ref.tokens)
        np.testing.assert_array_equal(acc, ref.accepted)
        if check_alpha and gpu.alpha is not None:
            np.testing.assert_array_equal(to_np(gpu.alpha), ref.alpha)
        amb = 0
    else:
        ok = ref.margin >= MARGIN
        amb = int((~ok).sum())
        bad = np.nonzero(ok & ((acc != ref.accepted) | np.any(tok != ref.tokens, axis=1)))[0]
        assert bad.size == 0, (f"{bad.size} unambiguous requests differ, e.g. b={bad[:5]} "
                               f"gpu={tok[bad[:3]]} ref={ref.tokens[bad[:3]]} margin={ref.margin[bad[:3]]}")
        for b in np.nonzero(~ok)[0]:
            assert consistent_within(w, int(b), tok[b], int(acc[b]), int(ref.depth[b])), (
                f"ambiguous request {b} inconsistent: gpu={tok[b]} ref={ref.tokens[b]} margin={ref.margin[b]}")
        if check_alpha and gpu.alpha is not None:
            np.testing.assert_allclose(to_np(gpu.alpha), ref.alpha, atol=ALPHA_ATOL, rtol=0)
    if check_alpha and getattr(gpu, "cum_alpha", None) is not None:
        np.testing.assert_allclose(to_np(gpu.cum_alpha), ref.cum_alpha, atol=CUM_ATOL, rtol=0)
        np.testing.assert_allclose(to_np(gpu.expected_len), ref.expected_len, atol=E_ATOL, rtol=0)
    return amb
