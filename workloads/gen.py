"""Seeded synthetic inputs for batched draft verification.

This module only draws random numbers and lays them out; it computes nothing
that the verification method computes.  Both the float64 oracle (through the
tests) and the CUDA path read the same tensors from here.

Every workload mirrors one configuration of the verification problem:
target logits ``[B, K+1, V]``, draft logits ``[B, K, V]``, draft tokens
``[B, K]`` (int32), uniforms ``[B, K+1]`` (float32, U(0,1)) and a temperature.
Logits are drawn in float32 and rounded once to the stated storage dtype
(bfloat16 rounding is round-to-nearest-even, done by torch), so the oracle
sees exactly the values the GPU reads after an exact upcast.

Recipes (the distribution shapes follow the verification configurations of
the AngelSpec / DFly pages: an MTP chain of depth 3 and a DFly block of 16):

* ``tiny_chain``      B=1, K=3, V=1024, fp32, z_T ~ N(0, 2^2),
                      z_D = z_T + N(0, 0.7^2), T = 1.0.
* ``greedy_mtp``      B=64, K=3, V=128000, bf16, z_T ~ N(0, 3^2) plus one +8
                      peak at a random index per row, z_D = z_T + N(0, 1),
                      T = 0, draft tokens = argmax of the draft row.
* ``stochastic_mtp``  B=64, K=3, V=128000, bf16, Zipf-shaped target
                      z_T[v] = -1.1 ln(rank_v) + N(0, 0.5^2) with rank a random
                      permutation of 1..V per row, z_D = z_T + N(0, 0.8^2),
                      T = 0.9.
* ``dfly_block``      B=32, K=16, V=128000, bf16, Zipf-shaped target, draft
                      noise sigma_k = 0.3 + 1.2 k / 15 along the block, T=0.9.
* ``budget_sweep``    B in {4,8,16,32,64}, K=16, V=128000, bf16, Zipf-shaped
                      target, per-request sigma ~ U(0.3, 1.5) constant along
                      the block, T = 0.9, budget N = 8 B.

At T > 0 the draft tokens are drawn from the draft's own tempered
distribution with the Gumbel-max trick (argmax of z_D / T + Gumbel noise),
which needs no normalisation; at T = 0 they are the draft argmax.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class Workload:
    name: str
    target: torch.Tensor            # [B, K+1, V] float32 or bfloat16 (CPU)
    draft: torch.Tensor             # [B, K, V]   same dtype (CPU)
    tokens: torch.Tensor            # [B, K] int32
    uniforms: torch.Tensor          # [B, K+1] float32 in [0, 1)
    temperature: float
    budget: Optional[int] = None    # global verification budget N, if any
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.target.shape[0]

    @property
    def K(self) -> int:
        return self.draft.shape[1]

    @property
    def V(self) -> int:
        return self.target.shape[2]

    def logits_bytes(self, with_draft: bool = True) -> int:
        e = self.target.element_size()
        n = self.target.numel() + (self.draft.numel() if with_draft else 0)
        return n * e


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _zipf_target(g: torch.Generator, B: int, R: int, V: int) -> torch.Tensor:
    """Zipf-shaped logits: -1.1 ln(rank) + N(0, 0.5^2), rank a per-row permutation."""
    perm = torch.argsort(torch.rand(B * R, V, generator=g), dim=1)  # values 0..V-1
    rank = (perm + 1).to(torch.float32)
    z = -1.1 * torch.log(rank) + 0.5 * torch.randn(B * R, V, generator=g)
    return z.view(B, R, V)


def _draft_tokens(g: torch.Generator, draft32: torch.Tensor, T: float) -> torch.Tensor:
    """Draft tokens: Gumbel-max sample from the tempered draft row, or argmax at T=0."""
    if T == 0.0:
        return torch.argmax(draft32, dim=-1).to(torch.int32)
    u = torch.rand(draft32.shape, generator=g).clamp_(min=1e-12, max=1.0 - 1e-7)
    gumbel = -torch.log(-torch.log(u))
    return torch.argmax(draft32 / T + gumbel, dim=-1).to(torch.int32)


def _finish(name, target32, draft32, dtype, T, g_tok, g_u, budget=None, meta=None) -> Workload:
    target = target32.to(dtype).contiguous()
    draft = draft32.to(dtype).contiguous()
    # draft tokens are drawn from the rounded draft logits the verifier sees
    tokens = _draft_tokens(g_tok, draft.to(torch.float32), T).contiguous()
    B, K1, _ = target.shape
    uniforms = torch.rand(B, K1, generator=g_u, dtype=torch.float32).contiguous()
    return Workload(name, target, draft, tokens, uniforms, float(T), budget, meta or {})


def tiny_chain(seed: int = 0, B: int = 1, K: int = 3, V: int = 1024, T: float = 1.0) -> Workload:
    g = _gen(seed)
    zt = 2.0 * torch.randn(B, K + 1, V, generator=g)
    zd = zt[:, :K] + 0.7 * torch.randn(B, K, V, generator=g)
    return _finish("tiny_chain", zt, zd, torch.float32, T, _gen(seed + 1000), _gen(seed))


def greedy_mtp(seed: int = 1, B: int = 64, K: int = 3, V: int = 128000,
               dtype=torch.bfloat16) -> Workload:
    g = _gen(seed)
    zt = 3.0 * torch.randn(B, K + 1, V, generator=g)
    peak = torch.randint(0, V, (B, K + 1), generator=g)
    zt.scatter_add_(2, peak.unsqueeze(-1), torch.full((B, K + 1, 1), 8.0))
    zd = zt[:, :K] + torch.randn(B, K, V, generator=g)
    return _finish("greedy_mtp", zt, zd, dtype, 0.0, _gen(seed + 1000), _gen(seed + 2000))


def stochastic_mtp(seed: int = 2, B: int = 64, K: int = 3, V: int = 128000,
                   T: float = 0.9, sigma: float = 0.8, dtype=torch.bfloat16) -> Workload:
    g = _gen(seed)
    zt = _zipf_target(g, B, K + 1, V)
    zd = zt[:, :K] + sigma * torch.randn(B, K, V, generator=g)
    return _finish("stochastic_mtp", zt, zd, dtype, T, _gen(seed + 1000), _gen(seed + 2000))


def dfly_block(seed: int = 3, B: int = 32, K: int = 16, V: int = 128000,
               T: float = 0.9, dtype=torch.bfloat16) -> Workload:
    g = _gen(seed)
    zt = _zipf_target(g, B, K + 1, V)
    k = torch.arange(K, dtype=torch.float32)
    sig = 0.3 + 1.2 * k / max(K - 1, 1)
    zd = zt[:, :K] + sig.view(1, K, 1) * torch.randn(B, K, V, generator=g)
    return _finish("dfly_block", zt, zd, dtype, T, _gen(seed + 1000), _gen(seed + 2000),
                   meta={"sigma": sig.tolist()})


def budget_sweep(B: int = 64, seed: int = 4, K: int = 16, V: int = 128000,
                 T: float = 0.9, dtype=torch.bfloat16, budget_per_req: int = 8) -> Workload:
    g = _gen(seed * 100 + B)
    zt = _zipf_target(g, B, K + 1, V)
    sig = 0.3 + 1.2 * torch.rand(B, generator=g)
    zd = zt[:, :K] + sig.view(B, 1, 1) * torch.randn(B, K, V, generator=g)
    return _finish("budget_sweep", zt, zd, dtype, T, _gen(seed * 100 + B + 1000),
                   _gen(seed * 100 + B + 2000), budget=budget_per_req * B,
                   meta={"sigma": sig.tolist()})


def random_case(seed: int, B: int, K: int, V: int, T: float, dtype=torch.float32,
                scale: float = 2.0, noise: float = 0.7) -> Workload:
    """A general Gaussian case of any shape (ragged V, small B/K) for parity sweeps."""
    g = _gen(seed)
    zt = scale * torch.randn(B, K + 1, V, generator=g)
    zd = zt[:, :K] + noise * torch.randn(B, K, V, generator=g)
    return _finish(f"random_{B}x{K}x{V}", zt, zd, dtype, T, _gen(seed + 1000), _gen(seed + 2000))


def verify_cost_table(B: int, K: int, points: int = 9):
    """A synthetic cost profile of verifying n positions in one target forward (arbitrary units),
    standing in for the profiled table a serving system would measure: flat up to 4 positions per
    request (the forward is bound by reading weights), then rising with n (bound by compute).
    Returns (n, cost) as float lists, n from B to B * (K + 1)."""
    lo, hi = float(B), float(B * (K + 1))
    n = [lo + (hi - lo) * i / (points - 1) for i in range(points)]
    knee = 4.0 * B
    return n, [1.0 + 0.02 * x / B + max(0.0, x - knee) * 0.25 / B for x in n]


CONFIGS = {
    "tiny_chain": tiny_chain,
    "greedy_mtp": greedy_mtp,
    "stochastic_mtp": stochastic_mtp,
    "dfly_block": dfly_block,
    "budget_sweep": budget_sweep,
}
