"""Batched draft verification for speculative decoding on GB300 (sm_103a).

Thin Python binding over the C ABI of libspecverify.so: it checks tensor
dtype / device / contiguity, allocates outputs with torch, and passes raw
device pointers.  Every step of the verification runs in the library's CUDA
kernels; nothing here computes on the data.

    from draft_verification_spec_gb300 import verify_chain, verify_block
    out = verify_chain(target, draft, tokens, uniforms, temperature=0.9)
    out.tokens, out.accepted          # [B, K+1] int32, [B] int32

The operation follows the AngelSpec / DFly description of verification:
alpha = sum min(p, q) = 1 - TV, serial acceptance with a first-rejection cut,
residual / bonus draws, greedy argmax matching at T = 0, and a batch-level
budget over prefix confidences prod alpha.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib

SPEC_F32, SPEC_BF16 = 0, 1
STATUS_NAMES = {0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_UNSUPPORTED", 3: "SPEC_ERR_CUDA",
                4: "SPEC_ERR_DEVICE_TIMEOUT", 5: "SPEC_ERR_TOKEN_RANGE", 6: "SPEC_ERR_WORKSPACE"}


class SpecError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} "
                         f"({lib().spec_error_string(code).decode()})")


def lib():
    return _lib.load()


def _check(code: int, where: str):
    if code != 0:
        raise SpecError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _need(t: Optional[torch.Tensor], name: str, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


class Workspace:
    """Device workspace of the library (status word, per-request counters, per-row records).

    Zero-filled once when (re)allocated; the kernels keep it consistent.  One
    workspace per stream: calls that share one must be ordered on a stream.
    """

    def __init__(self, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.buf: Optional[torch.Tensor] = None

    def get(self, B: int, K: int, V: int, dtype_code: int, stream) -> torch.Tensor:
        need = int(lib().spec_workspace_bytes(B, K, V, dtype_code))
        if self.buf is None or self.buf.numel() < need:
            # torch's allocator returns 512-byte aligned blocks (>= the 256 the library requires)
            self.buf = torch.empty(max(need, 4096), dtype=torch.uint8, device=self.device)
            _check(lib().spec_workspace_init(_ptr(self.buf), self.buf.numel(), _stream_ptr(stream)),
                   "spec_workspace_init")
        return self.buf

    def status(self, stream=None) -> int:
        """Read and clear the device status word (synchronises the stream)."""
        if self.buf is None:
            return 0
        out = ctypes.c_int32(0)
        _check(lib().spec_get_status(_ptr(self.buf), _stream_ptr(stream), ctypes.byref(out)), "spec_get_status")
        return out.value

    def reset(self, stream=None):
        if self.buf is not None:
            _check(lib().spec_workspace_init(_ptr(self.buf), self.buf.numel(), _stream_ptr(stream)),
                   "spec_workspace_init")


_workspaces: dict = {}


def default_workspace(stream=None) -> Workspace:
    s = torch.cuda.current_stream() if stream is None else stream
    key = (s.device.index if s.device.index is not None else torch.cuda.current_device(), s.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None:
        ws = Workspace(torch.device("cuda", key[0]))
        _workspaces[key] = ws
    return ws


@dataclass
class VerifyOutput:
    tokens: torch.Tensor                    # [B, K+1] int32; -1 after the emitted slot
    accepted: torch.Tensor                  # [B] int32
    alpha: Optional[torch.Tensor] = None    # [B, K] float32
    cum_alpha: Optional[torch.Tensor] = None
    expected_len: Optional[torch.Tensor] = None
    depth: Optional[torch.Tensor] = None


class Tuning:
    """Per-call test and tuning knobs (spec_tuning_t); the defaults leave every choice to the library.

    wait_limit_us: 0 default (200 ms), > 0 a limit, < 0 every bounded device wait gives up at once.
    cluster: sampling kernel CTAs per row (0 automatic).  greedy_variant: bit 1 separate cut kernel,
    bit 2 every resident CTA slot.  split_event: a torch.cuda.Event recorded between the row kernel
    and the kernel chained after it.  After the call, ``plan`` holds the launched plan.
    """

    KEYS = ("threads", "cluster", "clusters", "max_clusters", "slice", "items", "smem_bytes", "flags")

    def __init__(self, wait_limit_us: int = 0, cluster: int = 0, greedy_variant: int = 0, split_event=None):
        self._plan = (ctypes.c_int32 * 8)()
        ev = None if split_event is None else ctypes.c_void_p(split_event.cuda_event)
        self._c = _lib.SpecTuning(int(wait_limit_us), int(cluster), int(greedy_variant),
                                  ctypes.cast(self._plan, ctypes.c_void_p), ev)

    @property
    def plan(self) -> dict:
        return dict(zip(self.KEYS, list(self._plan)))

    def ref(self):
        return ctypes.byref(self._c)


def _validate(target, draft, tokens, uniforms, temperature, draft_needed, tokens_needed=True):
    if target.dim() != 3:
        raise ValueError("target logits must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    _need(target, "target", shape=(B, K1, V))
    code = _dtype_code(target)
    if draft is not None:
        _need(draft, "draft", dtype=target.dtype, shape=(B, K, V), device=dev)
    elif draft_needed:
        raise ValueError("draft logits are required here")
    if K > 0 and tokens_needed:
        if tokens is None:
            raise ValueError("tokens [B, K] are required")
        _need(tokens, "tokens", dtype=torch.int32, shape=(B, K), device=dev)
    if temperature > 0 and tokens_needed:
        if uniforms is None:
            raise ValueError("uniforms [B, K+1] are required at T > 0")
        _need(uniforms, "uniforms", dtype=torch.float32, shape=(B, K1), device=dev)
    return B, K, V, code


def verify_chain(target, draft, tokens, uniforms, temperature: float, depth=None, want_alpha=False,
                 stream=None, workspace: Optional[Workspace] = None, out: Optional[VerifyOutput] = None,
                 tuning: Optional[Tuning] = None):
    """MTP-chain verification (spec_verify_chain; spec_verify_tuned when `tuning` is given)."""
    B, K, V, code = _validate(target, draft, tokens, uniforms, temperature,
                              draft_needed=(K_pos(target) > 0 and (temperature > 0 or want_alpha)))
    dev = target.device
    if depth is not None:
        _need(depth, "depth", dtype=torch.int32, shape=(B,), device=dev)
    if out is None:
        out = VerifyOutput(torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                           torch.empty(B, dtype=torch.int32, device=dev),
                           torch.empty(B, K, dtype=torch.float32, device=dev) if want_alpha else None)
    ws = (workspace or default_workspace(stream))
    buf = ws.get(B, K, V, code, stream)
    if tuning is not None:
        _check(lib().spec_verify_tuned(_ptr(target), _ptr(draft), code, _ptr(tokens), _ptr(uniforms), B, K, V,
                                       float(temperature), _ptr(depth), -1, 0, _ptr(out.tokens),
                                       _ptr(out.accepted), _ptr(out.alpha), None, None, None, _ptr(buf),
                                       buf.numel(), _stream_ptr(stream), tuning.ref()), "spec_verify_tuned")
        return out
    _check(lib().spec_verify_chain(_ptr(target), _ptr(draft), code, _ptr(tokens), _ptr(uniforms), B, K, V,
                                   float(temperature), _ptr(depth), _ptr(out.tokens), _ptr(out.accepted),
                                   _ptr(out.alpha), _ptr(buf), buf.numel(), _stream_ptr(stream)),
           "spec_verify_chain")
    return out


def K_pos(target) -> int:
    return int(target.shape[1]) - 1


def verify_block(target, draft, tokens, uniforms, temperature: float, depth=None, budget: Optional[int] = None,
                 want_stats=True, stream=None, workspace: Optional[Workspace] = None,
                 out: Optional[VerifyOutput] = None, tuning: Optional[Tuning] = None):
    """DFly-block verification (spec_verify_block): alpha, prefix confidences, expected length,
    and optionally the batch-level budget (depth chosen in the same call)."""
    need_draft = K_pos(target) > 0 and (temperature > 0 or want_stats or budget is not None)
    B, K, V, code = _validate(target, draft, tokens, uniforms, temperature, draft_needed=need_draft)
    dev = target.device
    if depth is not None:
        _need(depth, "depth", dtype=torch.int32, shape=(B,), device=dev)
    if out is None:
        f = lambda *s: torch.empty(*s, dtype=torch.float32, device=dev)  # noqa: E731
        out = VerifyOutput(torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                           torch.empty(B, dtype=torch.int32, device=dev),
                           f(B, K) if want_stats else None, f(B, K) if want_stats else None,
                           f(B) if want_stats else None,
                           torch.empty(B, dtype=torch.int32, device=dev) if budget is not None else None)
    ws = (workspace or default_workspace(stream))
    buf = ws.get(B, K, V, code, stream)
    if tuning is not None:
        _check(lib().spec_verify_tuned(_ptr(target), _ptr(draft), code, _ptr(tokens), _ptr(uniforms), B, K, V,
                                       float(temperature), _ptr(depth), -1 if budget is None else int(budget), 0,
                                       _ptr(out.tokens), _ptr(out.accepted), _ptr(out.alpha), _ptr(out.cum_alpha),
                                       _ptr(out.expected_len), _ptr(out.depth), _ptr(buf), buf.numel(),
                                       _stream_ptr(stream), tuning.ref()), "spec_verify_tuned")
        return out
    _check(lib().spec_verify_block(_ptr(target), _ptr(draft), code, _ptr(tokens), _ptr(uniforms), B, K, V,
                                   float(temperature), _ptr(depth), -1 if budget is None else int(budget),
                                   _ptr(out.tokens), _ptr(out.accepted), _ptr(out.alpha), _ptr(out.cum_alpha),
                                   _ptr(out.expected_len), _ptr(out.depth), _ptr(buf), buf.numel(),
                                   _stream_ptr(stream)),
           "spec_verify_block")
    return out


def overlap_alpha(target, draft, temperature: float, stream=None, workspace: Optional[Workspace] = None,
                  tuning: Optional[Tuning] = None):
    """alpha [B, K], prefix confidences [B, K], expected length [B] (spec_overlap_alpha)."""
    B, K, V, code = _validate(target, draft, None, None, temperature, draft_needed=True, tokens_needed=False)
    dev = target.device
    alpha = torch.empty(B, K, dtype=torch.float32, device=dev)
    cum = torch.empty(B, K, dtype=torch.float32, device=dev)
    E = torch.empty(B, dtype=torch.float32, device=dev)
    ws = (workspace or default_workspace(stream))
    buf = ws.get(B, K, V, code, stream)
    if tuning is not None:
        _check(lib().spec_verify_tuned(_ptr(target), _ptr(draft), code, None, None, B, K, V, float(temperature),
                                       None, -1, 1, None, None, _ptr(alpha), _ptr(cum), _ptr(E), None, _ptr(buf),
                                       buf.numel(), _stream_ptr(stream), tuning.ref()), "spec_verify_tuned")
        return alpha, cum, E
    _check(lib().spec_overlap_alpha(_ptr(target), _ptr(draft), code, B, K, V, float(temperature), _ptr(alpha),
                                    _ptr(cum), _ptr(E), _ptr(buf), buf.numel(), _stream_ptr(stream)),
           "spec_overlap_alpha")
    return alpha, cum, E


def alloc_budget(alpha, budget: int, stream=None, workspace: Optional[Workspace] = None):
    """Per-request depth [B] int32 and prefix confidences [B, K] (spec_alloc_budget)."""
    B, K = alpha.shape
    _need(alpha, "alpha", dtype=torch.float32, shape=(B, K))
    dev = alpha.device
    depth = torch.empty(B, dtype=torch.int32, device=dev)
    conf = torch.empty(B, K, dtype=torch.float32, device=dev)
    ws = (workspace or default_workspace(stream))
    buf = ws.get(B, K, 1, SPEC_F32, stream)
    _check(lib().spec_alloc_budget(_ptr(alpha), B, K, int(budget), _ptr(depth), _ptr(conf), _ptr(buf),
                                   buf.numel(), _stream_ptr(stream)), "spec_alloc_budget")
    return depth, conf


def _cost_table(cost, dev):
    """(cost_n, cost_t) as float32 device tensors on `dev`, or (None, None, 0)."""
    if cost is None:
        return None, None, 0
    cn = torch.as_tensor(cost[0], dtype=torch.float32, device=dev).contiguous()
    ct = torch.as_tensor(cost[1], dtype=torch.float32, device=dev).contiguous()
    if cn.dim() != 1 or cn.shape != ct.shape or cn.numel() < 1:
        raise ValueError("cost must be (cost_n, cost_t): two 1-D sequences of one length >= 1")
    return cn, ct, cn.numel()


def alloc_budget_adaptive(alpha, cost, stream=None, workspace: Optional[Workspace] = None):
    """The budget with N chosen by utility / cost (spec_alloc_budget_adaptive).

    cost = (cost_n, cost_t): positions verified -> cost, cost_n strictly increasing.  Returns the
    chosen N (int32 [1]), depth [B] int32 and prefix confidences [B, K].
    """
    B, K = alpha.shape
    _need(alpha, "alpha", dtype=torch.float32, shape=(B, K))
    dev = alpha.device
    cn, ct, nc = _cost_table(cost, dev)
    if nc == 0:
        raise ValueError("alloc_budget_adaptive needs a cost table")
    n_out = torch.zeros(1, dtype=torch.int32, device=dev)
    depth = torch.empty(B, dtype=torch.int32, device=dev)
    conf = torch.empty(B, K, dtype=torch.float32, device=dev)
    ws = (workspace or default_workspace(stream))
    buf = ws.get(B, K, 1, SPEC_F32, stream)
    _check(lib().spec_alloc_budget_adaptive(_ptr(alpha), B, K, _ptr(cn), _ptr(ct), nc, _ptr(n_out), _ptr(depth),
                                            _ptr(conf), _ptr(buf), buf.numel(), _stream_ptr(stream)),
           "spec_alloc_budget_adaptive")
    return n_out, depth, conf


def draft_budget(draft, tokens, temperature: float, budget: Optional[int] = None, cost=None, stream=None,
                 workspace: Optional[Workspace] = None, out=None):
    """The budget from the draft alone, before the target runs (spec_draft_budget).

    draft [B, K, V] bf16/fp32, tokens [B, K] int32.  Either `budget` (N >= 0) or `cost`
    ((cost_n, cost_t), N chosen by utility / cost; float32 CUDA tensors are used as they are).
    Returns N (int32 [1]), depth [B] int32 and the prefix confidences prod q_k(x_k) [B, K], in
    `out` = (N, depth, conf) when given.
    """
    if draft.dim() != 3:
        raise ValueError("draft logits must be [B, K, V]")
    B, K, V = draft.shape
    dev = draft.device
    _need(draft, "draft", shape=(B, K, V))
    code = _dtype_code(draft)
    _need(tokens, "tokens", dtype=torch.int32, shape=(B, K), device=dev)
    cn, ct, nc = _cost_table(cost, dev)
    if nc == 0 and (budget is None or budget < 0):
        raise ValueError("draft_budget needs budget >= 0 or a cost table")
    if out is not None:
        n_out, depth, conf = out
        _need(n_out, "out N", dtype=torch.int32, shape=(1,), device=dev)
        _need(depth, "out depth", dtype=torch.int32, shape=(B,), device=dev)
        _need(conf, "out conf", dtype=torch.float32, shape=(B, K), device=dev)
    else:
        n_out = torch.zeros(1, dtype=torch.int32, device=dev)
        depth = torch.empty(B, dtype=torch.int32, device=dev)
        conf = torch.empty(B, K, dtype=torch.float32, device=dev)
    ws = (workspace or default_workspace(stream))
    buf = ws.get(B, K, V, code, stream)
    _check(lib().spec_draft_budget(_ptr(draft), code, _ptr(tokens), B, K, V, float(temperature),
                                   -1 if budget is None else int(budget), _ptr(cn), _ptr(ct), nc, _ptr(n_out),
                                   _ptr(depth), _ptr(conf), _ptr(buf), buf.numel(), _stream_ptr(stream)),
           "spec_draft_budget")
    return n_out, depth, conf


__all__ = ["verify_chain", "verify_block", "overlap_alpha", "alloc_budget", "alloc_budget_adaptive",
           "draft_budget", "Workspace", "VerifyOutput", "Tuning", "SpecError", "lib"]
