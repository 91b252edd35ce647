"""The workspace-free greedy entry point, for callers that cannot give the library device memory.

Engines that pre-reserve all device memory in their own pool, or hosts that forbid cudaMalloc /
cudaFree after start-up (those calls can synchronise the whole device), call
spec_verify_chain_greedy_static instead of spec_verify_chain.  It must give the same tokens,
accepted counts and one-hot alpha as the workspace entry point, call after call, although every
call reuses the same fixed device scratch.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests.parity_utils import oracle_verify

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_static_entry_matches_workspace_entry_twice():
    import draft_verification_spec_gb300 as sv
    lib = sv.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cases = [W.greedy_mtp(seed=11, B=16), W.random_case(seed=5, B=3, K=4, V=1023, T=0.0, dtype=torch.bfloat16)]
    for w in cases:
        t, d, x = w.target.to(dev), w.draft.to(dev), w.tokens.to(dev)
        ref = sv.verify_chain(t, d, x, None, 0.0, want_alpha=True)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        for _ in range(2):
            tok = torch.full((w.B, w.K + 1), -7, dtype=torch.int32, device=dev)
            acc = torch.full((w.B,), -7, dtype=torch.int32, device=dev)
            alpha = torch.full((w.B, w.K), -1.0, dtype=torch.float32, device=dev)
            status = torch.full((1,), -1, dtype=torch.int32, device=dev)
            code = lib.spec_verify_chain_greedy_static(
                _p(t), _p(d), 1 if t.dtype == torch.bfloat16 else 0, _p(x), w.B, w.K, w.V, None,
                _p(tok), _p(acc), _p(alpha), _p(status), ctypes.c_void_p(stream.cuda_stream))
            assert code == 0
            torch.cuda.synchronize()
            assert torch.equal(tok, ref.tokens)
            assert torch.equal(acc, ref.accepted)
            np.testing.assert_array_equal(alpha.cpu().numpy(), ref.alpha.cpu().numpy())
            assert int(status.item()) == 0


def _static_call(lib, w, dev, depth=None, want_alpha=True, tokens=None):
    t, d = w.target.to(dev), w.draft.to(dev)
    x = (w.tokens if tokens is None else tokens).to(dev)
    tok = torch.full((w.B, w.K + 1), -7, dtype=torch.int32, device=dev)
    acc = torch.full((w.B,), -7, dtype=torch.int32, device=dev)
    alpha = torch.full((w.B, w.K), -1.0, dtype=torch.float32, device=dev) if want_alpha else None
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    dep = None if depth is None else torch.as_tensor(depth, dtype=torch.int32, device=dev)
    code = lib.spec_verify_chain_greedy_static(
        _p(t), _p(d) if want_alpha else None, 1 if t.dtype == torch.bfloat16 else 0, _p(x), w.B, w.K, w.V,
        _p(dep), _p(tok), _p(acc), _p(alpha), _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return code, tok, acc, alpha, int(status.item())


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 20000), (torch.float32, 12300)])
def test_static_entry_matches_oracle_with_depth(dtype, V):
    """Tokens, accepted counts and one-hot alpha against the float64 oracle, with a depth vector."""
    import draft_verification_spec_gb300 as sv
    lib = sv.lib()
    dev = torch.device("cuda", 0)
    w = W.random_case(seed=41, B=6, K=4, V=V, T=0.0, dtype=dtype)
    depth = np.array([0, 1, 4, 2, 3, 4], dtype=np.int32)
    ref = oracle_verify(w, depth=depth)
    code, tok, acc, alpha, status = _static_call(lib, w, dev, depth=depth)
    assert code == 0 and status == 0
    np.testing.assert_array_equal(tok.cpu().numpy(), ref.tokens)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref.accepted)
    np.testing.assert_array_equal(alpha.cpu().numpy(), ref.alpha)
    assert np.all(acc.cpu().numpy() <= depth)


def test_static_entry_token_out_of_range_sets_status_bit():
    import draft_verification_spec_gb300 as sv
    lib = sv.lib()
    dev = torch.device("cuda", 0)
    w = W.random_case(seed=43, B=3, K=3, V=5000, T=0.0, dtype=torch.bfloat16)
    x = w.tokens.clone()
    x[1, 0] = w.V + 9                                   # request 1 drafts an id outside [0, V)
    code, tok, acc, _, status = _static_call(lib, w, dev, want_alpha=False, tokens=x)
    assert code == 0
    assert status & 2                                   # the token-range bit of the raw status word
    assert int(acc[1].item()) == 0                      # the bad draft is rejected at position 0
    code, _, _, _, status = _static_call(lib, w, dev, want_alpha=False)
    assert code == 0 and status == 0                    # the next call starts from a clear word


def test_static_entry_rejects_oversize_batch():
    import draft_verification_spec_gb300 as sv
    lib = sv.lib()
    # 2000 requests x 3 rows exceed the 4096-row scratch: refused before any launch
    assert lib.spec_verify_chain_greedy_static(None, None, 1, None, 2000, 2, 128000, None, None, None, None,
                                               None, None) == 2
