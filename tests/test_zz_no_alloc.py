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


def test_static_entry_rejects_oversize_batch():
    import draft_verification_spec_gb300 as sv
    lib = sv.lib()
    # 2000 requests x 3 rows exceed the 4096-row scratch: refused before any launch
    assert lib.spec_verify_chain_greedy_static(None, None, 1, None, 2000, 2, 128000, None, None, None, None,
                                               None, None) == 2
