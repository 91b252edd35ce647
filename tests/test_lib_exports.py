"""CPU checks of the C-ABI library: it builds, loads, and exports every symbol the header declares.

No compute call is made here (there is no GPU on this machine).
"""
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    from draft_verification_spec_gb300 import build as B
    B.build(quiet=True)
    from draft_verification_spec_gb300 import _lib
    return _lib.load()


def test_header_declares_the_four_entry_points():
    from draft_verification_spec_gb300._lib import header_symbols
    names = header_symbols(HEADER)
    for n in ("spec_verify_chain", "spec_verify_block", "spec_overlap_alpha", "spec_alloc_budget"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from draft_verification_spec_gb300._lib import SIGNATURES, header_symbols
    names = header_symbols(HEADER)
    for n in names:
        assert hasattr(lib, n), n
        assert n in SIGNATURES, f"{n} has no ctypes signature"


def test_host_only_calls(lib):
    assert lib.spec_version() >= 100
    assert lib.spec_error_string(0) == b"ok"
    assert lib.spec_error_string(5).startswith(b"draft token")
    ws = lib.spec_workspace_bytes(64, 3, 128000, 1)
    assert ws >= 64 * 4 * 32 and ws % 256 == 0
    assert lib.spec_workspace_bytes(-1, 3, 10, 0) == 0


def test_argument_errors_need_no_device(lib):
    # rejected before any CUDA call: bad dtype, negative sizes, bad temperature, oversize shapes
    assert lib.spec_verify_chain(None, None, 7, None, None, 1, 1, 10, 1.0, None, None, None, None, None, 0,
                                 None) == 1
    assert lib.spec_verify_chain(None, None, 0, None, None, -1, 1, 10, 1.0, None, None, None, None, None, 0,
                                 None) == 1
    assert lib.spec_verify_chain(None, None, 0, None, None, 1, 1, 10, -0.5, None, None, None, None, None, 0,
                                 None) == 1
    assert lib.spec_verify_chain(None, None, 0, None, None, 1, 33, 10, 1.0, None, None, None, None, None, 0,
                                 None) == 2
    assert lib.spec_verify_chain(None, None, 0, None, None, 1, 3, 300000, 1.0, None, None, None, None, None,
                                 0, None) == 2
    assert lib.spec_verify_chain(None, None, 0, None, None, 0, 3, 100, 1.0, None, None, None, None, None,
                                 0, None) == 0      # B == 0 is a no-op
    assert lib.spec_alloc_budget(None, 200, 64, 5, None, None, None, 0, None) == 2
    assert lib.spec_alloc_budget(None, 2, 2, -1, None, None, None, 0, None) == 1


def test_product_path_has_no_oracle_import():
    pkg = os.path.join(ROOT, "draft_verification_spec_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("the oracle", ""), f
