"""ctypes view of libspecverify.so (the C ABI declared in include/spec_verify.h).

Loading fails loudly if the library has not been built: there is no
fallback implementation on the product path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")

c_int, c_float, c_size_t, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p
c_longlong = ctypes.c_longlong


class SpecTuning(ctypes.Structure):
    """spec_tuning_t: per-call test and tuning knobs (all zero = defaults)."""
    _fields_ = [("wait_limit_us", c_longlong), ("cluster", c_int), ("greedy_variant", c_int),
                ("plan_out", c_void_p), ("split_event", c_void_p)]

# name -> (restype, argtypes), mirroring include/spec_verify.h
SIGNATURES = {
    "spec_version": (c_int, []),
    "spec_error_string": (ctypes.c_char_p, [c_int]),
    "spec_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int]),
    "spec_workspace_init": (c_int, [c_void_p, c_size_t, c_void_p]),
    "spec_get_status": (c_int, [c_void_p, c_void_p, c_void_p]),
    "spec_verify_chain": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                                  c_float, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                  c_void_p]),
    "spec_verify_block": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                                  c_float, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "spec_overlap_alpha": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_float, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "spec_alloc_budget": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_size_t,
                                  c_void_p]),
    "spec_alloc_budget_adaptive": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_int, c_void_p,
                                           c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "spec_draft_budget": (c_int, [c_void_p, c_int, c_void_p, c_int, c_int, c_int, c_float, c_int, c_void_p,
                                  c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "spec_verify_chain_greedy_static": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_int,
                                                c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "spec_verify_tuned": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                                  c_float, c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library once and attach the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
            "or python draft_verification_spec_gb300/build.py); there is no non-CUDA fallback")
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_symbols(header: str) -> list[str]:
    """Function names declared in a C header (for the export check)."""
    import re
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))
