"""ctypes view of the C ABI in include/spec_verify.h (libspecverify.so).

Loading fails loudly when the shared library has not been built: there is no
other implementation behind these calls."""
from __future__ import annotations

import ctypes
import os
import re

from .build import INCLUDE, LIB, LIB_BOUNDS

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_DTYPE = 2
SPEC_ERR_WORKSPACE = 3
SPEC_ERR_CUDA = 6
SPEC_ERR_TOO_LARGE = 7
SPEC_STATIC_SCRATCH_BYTES = 1 << 20

SPEC_DEV_TOKEN_RANGE = 1
SPEC_DEV_NONFINITE = 2
SPEC_DEV_OFFSETS = 4
SPEC_DEV_TIMEOUT = 8
SPEC_DEV_POSITION = 16
SPEC_DEV_BOUNDS = 32  # only set by the bounds-checked build

SPEC_F32 = 0
SPEC_BF16 = 1

SPEC_MODE_STOCHASTIC = 0
SPEC_MODE_GREEDY = 1
SPEC_MODE_NKL = 2

SPEC_MAX_GAMMA = 128
SPEC_MAX_TREE_NODES = 64
SPEC_STATS_SLOTS = 64
SPEC_MAX_CANDIDATES = 4


class SpecBatch(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("gamma", ctypes.c_int32), ("V", ctypes.c_int32),
                ("total_draft", ctypes.c_int32), ("cu_draft", ctypes.c_void_p)]


class SpecMultiBatch(ctypes.Structure):
    _fields_ = [("G", ctypes.c_int32), ("K", ctypes.c_int32), ("gamma", ctypes.c_int32), ("V", ctypes.c_int32)]


class SpecStatsSlot(ctypes.Structure):
    _fields_ = [("bucket", ctypes.c_int64), ("rounds", ctypes.c_uint64), ("accepted", ctypes.c_uint64),
                ("drafted", ctypes.c_uint64), ("rate_fx", ctypes.c_uint64), ("rate2_fx", ctypes.c_uint64)]


STATS_BYTES = ctypes.sizeof(SpecStatsSlot) * SPEC_STATS_SLOTS   # sizeof(spec_accept_stats)


class SpecOptions(ctypes.Structure):
    _fields_ = [("temperature_draft", ctypes.c_float), ("position", ctypes.c_void_p),
                ("delta_alpha", ctypes.c_float), ("delta_max", ctypes.c_float),
                ("min_block_len", ctypes.c_int32), ("block_n", ctypes.c_void_p),
                ("block_tokens", ctypes.c_void_p), ("stats", ctypes.c_void_p), ("stats_bucket", ctypes.c_int64)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_F = ctypes.c_float
_S = ctypes.c_size_t

SIGNATURES = {
    "spec_workspace_bytes": (_S, [SpecBatch, ctypes.c_int, ctypes.c_int]),
    "spec_tree_workspace_bytes": (_S, [_I, _I, _I]),
    "spec_tree_depth": (_I, [_P, _I]),
    "spec_verify_stochastic": (ctypes.c_int, [SpecBatch, ctypes.c_int, _P, _P, _P, _F, _P, _P, _P, _P, _P, _P, _P,
                                              _P, _P, _F, _P, _P, _P, _P, _S, _P]),
    "spec_verify_stochastic_static": (ctypes.c_int, [SpecBatch, ctypes.c_int, _P, _P, _P, _F, _P, _P, _P, _P, _P,
                                                     _P, _P, _P, _P, _F, _P, _P, _P, _P]),
    "spec_verify_greedy": (ctypes.c_int, [SpecBatch, ctypes.c_int, _P, _P, _P, _P, _P, _P, _S, _P]),
    "spec_verify_tree": (ctypes.c_int, [_I, _I, _I, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "spec_nkl": (ctypes.c_int, [SpecBatch, ctypes.c_int, _P, _P, _F, _F, _P, _P, _P, _P, _S, _P]),
    "spec_verify_stochastic_ex": (ctypes.c_int, [SpecBatch, ctypes.c_int, _P, _P, _P, _F, _P, _P, _P, _P, _P, _P,
                                                 _P, _P, _P, _F, _P, _P, ctypes.POINTER(SpecOptions), _P, _P, _S,
                                                 _P]),
    "spec_verify_greedy_ex": (ctypes.c_int, [SpecBatch, ctypes.c_int, _P, _P, _P, _P, ctypes.POINTER(SpecOptions),
                                             _P, _P, _S, _P]),
    "spec_nkl_ex": (ctypes.c_int, [SpecBatch, ctypes.c_int, _P, _P, _F, _F, _P, _P, ctypes.POINTER(SpecOptions),
                                   _P, _P, _S, _P]),
    "spec_accept_summary": (ctypes.c_int, [_P, ctypes.c_int64, _I, _P, _P]),
    "spec_multi_workspace_bytes": (_S, [SpecMultiBatch, ctypes.c_int, _I]),
    "spec_verify_multi": (ctypes.c_int, [SpecMultiBatch, ctypes.c_int, _I, _P, _P, _P, _F, _P, _P, _F, _F, _P, _P,
                                         _P, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "spec_selftest_wait_timeout": (ctypes.c_int, [_P, _P, _S, _P]),
    "spec_status_str": (ctypes.c_char_p, [ctypes.c_int]),
}

_LIB = None


def declared_functions() -> list:
    """Names of the functions include/spec_verify.h declares."""
    with open(os.path.join(INCLUDE, "spec_verify.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def load(path: str) -> ctypes.CDLL:
    """The library at `path` with every declared function's signature set."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load(LIB)
    return _LIB


def bounds_lib() -> ctypes.CDLL:
    """The bounds-checked debug variant (SPEC_BOUNDS_CHECK=1), for tests: every computed
    access is checked against its buffer and one outside it sets SPEC_DEV_BOUNDS."""
    return load(LIB_BOUNDS)


def status_str(code: int) -> str:
    return lib().spec_status_str(code).decode()


class SpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({status_str(code)})")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != SPEC_OK:
        raise SpecError(fn, code)
