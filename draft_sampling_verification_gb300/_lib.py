"""ctypes loader of libdspark.so and the C signatures of include/dspark.h.

The product path has no fallback: if the shared library is missing or fails
to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdspark.so")
INCLUDE = os.path.join(os.path.dirname(_HERE), "include")
HEADERS = [os.path.join(INCLUDE, "dspark.h"), os.path.join(INCLUDE, "dspark_debug.h")]

_P = ctypes.c_void_p
_I32, _I64, _U64, _U32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32

SIGNATURES = {
    "dspark_q_build": [_P, _I32, _I64, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P],
    "dspark_draft_sample": [_P, _P, _P, _I32, _I32, _I32, _I32, _U64, _P, _P, _P, _P],
    "dspark_q_build_sample": [_P, _I32, _I64, _I32, _I32, _I32, _P, _I32, _U64, _P, _P, _P, _P,
                              _P, _P, _P],
    "dspark_verify_greedy": [_P, _I32, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _P],
    "dspark_verify_ratio": [_P, _I32, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _I32, _U64, _P,
                            _P, _P, _P, _P, _P],
    "dspark_target_probs": [_P, _I32, _I64, _I32, _I32, _P, _P, _P, _P],
    "dspark_verify_stats": [_P, _I32, _P, _P],
    "dspark_verify": [_P, _I32, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _I32, _U64, _P, _P, _P,
                      _P, _P, _P, _P, _P, _P],
    "dspark_spec_step_schedule": [_I32, _I32],
    "dspark_q_pack": [_P, _P, _P, _I32, _I32, _I32, _P, _P, _P],
    "dspark_q_build_sample_sharded": [_P, _I32, _I64, _I32, _I32, _I32, _I32, _P, _I32, _U64,
                                      _P, _P, _P, _P, _P, _P, _P, _P],
    "dspark_q_chain_sample": [_P, _I32, _I64, _I32, _I32, _I32, _P, _P, _I64, _I32, _P, _U64, _P,
                              _P, _P, _P, _P, _P, _P],
    "dspark_verify_match": [_P, _I32, _I64, _I32, _I32, _I32, _P, _U64, _P, _P, _P, _P, _P, _P],
    "dspark_q_validate": [_P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P],
    "dspark_spec_step_noalloc": [_P, _I32, _I64, _P, _I32, _I64, _I32, _I32, _I32, _P, _U64, _P,
                                 _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _P],
    "dspark_spec_step": [_P, _I32, _I64, _P, _I32, _I64, _I32, _I32, _I32, _P, _U64, _P, _P, _P,
                         _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _P],
    "dspark_spec_step_host": [_P, _I32, _P, _I32, _I32, _I32, _I32, _P, _U64, _P, _P, _P, _P, _P,
                              _P, _P, _P, _P, _P, _P, _I32, _P],
    "dspark_debug_exp_weights": [_P, _I64, _P, _P, _P],
    "dspark_debug_philox": [_P, _U64, _I64, _P, _P],
    "dspark_debug_alloc_scale": [_P, _I64, _P, _P, _P, _P, _P],
    "dspark_debug_wait": [_I32, _P, _U32, _P, _P],
    "dspark_checked_status": [_P],
    "dspark_debug_check_selftest": [_P],
}

_lock = threading.Lock()
_lib = None


def header_symbols(paths=None):
    """Function names declared in the public headers."""
    names = set()
    for path in paths or HEADERS:
        text = open(path).read()
        names.update(re.findall(r"^\s*(?:int|int64_t|const char\*)\s+(dspark_\w+)\s*\(", text, re.M))
    return sorted(names)


def load(path: str = LIB_PATH):
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    "libdspark.so is not built (%s); run draft_sampling_verification_gb300.build"
                    % path)
            lib = ctypes.CDLL(path)
            for name, args in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.dspark_q_sharded_workspace_bytes.argtypes = [_I32]
            lib.dspark_q_sharded_workspace_bytes.restype = ctypes.c_int64
            lib.dspark_spec_step_host_staging_bytes.argtypes = [_I32, _I32, _I32, _I32, _I32]
            lib.dspark_spec_step_host_staging_bytes.restype = ctypes.c_int64
            lib.dspark_version.argtypes = []
            lib.dspark_version.restype = ctypes.c_char_p
            _lib = lib
    return _lib
