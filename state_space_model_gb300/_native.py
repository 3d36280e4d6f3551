"""Loads ``libssd_gb300.so`` and declares its C ABI (include/ssd.h) for ctypes.

There is no fallback: if the library has not been built, loading fails with
an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
# SSD_DEBUG_BOUNDS=1 selects the debug build (device-side bounds checks,
# `python -m state_space_model_gb300.build --debug-bounds`); read at import.
LIB_PATH = os.path.join(_PKG, "libssd_gb300_debug.so" if os.environ.get("SSD_DEBUG_BOUNDS") == "1"
                        else "libssd_gb300.so")

SSD_F32, SSD_BF16, SSD_I32 = 0, 1, 2
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED",
          3: "SSD_ERR_ALIGNMENT", 4: "SSD_ERR_WORKSPACE", 5: "SSD_ERR_CUDA",
          6: "SSD_ERR_TIMEOUT", 7: "SSD_ERR_DEVICE_BOUNDS"}


class SsdTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * 5),
                ("stride", ctypes.c_int64 * 5)]


class SsdError(RuntimeError):
    def __init__(self, status: int, detail: str, call: str):
        self.status = status
        self.status_name = STATUS.get(status, f"status {status}")
        self.detail = detail
        super().__init__(f"{call}: {self.status_name}: {detail}")


_lib = None
_lock = threading.Lock()

_T = ctypes.POINTER(SsdTensor)
_VP, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t

# name -> argtypes; every entry point returns an ssd_status (int)
SIGNATURES = {
    "ssd_workspace_size": [_I64, _I64, _I64, _I64, _I64, _I64, _I64, _I32,
                           ctypes.POINTER(ctypes.c_size_t)],
    "ssd_chunked_fwd": [_T, _T, _T, _T, _T, _T, _T, _I64, _I64, _T, _T, _VP, _SZ, _VP],
    "ssd_chunked_fwd_gated": [_T, _T, _T, _T, _T, _T, _T, _T, _I64, _I64, _T, _T, _VP, _SZ, _VP],
    "ssd_chunked_fwd_static_scratch": [_T, _T, _T, _T, _T, _T, _T, _I64, _I64, _T, _T, _VP],
    "ssd_device_status": [_VP],
    "ssd_selftest_wait_timeout": [ctypes.c_uint64, _VP],
    "ssd_selftest_bounds_check": [_VP],
    "ssd_segment_logdecay": [_T, _T, _T, _VP],
    "ssd_sequence_combine": [_T, _T, _T, _I32, _T, _VP],
    "ssd_shard_correct": [_T, _T, _T, _T, _T, _I64, _T, _T, _VP],
    "ssd_state_update": [_T, _T, _T, _T, _T, _T, _T, _T, _T, _I32, _I64, _T, _VP],
    "ssd_state_update_tokens": [_T, _T, _T, _T, _T, _T, _T, _T, _T, _I32, _I64, _T, _T, _T, _T,
                                _I32, _VP],
    "ssd_mixer_prologue": [_T, _T, _T, _T, _T, _T, _T, _T, _I32, _I64, _T, _T, _T, _T, _VP],
    "ssd_stage_chunk_cumsum": [_T, _T, _I64, _T, _VP],
    "ssd_stage_chunk_state": [_T, _T, _T, _T, _I64, _I64, _T, _VP],
    "ssd_stage_state_passing": [_T, _T, _T, _I64, _T, _T, _VP],
    "ssd_stage_chunk_scan": [_T, _T, _T, _T, _T, _T, _T, _I64, _I64, _T, _VP],
}


def load():
    """Returns the loaded library, raising if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -m state_space_model_gb300.build` "
                    "(or __graft_entry__.build()) first")
            lib = ctypes.CDLL(LIB_PATH)
            for name, args in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.ssd_status_string.argtypes = [ctypes.c_int]
            lib.ssd_status_string.restype = ctypes.c_char_p
            lib.ssd_last_error_detail.argtypes = []
            lib.ssd_last_error_detail.restype = ctypes.c_char_p
            lib.ssd_describe_plan.argtypes = [_I64] * 7 + [_I32]
            lib.ssd_describe_plan.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def check(status: int, call: str) -> None:
    if status != 0:
        detail = load().ssd_last_error_detail().decode(errors="replace")
        raise SsdError(status, detail, call)
