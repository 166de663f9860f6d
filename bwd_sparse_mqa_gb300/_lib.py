"""ctypes view of libsparse_mqa.so (the C ABI in include/sparse_mqa.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library.  Loading fails loudly if the library is missing;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

SMQA_OK = 0
SMQA_ERR_INVALID_ARG = 1
SMQA_ERR_UNSUPPORTED = 2
SMQA_ERR_CUDA = 3
SMQA_ERR_DEVICE_TIMEOUT = 4
FLAG_RETURN_DKV_FP32 = 1
FLAG_REFERENCE_ROUNDING = 2
FLAG_DETERMINISTIC_DKV = 4

# Every symbol include/sparse_mqa.h declares (checked by the tests).
EXPORTS = [
    "smqa_fwd", "smqa_bwd_workspace_bytes", "smqa_bwd", "smqa_bwd_preprocess", "smqa_bwd_main",
    "smqa_bwd_postprocess", "smqa_device_status", "smqa_status_string", "smqa_last_error",
    "smqa_abi_version", "smqa_bwd_static_scratch", "smqa_bwd_exchange_bytes",
    "smqa_fwd_workspace_bytes", "smqa_fwd_static_scratch", "smqa_bwd_sink_grad",
    "smqa_fwd_host_workspace_bytes", "smqa_fwd_bwd_host_workspace_bytes", "smqa_fwd_host",
    "smqa_fwd_bwd_host", "smqa_host_chunk_plan", "smqa_set_wait_limit_ns", "smqa_debug_stall",
    "smqa_indexer_bwd", "smqa_batched_indexer_bwd",
]
STATIC_SCRATCH_BYTES = 64 << 20


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("S", ctypes.c_int32), ("S_kv", ctypes.c_int32),
                ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("topk", ctypes.c_int32)]


class SMQAError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        self.status = status
        super().__init__(f"{fn} failed: {status_name(status)} ({detail})")


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P, S, F, U = ctypes.c_void_p, Shape, ctypes.c_float, ctypes.c_uint
    st = ctypes.c_int
    lib.smqa_fwd.argtypes = [P, P, P, P, S, F, P, P, P, ctypes.c_size_t, U, P]
    lib.smqa_fwd.restype = st
    lib.smqa_fwd_workspace_bytes.argtypes = [S]
    lib.smqa_fwd_workspace_bytes.restype = ctypes.c_size_t
    lib.smqa_fwd_static_scratch.argtypes = [P, P, P, P, S, F, P, P, U, P]
    lib.smqa_fwd_static_scratch.restype = st
    lib.smqa_bwd_workspace_bytes.argtypes = [S, U]
    lib.smqa_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.smqa_bwd.argtypes = [P, P, P, P, P, P, P, S, F, P, P, P, P, ctypes.c_size_t, U, P]
    lib.smqa_bwd.restype = st
    lib.smqa_bwd_preprocess.argtypes = [P, P, S, P, P, P]
    lib.smqa_bwd_preprocess.restype = st
    lib.smqa_bwd_main.argtypes = [P, P, P, P, P, P, P, S, F, P, P, P, ctypes.c_size_t, P]
    lib.smqa_bwd_exchange_bytes.argtypes = [S]
    lib.smqa_bwd_exchange_bytes.restype = ctypes.c_size_t
    lib.smqa_bwd_main.restype = st
    lib.smqa_bwd_postprocess.argtypes = [P, S, P, P]
    lib.smqa_bwd_postprocess.restype = st
    lib.smqa_bwd_static_scratch.argtypes = [P, P, P, P, P, P, P, S, F, P, P, P, U, P]
    lib.smqa_bwd_sink_grad.argtypes = [P, P, P, S, P, P]
    lib.smqa_bwd_sink_grad.restype = st
    lib.smqa_bwd_static_scratch.restype = st
    lib.smqa_fwd_host_workspace_bytes.argtypes = [S]
    lib.smqa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.smqa_fwd_bwd_host_workspace_bytes.argtypes = [S, U]
    lib.smqa_fwd_bwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.smqa_host_chunk_plan.argtypes = [S, P, ctypes.c_int]
    lib.smqa_host_chunk_plan.restype = ctypes.c_int
    lib.smqa_fwd_host.argtypes = [P, P, P, P, S, F, P, P, P, ctypes.c_size_t, U, P]
    lib.smqa_fwd_host.restype = st
    lib.smqa_fwd_bwd_host.argtypes = [P, P, P, P, P, S, F, P, P, P, P, P, P, ctypes.c_size_t, U,
                                      P]
    lib.smqa_fwd_bwd_host.restype = st
    lib.smqa_indexer_bwd.argtypes = [P, P, P, P, P, S, P, P]
    lib.smqa_indexer_bwd.restype = st
    lib.smqa_batched_indexer_bwd.argtypes = [P, P, P, P, P, S, P, P]
    lib.smqa_batched_indexer_bwd.restype = st
    lib.smqa_debug_stall.argtypes = [ctypes.c_int]
    lib.smqa_debug_stall.restype = None
    lib.smqa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.smqa_set_wait_limit_ns.restype = ctypes.c_uint64
    lib.smqa_device_status.argtypes = [ctypes.c_int]
    lib.smqa_device_status.restype = st
    lib.smqa_status_string.argtypes = [st]
    lib.smqa_status_string.restype = ctypes.c_char_p
    lib.smqa_last_error.argtypes = []
    lib.smqa_last_error.restype = ctypes.c_char_p
    lib.smqa_abi_version.argtypes = []
    lib.smqa_abi_version.restype = ctypes.c_int
    return lib


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """The loaded library; builds it first when the toolkit is present."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if build_if_missing:
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libsparse_mqa.so not found at {path}; run "
                                   "`python -m bwd_sparse_mqa_gb300.build` (needs nvcc)")
            _lib = _bind(ctypes.CDLL(path))
    return _lib


def status_name(status: int) -> str:
    names = {0: "SMQA_OK", 1: "SMQA_ERR_INVALID_ARG", 2: "SMQA_ERR_UNSUPPORTED",
             3: "SMQA_ERR_CUDA", 4: "SMQA_ERR_DEVICE_TIMEOUT"}
    return names.get(status, f"status {status}")


def check(fn: str, status: int) -> None:
    if status != SMQA_OK:
        detail = load().smqa_last_error().decode(errors="replace")
        raise SMQAError(fn, status, detail)
