"""ctypes binding of ``libwkv7.so`` (the C ABI in include/wkv7.h).

Loading never falls back to anything: if the library is missing or does not
load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libwkv7.so")

# wkv7_status codes
OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_ALIGNMENT = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_WORKSPACE = 6
ERR_DEVICE_BOUNDS = 7

F32 = 0
BF16 = 1
F16 = 2
TF32 = 3

EXPORTS = (
    "wkv7_step",
    "wkv7_step_cast",
    "wkv7_step_state",
    "wkv7_step_tail",
    "wkv7_tmix_tail",
    "wkv7_verify",
    "wkv7_verify_commit",
    "wkv7_prefill_workspace_size",
    "wkv7_prefill",
    "wkv7_prefill_cast",
    "wkv7_prefill_state",
    "wkv7_prefill_padded",
    "wkv7_prefill_noalloc",
    "wkv7_prefill_backward_workspace_size",
    "wkv7_prefill_backward",
    "wkv7_diag_bounded_wait",
    "wkv7_status_string",
    "wkv7_check_device_status",
    "wkv7_last_cuda_error",
    "wkv7_abi_version",
)

_lock = threading.Lock()
_lib = None


class WKV7Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.wkv7_step.restype = I
    lib.wkv7_step.argtypes = [I, I, I, P, P, P, P, P, P, P, P, P]
    lib.wkv7_step_cast.restype = I
    lib.wkv7_step_cast.argtypes = [I, I, I, P, P, P, P, P, P, P, P, I, P]
    lib.wkv7_step_state.restype = I
    lib.wkv7_step_state.argtypes = [I, I, I, P, P, P, P, P, P, P, I, P, I, P]
    lib.wkv7_prefill_padded.restype = I
    lib.wkv7_prefill_padded.argtypes = [I, I, I, I, P, P, I, P, P, P, P, P, P, P, P, P, I, P, S, P]
    lib.wkv7_prefill_cast.restype = I
    lib.wkv7_prefill_cast.argtypes = [I, I, I, I, P, P, I, P, P, P, P, P, P, P, P, P, I, P, S, P]
    lib.wkv7_prefill_state.restype = I
    lib.wkv7_prefill_state.argtypes = [I, I, I, I, P, P, I, P, P, P, P, P, P, P, P, I, P, I, P, S, P]
    F = ctypes.c_float
    lib.wkv7_step_tail.restype = I
    lib.wkv7_step_tail.argtypes = [I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, F, P, P]
    lib.wkv7_verify.restype = I
    lib.wkv7_verify.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, P]
    lib.wkv7_verify_commit.restype = I
    lib.wkv7_verify_commit.argtypes = [I, I, I, I, P, P, P, P]
    lib.wkv7_tmix_tail.restype = I
    lib.wkv7_tmix_tail.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, F, P, P]
    lib.wkv7_prefill_workspace_size.restype = S
    lib.wkv7_prefill_workspace_size.argtypes = [I, I, I, I]
    lib.wkv7_prefill.restype = I
    lib.wkv7_prefill.argtypes = [I, I, I, I, P, P, I, P, P, P, P, P, P, P, P, P, P, S, P]
    lib.wkv7_prefill_noalloc.restype = I
    lib.wkv7_prefill_noalloc.argtypes = [I, I, I, I, P, P, I, P, P, P, P, P, P, P, P, P, P]
    lib.wkv7_prefill_backward_workspace_size.restype = S
    lib.wkv7_prefill_backward_workspace_size.argtypes = [I, I, I, I]
    lib.wkv7_prefill_backward.restype = I
    lib.wkv7_prefill_backward.argtypes = [I, I, I, I, P, P, I] + [P] * 6 + [P] * 3 + [P] * 7 + [P, S, P]
    lib.wkv7_diag_bounded_wait.restype = I
    lib.wkv7_diag_bounded_wait.argtypes = [ctypes.c_uint, P]
    lib.wkv7_status_string.restype = ctypes.c_char_p
    lib.wkv7_status_string.argtypes = [I]
    lib.wkv7_check_device_status.restype = I
    lib.wkv7_check_device_status.argtypes = [P]
    lib.wkv7_last_cuda_error.restype = ctypes.c_char_p
    lib.wkv7_last_cuda_error.argtypes = []
    lib.wkv7_abi_version.restype = I
    lib.wkv7_abi_version.argtypes = []
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it is missing or does not load)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m rwkv_linear_attention_gb300.build` (there is no fallback path)")
            _lib = _bind(ctypes.CDLL(LIB_PATH))
        return _lib


def check(status: int, what: str) -> None:
    if status != OK:
        lib = load()
        msg = lib.wkv7_status_string(status).decode()
        if status == ERR_CUDA:
            msg += " (" + lib.wkv7_last_cuda_error().decode() + ")"
        raise WKV7Error(status, f"{what}: {msg}")
