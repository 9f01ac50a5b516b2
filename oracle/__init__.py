"""fp64 CPU oracle for the WKV-7 recurrence.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only users.  The product
library never imports this package, and this package never imports the
product library: the two share nothing but the seeded input generator.

The arithmetic lives in ``wkv7_oracle.c`` (plain C, double precision, one
token at a time; the formula is the per-head WKV7 update of the Core AI model
zoo note "Recurrent / linear-attention LLMs on Core AI", section 1).  This
module only compiles it with gcc, loads it with ctypes and marshals numpy
arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "wkv7_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libwkv7_oracle.so")

_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile one oracle source file into a shared object with gcc."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build(force: bool = False) -> str:
    """Build ``libwkv7_oracle.so`` next to the source if it is missing or stale."""
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE):
        tmp = LIB_PATH + f".{os.getpid()}.tmp"
        compile_source(SOURCE, tmp)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    f = lib.wkv7_oracle_run
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    f.argtypes = [ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                  P, P, P, P, P, P, P, P, P, ctypes.c_int]
    t = lib.wkv7_oracle_tail
    t.restype = ctypes.c_int
    t.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P, P, ctypes.c_double, P]
    b = lib.wkv7_oracle_backward
    b.restype = ctypes.c_int
    b.argtypes = [ctypes.c_int, P, ctypes.c_int, ctypes.c_int] + [P] * 6 + [P] * 3 + [P] * 7 + [ctypes.c_int]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first when ``path`` is None)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _as_f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: widen exactly to fp32 on the host
        x = x.detach().float().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(x: np.ndarray | None):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def run(r, w, k, v, kk, a, cu_seqlens=None, s0=None, nthreads: int | None = None, lib=None):
    """Run the recurrence on packed sequences.

    r, w, k, v, kk, a: [T_total, H, N] arrays holding the exact stored values
    (bf16 tensors are widened to fp32, which is exact).  ``cu_seqlens`` is
    [num_seqs + 1] (default: one sequence of T_total tokens).  ``s0`` is the
    initial state [num_seqs, H, N, N] (None = zeros); it is taken in double so
    that a carried oracle state is not rounded.

    Returns ``(o, s_final)``: o [T_total, H, N] and s_final [num_seqs, H, N, N],
    both float64.
    """
    lib = lib or load()
    arrs = [_as_f32(x) for x in (r, w, k, v, kk, a)]
    T_total, H, N = arrs[0].shape
    for x in arrs:
        if x.shape != (T_total, H, N):
            raise ValueError(f"input shape {x.shape} != {(T_total, H, N)}")
    if cu_seqlens is None:
        cu = np.array([0, T_total], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    num_seqs = cu.shape[0] - 1
    if num_seqs < 0 or cu[-1] != T_total:
        raise ValueError("cu_seqlens must end at T_total")
    s0d = None
    if s0 is not None:
        if hasattr(s0, "detach"):
            s0 = s0.detach().cpu().double().numpy()
        s0d = np.ascontiguousarray(s0, dtype=np.float64).reshape(num_seqs, H, N, N)
    o = np.zeros((T_total, H, N), dtype=np.float64)
    s_final = np.zeros((num_seqs, H, N, N), dtype=np.float64)
    rc = lib.wkv7_oracle_run(num_seqs, _ptr(cu), H, N, *[_ptr(x) for x in arrs],
                             _ptr(s0d), _ptr(o), _ptr(s_final),
                             int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"wkv7_oracle_run failed with code {rc}")
    return o, s_final


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def backward(r, w, k, v, kk, a, d_o, cu_seqlens=None, s0=None, d_sfinal=None,
             nthreads: int | None = None, lib=None):
    """Reverse-mode derivative of ``run`` for L = <d_o, o> + <d_sfinal, s_final>.

    Inputs as for ``run``; ``d_o`` [T_total, H, N] and ``d_sfinal``
    [num_seqs, H, N, N] (None = zeros) are taken in double.  Returns
    ``(dr, dw, dk, dv, dkk, da, d_s0)``, all float64: the first six
    [T_total, H, N], d_s0 [num_seqs, H, N, N].
    """
    lib = lib or load()
    arrs = [_as_f32(x) for x in (r, w, k, v, kk, a)]
    T_total, H, N = arrs[0].shape
    for x in arrs:
        if x.shape != (T_total, H, N):
            raise ValueError(f"input shape {x.shape} != {(T_total, H, N)}")
    if cu_seqlens is None:
        cu = np.array([0, T_total], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    num_seqs = cu.shape[0] - 1
    if num_seqs < 0 or cu[-1] != T_total:
        raise ValueError("cu_seqlens must end at T_total")
    dod = _as_f64(d_o).reshape(T_total, H, N)
    s0d = None if s0 is None else _as_f64(s0).reshape(num_seqs, H, N, N)
    dsf = None if d_sfinal is None else _as_f64(d_sfinal).reshape(num_seqs, H, N, N)
    outs = [np.zeros((T_total, H, N), dtype=np.float64) for _ in range(6)]
    d_s0 = np.zeros((num_seqs, H, N, N), dtype=np.float64)
    rc = lib.wkv7_oracle_backward(num_seqs, _ptr(cu), H, N, *[_ptr(x) for x in arrs],
                                  _ptr(s0d), _ptr(dod), _ptr(dsf), *[_ptr(x) for x in outs], _ptr(d_s0),
                                  int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"wkv7_oracle_backward failed with code {rc}")
    return (*outs, d_s0)


def step(r, w, k, v, kk, a, state, nthreads: int | None = None, lib=None):
    """One decode token for B x H heads: inputs [B, H, N], state [B, H, N, N].

    Each (b, h) is a one-token sequence of the packed form; returns
    ``(o [B, H, N], new_state [B, H, N, N])`` in float64.
    """
    arrs = [_as_f32(x) for x in (r, w, k, v, kk, a)]
    B = arrs[0].shape[0]
    cu = np.arange(B + 1, dtype=np.int64)
    return run(*arrs, cu_seqlens=cu, s0=state, nthreads=nthreads, lib=lib)


def tail(o, r, k, v, rk, ln_w, ln_b, g, eps, lib=None):
    """The time-mix tail after WKV (group norm per head, bonus, gate), in double.

    o: WKV outputs [rows, H, N] (taken in double); r, k, v, g: [rows, H, N];
    rk, ln_w, ln_b: [H, N]; eps: the norm's epsilon.  Returns y [rows, H, N]
    float64.
    """
    lib = lib or load()
    if hasattr(o, "detach"):
        o = o.detach().cpu().double().numpy()
    od = np.ascontiguousarray(o, dtype=np.float64)
    rows, H, N = od.shape
    xs = [_as_f32(x) for x in (r, k, v)]
    params = [_as_f32(x) for x in (rk, ln_w, ln_b)]
    gg = _as_f32(g)
    for x in xs + [gg]:
        if x.shape != (rows, H, N):
            raise ValueError(f"row input shape {x.shape} != {(rows, H, N)}")
    for x in params:
        if x.shape != (H, N):
            raise ValueError(f"parameter shape {x.shape} != {(H, N)}")
    y = np.zeros((rows, H, N), dtype=np.float64)
    rc = lib.wkv7_oracle_tail(rows, H, N, _ptr(od), *[_ptr(x) for x in xs], *[_ptr(x) for x in params],
                              _ptr(gg), float(eps), _ptr(y))
    if rc != 0:
        raise ValueError(f"wkv7_oracle_tail failed with code {rc}")
    return y
