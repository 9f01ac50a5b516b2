"""WKV-7 recurrence on one NVIDIA GB300: Python binding of the C ABI.

Two calls, both thin argument marshalling over ``libwkv7.so`` -- every step
of the computation runs in the library's CUDA kernels:

* :func:`step` -- one decode token for B x H heads, the fp32 state updated in
  place;
* :func:`prefill` -- packed variable-length sequences (``cu_seqlens``), with
  optional initial states and final states out.

Per head, with state S = [K, V] (Core AI model zoo note "Recurrent /
linear-attention LLMs on Core AI", section 1):
``S = diag(exp w) S - (kk*a)(kk^T S) + k v^T ; o = S^T r``.

Tensors must be CUDA, contiguous, 16-byte aligned; the current torch stream
is used.  There is no CPU path: without the CUDA library every call raises.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import WKV7Error  # noqa: F401

__all__ = ["step", "step_tail", "tmix_tail", "verify", "verify_commit", "prefill", "prefill_padded", "prefill_workspace_size",
           "prefill_backward", "prefill_backward_workspace_size", "check_device_status", "diag_bounded_wait",
           "WKV7Error", "HEAD_SIZE"]

HEAD_SIZE = 64


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _stream_handle(stream, device):
    """The cudaStream_t of ``stream`` (or of the current stream of ``device``) as an int."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(device.index if device.index is not None else torch.cuda.current_device())
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(name, t, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _out_code(dtype):
    if dtype == torch.float32:
        return _lib.F32
    if dtype == torch.bfloat16:
        return _lib.BF16
    raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")


_STATE_CODES = {torch.float32: _lib.F32, torch.float16: _lib.F16, torch.bfloat16: _lib.BF16}


def _x_code(xdt, tf32):
    """The prefill input code: bf16; fp32 contracted at tf32 by the chunked kernel
    (``tf32``); or fp32 through the exact token-serial kernel."""
    if xdt == torch.bfloat16:
        return _lib.BF16
    return _lib.TF32 if tf32 else _lib.F32
_STEP_IN = ("r", "w", "k", "v", "kk", "a")


def step(r, w, k, v, kk, a, state, o=None, stream=None, out_dtype=torch.float32):
    """One decode token: inputs fp32 [B, H, N]; ``state`` [B, H, N, N] updated
    in place, fp32 or a 16-bit type (fp16 / bf16: widened to fp32 for the
    update, rounded to nearest even on store).  Returns ``o`` [B, H, N] in
    ``out_dtype`` (fp32, or bf16 rounded to nearest even; allocated if None).

    This is the per-token call of a decode loop, so the checks are one cheap
    pass (the C ABI validates sizes, alignment and overlaps again); a tensor that
    fails it is re-checked field by field for a precise error."""
    B, H, N = shp = r.shape
    ins = (r, w, k, v, kk, a)
    for t in ins:
        if not (t.is_cuda and t.dtype is torch.float32 and t.shape == shp and t.is_contiguous()):
            for name, u in zip(_STEP_IN, ins):
                _need_cuda(name, u, torch.float32, (B, H, N))
    scode = _STATE_CODES.get(state.dtype)
    if scode is None:
        raise TypeError("state must be float32, float16 or bfloat16")
    if not (state.is_cuda and state.shape == (B, H, N, N) and state.is_contiguous()):
        _need_cuda("state", state, state.dtype, (B, H, N, N))
    code = _out_code(out_dtype)
    if o is None:
        o = torch.empty((B, H, N), device=r.device, dtype=out_dtype)
    elif not (o.is_cuda and o.dtype is out_dtype and o.shape == shp and o.is_contiguous()):
        _need_cuda("o", o, out_dtype, (B, H, N))
    lib = _lib._lib or _lib.load()
    sh = _stream_handle(stream, r.device)
    if scode == _lib.F32:
        st = lib.wkv7_step_cast(B, H, N, r.data_ptr(), w.data_ptr(), k.data_ptr(), v.data_ptr(), kk.data_ptr(),
                                a.data_ptr(), state.data_ptr(), o.data_ptr(), code, sh)
    else:
        st = lib.wkv7_step_state(B, H, N, r.data_ptr(), w.data_ptr(), k.data_ptr(), v.data_ptr(), kk.data_ptr(),
                                 a.data_ptr(), state.data_ptr(), scode, o.data_ptr(), code, sh)
    if st:
        _lib.check(st, "wkv7_step")
    return o


def step_tail(r, w, k, v, kk, a, state, r_k, ln_w, ln_b, g, eps, y=None, o=None, want_o=False, stream=None):
    """One decode token with the time-mix tail fused:
    ``y = (GroupNorm_head(o) * ln_w + ln_b + (sum_i r_i k_i r_k_i) v) * g``.

    Inputs and ``g`` fp32 [B, H, N]; ``r_k``, ``ln_w``, ``ln_b`` fp32 [H, N];
    ``state`` updated in place.  Returns ``y`` (and ``o``, the WKV output, when
    ``want_o`` or ``o`` is given: ``(y, o)``).
    """
    B, H, N = r.shape
    for name, t in (("r", r), ("w", w), ("k", k), ("v", v), ("kk", kk), ("a", a), ("g", g)):
        _need_cuda(name, t, torch.float32, (B, H, N))
    for name, t in (("r_k", r_k), ("ln_w", ln_w), ("ln_b", ln_b)):
        _need_cuda(name, t, torch.float32, (H, N))
    _need_cuda("state", state, torch.float32, (B, H, N, N))
    if y is None:
        y = torch.empty((B, H, N), device=r.device, dtype=torch.float32)
    _need_cuda("y", y, torch.float32, (B, H, N))
    if o is None and want_o:
        o = torch.empty((B, H, N), device=r.device, dtype=torch.float32)
    if o is not None:
        _need_cuda("o", o, torch.float32, (B, H, N))
    lib = _lib.load()
    st = lib.wkv7_step_tail(B, H, N, _ptr(r), _ptr(w), _ptr(k), _ptr(v), _ptr(kk), _ptr(a), _ptr(state),
                            _ptr(o), _ptr(r_k), _ptr(ln_w), _ptr(ln_b), _ptr(g), float(eps), _ptr(y),
                            _stream(stream))
    _lib.check(st, "wkv7_step_tail")
    return (y, o) if o is not None else y


def tmix_tail(o, r, k, v, g, r_k, ln_w, ln_b, eps, y=None, stream=None):
    """The time-mix tail over packed rows (e.g. a prefill's outputs):
    ``o`` fp32 [rows, H, N]; ``r``, ``k``, ``v``, ``g`` fp32 or bf16 [rows, H, N]
    (one dtype); ``r_k``, ``ln_w``, ``ln_b`` fp32 [H, N].  ``y`` may be ``o``
    (in place); allocated when None.  Returns ``y``.
    """
    rows, H, N = o.shape
    _need_cuda("o", o, torch.float32, (rows, H, N))
    xdt = r.dtype
    if xdt not in (torch.float32, torch.bfloat16):
        raise TypeError("r, k, v, g must be float32 or bfloat16")
    for name, t in (("r", r), ("k", k), ("v", v), ("g", g)):
        _need_cuda(name, t, xdt, (rows, H, N))
    for name, t in (("r_k", r_k), ("ln_w", ln_w), ("ln_b", ln_b)):
        _need_cuda(name, t, torch.float32, (H, N))
    if y is None:
        y = torch.empty((rows, H, N), device=o.device, dtype=torch.float32)
    _need_cuda("y", y, torch.float32, (rows, H, N))
    lib = _lib.load()
    st = lib.wkv7_tmix_tail(rows, H, N, _lib.BF16 if xdt == torch.bfloat16 else _lib.F32, _ptr(o), _ptr(r), _ptr(k),
                            _ptr(v), _ptr(g), _ptr(r_k), _ptr(ln_w), _ptr(ln_b), float(eps), _ptr(y),
                            _stream(stream))
    _lib.check(st, "wkv7_tmix_tail")
    return y


def verify(r, w, k, v, kk, a, state, o=None, states=None, stream=None):
    """T tokens per row from a read-only state, keeping every position's state
    (the WKV part of a speculative step).  Inputs fp32 [B, T, H, N] (T <= 8);
    ``state`` fp32 [B, H, N, N] (not modified).  Returns ``(o [B, T, H, N],
    states [T, B, H, N, N])``.  Roll back with :func:`verify_commit`."""
    B, T, H, N = r.shape
    for name, t in (("r", r), ("w", w), ("k", k), ("v", v), ("kk", kk), ("a", a)):
        _need_cuda(name, t, torch.float32, (B, T, H, N))
    _need_cuda("state", state, torch.float32, (B, H, N, N))
    if o is None:
        o = torch.empty((B, T, H, N), device=r.device, dtype=torch.float32)
    if states is None:
        states = torch.empty((T, B, H, N, N), device=r.device, dtype=torch.float32)
    _need_cuda("o", o, torch.float32, (B, T, H, N))
    _need_cuda("states", states, torch.float32, (T, B, H, N, N))
    st = _lib.load().wkv7_verify(B, T, H, N, _ptr(r), _ptr(w), _ptr(k), _ptr(v), _ptr(kk), _ptr(a), _ptr(state),
                                 _ptr(o), _ptr(states), _stream(stream))
    _lib.check(st, "wkv7_verify")
    return o, states


def verify_commit(states, accept_len, state, stream=None):
    """Roll ``state`` [B, H, N, N] forward to each row's accepted length:
    ``state[b] = states[accept_len[b] - 1, b]`` (unchanged for 0).
    ``accept_len``: int32 CUDA [B]."""
    T, B, H, N, _ = states.shape
    _need_cuda("states", states, torch.float32, (T, B, H, N, N))
    _need_cuda("accept_len", accept_len, torch.int32, (B,))
    _need_cuda("state", state, torch.float32, (B, H, N, N))
    st = _lib.load().wkv7_verify_commit(B, T, H, N, _ptr(states), _ptr(accept_len), _ptr(state), _stream(stream))
    _lib.check(st, "wkv7_verify_commit")
    return state


def prefill_workspace_size(num_seqs: int, T_total: int, H: int, N: int = HEAD_SIZE) -> int:
    return int(_lib.load().wkv7_prefill_workspace_size(num_seqs, T_total, H, N))


def prefill(r, w, k, v, kk, a, cu_seqlens, initial_state=None, final_state=None, o=None,
            workspace=None, cu_seqlens_host=None, want_final_state=True, stream=None, out_dtype=torch.float32,
            state_dtype=None, tf32=False):
    """Packed varlen prefill.

    r, k, v, kk, a: [T_total, H, N] fp32 or bf16 (one dtype for all five);
    bf16 inputs run the chunked tensor-core kernel, fp32 inputs the exact
    token-serial kernel, or with ``tf32`` the chunked kernel (fp32 read in full,
    contracted at tf32: the bf16 inputs' error bound and domain w >= -1);
    w: fp32 [T_total, H, N]; ``cu_seqlens``: int32 CUDA [num_seqs + 1].
    ``initial_state``: fp32 [num_seqs, H, N, N] or None (zeros).
    ``final_state``: output buffer (may be ``initial_state`` for an in-place
    carry); allocated when None and ``want_final_state``.
    ``cu_seqlens_host``: optional CPU int32 copy (validated on the host, used
    for scheduling).  ``workspace``: uint8 CUDA buffer; ``prefill_workspace_size``
    bytes enable every schedule, and a smaller one is accepted as long as it
    holds the sequence order (the tail split is then skipped); allocated when
    None.  ``out_dtype``: the type of ``o`` (fp32, or bf16 rounded to nearest
    even).  ``state_dtype``: the type of both states (fp32, fp16 or bf16; by
    default that of ``initial_state`` or ``final_state``, else fp32); a 16-bit
    final state is rounded to nearest even once, when it is stored.  Returns
    ``(o, final_state)``.
    """
    T_total, H, N = r.shape
    xdt = r.dtype
    if xdt not in (torch.float32, torch.bfloat16):
        raise TypeError("r, k, v, kk, a must be float32 or bfloat16")
    for name, t in (("r", r), ("k", k), ("v", v), ("kk", kk), ("a", a)):
        _need_cuda(name, t, xdt, (T_total, H, N))
    _need_cuda("w", w, torch.float32, (T_total, H, N))
    _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    num_seqs = cu_seqlens.shape[0] - 1
    if state_dtype is None:
        state_dtype = (initial_state if initial_state is not None else
                       final_state if final_state is not None else torch.zeros(0)).dtype
    if state_dtype not in _STATE_CODES:
        raise TypeError("states must be float32, float16 or bfloat16")
    if initial_state is not None:
        _need_cuda("initial_state", initial_state, state_dtype, (num_seqs, H, N, N))
    if final_state is None and want_final_state:
        final_state = torch.empty((num_seqs, H, N, N), device=r.device, dtype=state_dtype)
    if final_state is not None:
        _need_cuda("final_state", final_state, state_dtype, (num_seqs, H, N, N))
    code = _out_code(out_dtype)
    if o is None:
        o = torch.empty((T_total, H, N), device=r.device, dtype=out_dtype)
    _need_cuda("o", o, out_dtype, (T_total, H, N))
    host_ptr = None
    if cu_seqlens_host is not None:
        if cu_seqlens_host.device.type != "cpu" or cu_seqlens_host.dtype != torch.int32:
            raise TypeError("cu_seqlens_host must be a CPU int32 tensor")
        cu_seqlens_host = cu_seqlens_host.contiguous()
        host_ptr = _ptr(cu_seqlens_host)
    lib = _lib.load()
    need = int(lib.wkv7_prefill_workspace_size(num_seqs, T_total, H, N))
    ws_bytes = 0
    if need > 0:
        if workspace is None:
            workspace = torch.empty(need, device=r.device, dtype=torch.uint8)
        _need_cuda("workspace", workspace, torch.uint8)
        ws_bytes = workspace.numel()
    st = lib.wkv7_prefill_state(num_seqs, T_total, H, N, _ptr(cu_seqlens), host_ptr, _x_code(xdt, tf32),
                                _ptr(r), _ptr(w), _ptr(k), _ptr(v), _ptr(kk), _ptr(a),
                                _ptr(initial_state), _ptr(final_state), _STATE_CODES[state_dtype], _ptr(o), code,
                                _ptr(workspace) if need > 0 else None, ws_bytes, _stream(stream))
    _lib.check(st, "wkv7_prefill")
    return o, final_state


def prefill_backward_workspace_size(num_seqs: int, T_total: int, H: int, N: int = HEAD_SIZE) -> int:
    return int(_lib.load().wkv7_prefill_backward_workspace_size(num_seqs, T_total, H, N))


def prefill_backward(r, w, k, v, kk, a, cu_seqlens, d_o, initial_state=None, d_final_state=None,
                     want_d_initial_state=True, grads=None, workspace=None, cu_seqlens_host=None, stream=None,
                     tf32=False):
    """Gradients of a :func:`prefill` call for L = <d_o, o> + <d_final_state, final_state>.

    The first seven arguments and ``initial_state`` are those of the forward
    call; ``d_o``: fp32 [T_total, H, N]; ``d_final_state``: fp32
    [num_seqs, H, N, N] or None (zeros).  ``grads``: optional tuple of six fp32
    [T_total, H, N] output buffers (dr, dw, dk, dv, dkk, da); ``workspace``:
    uint8 CUDA buffer of ``prefill_backward_workspace_size`` bytes (allocated
    when None).  Returns ``(dr, dw, dk, dv, dkk, da, d_initial_state)``
    (the last None unless ``want_d_initial_state``).
    """
    T_total, H, N = r.shape
    xdt = r.dtype
    if xdt not in (torch.float32, torch.bfloat16):
        raise TypeError("r, k, v, kk, a must be float32 or bfloat16")
    for name, t in (("r", r), ("k", k), ("v", v), ("kk", kk), ("a", a)):
        _need_cuda(name, t, xdt, (T_total, H, N))
    _need_cuda("w", w, torch.float32, (T_total, H, N))
    _need_cuda("d_o", d_o, torch.float32, (T_total, H, N))
    _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    num_seqs = cu_seqlens.shape[0] - 1
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None:
            _need_cuda(name, t, torch.float32, (num_seqs, H, N, N))
    if grads is None:
        grads = tuple(torch.empty((T_total, H, N), device=r.device, dtype=torch.float32) for _ in range(6))
    if len(grads) != 6:
        raise ValueError("grads must hold six tensors")
    for name, t in zip(("dr", "dw", "dk", "dv", "dkk", "da"), grads):
        _need_cuda(name, t, torch.float32, (T_total, H, N))
    ds0 = torch.empty((num_seqs, H, N, N), device=r.device, dtype=torch.float32) if want_d_initial_state else None
    host_ptr = None
    if cu_seqlens_host is not None:
        if cu_seqlens_host.device.type != "cpu" or cu_seqlens_host.dtype != torch.int32:
            raise TypeError("cu_seqlens_host must be a CPU int32 tensor")
        cu_seqlens_host = cu_seqlens_host.contiguous()
        host_ptr = _ptr(cu_seqlens_host)
    lib = _lib.load()
    need = int(lib.wkv7_prefill_backward_workspace_size(num_seqs, T_total, H, N))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=r.device, dtype=torch.uint8)
    _need_cuda("workspace", workspace, torch.uint8)
    st = lib.wkv7_prefill_backward(num_seqs, T_total, H, N, _ptr(cu_seqlens), host_ptr, _x_code(xdt, tf32),
                                   _ptr(r), _ptr(w), _ptr(k), _ptr(v), _ptr(kk), _ptr(a),
                                   _ptr(initial_state), _ptr(d_o), _ptr(d_final_state),
                                   *[_ptr(t) for t in grads], _ptr(ds0),
                                   _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check(st, "wkv7_prefill_backward")
    return (*grads, ds0)


def prefill_padded(r, w, k, v, kk, a, lens, initial_state=None, final_state=None, o=None, workspace=None,
                   lens_host=None, want_final_state=True, stream=None, out_dtype=torch.float32, tf32=False):
    """Prefill over a right-padded batch: inputs [B, T_max, H, N] (r, k, v, kk, a
    fp32 or bf16, w fp32; ``tf32`` as in :func:`prefill`); row b holds ``lens[b]`` real tokens (``lens`` int32
    CUDA [B]; ``lens_host`` an optional CPU copy, used for scheduling).  Returns
    ``(o [B, T_max, H, N] in out_dtype, final_state)``; o past each row's length
    is left as it was."""
    B, T_max, H, N = r.shape
    xdt = r.dtype
    if xdt not in (torch.float32, torch.bfloat16):
        raise TypeError("r, k, v, kk, a must be float32 or bfloat16")
    for name, t in (("r", r), ("k", k), ("v", v), ("kk", kk), ("a", a)):
        _need_cuda(name, t, xdt, (B, T_max, H, N))
    _need_cuda("w", w, torch.float32, (B, T_max, H, N))
    _need_cuda("lens", lens, torch.int32, (B,))
    if initial_state is not None:
        _need_cuda("initial_state", initial_state, torch.float32, (B, H, N, N))
    if final_state is None and want_final_state:
        final_state = torch.empty((B, H, N, N), device=r.device, dtype=torch.float32)
    if final_state is not None:
        _need_cuda("final_state", final_state, torch.float32, (B, H, N, N))
    code = _out_code(out_dtype)
    if o is None:
        o = torch.zeros((B, T_max, H, N), device=r.device, dtype=out_dtype)
    _need_cuda("o", o, out_dtype, (B, T_max, H, N))
    host_ptr = None
    if lens_host is not None:
        if lens_host.device.type != "cpu" or lens_host.dtype != torch.int32:
            raise TypeError("lens_host must be a CPU int32 tensor")
        lens_host = lens_host.contiguous()
        host_ptr = _ptr(lens_host)
    lib = _lib.load()
    need = int(lib.wkv7_prefill_workspace_size(B, B * T_max, H, N))
    ws_bytes = 0
    if need > 0:
        if workspace is None:
            workspace = torch.empty(need, device=r.device, dtype=torch.uint8)
        _need_cuda("workspace", workspace, torch.uint8)
        ws_bytes = workspace.numel()
    st = lib.wkv7_prefill_padded(B, T_max, H, N, _ptr(lens), host_ptr, _x_code(xdt, tf32),
                                 _ptr(r), _ptr(w), _ptr(k), _ptr(v), _ptr(kk), _ptr(a), _ptr(initial_state),
                                 _ptr(final_state), _ptr(o), code, _ptr(workspace) if need > 0 else None, ws_bytes,
                                 _stream(stream))
    _lib.check(st, "wkv7_prefill_padded")
    return o, final_state


def diag_bounded_wait(timeout_us: int = 20000, stream=None) -> None:
    """Run one device-side wait that nothing completes, bounded by ``timeout_us``;
    the device reports the expiry through the status word, so the next
    :func:`check_device_status` raises ``WKV7Error`` with the timeout status."""
    _lib.check(_lib.load().wkv7_diag_bounded_wait(int(timeout_us), _stream(stream)), "wkv7_diag_bounded_wait")


def check_device_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a device-side error."""
    st = _lib.load().wkv7_check_device_status(_stream(stream))
    _lib.check(st, "device status")
