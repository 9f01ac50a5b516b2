"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks return the documented status codes.  No GPU is needed: every
call here is rejected on the host before any CUDA call is made."""
import ctypes
import os
import re

import pytest

from rwkv_linear_attention_gb300 import _lib
from rwkv_linear_attention_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wkv7.h")

FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"WKV7_API\s+[\w\s\*]+?\b(wkv7_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_no_torch_types_in_the_abi():
    text = open(HEADER).read()
    assert "torch" not in text.lower().replace("pytorch", "")
    assert "at::" not in text and "Tensor" not in text


def test_status_strings(lib):
    for code in range(8):
        s = lib.wkv7_status_string(code)
        assert s and isinstance(s, bytes)
    assert lib.wkv7_status_string(0) == b"ok"
    assert lib.wkv7_abi_version() == 100


def _step(lib, B=2, H=3, N=64, ptrs=None):
    ptrs = ptrs or [FAKE + i * (1 << 24) for i in range(8)]
    P = ctypes.c_void_p
    return lib.wkv7_step(B, H, N, *[P(p) for p in ptrs], P(0))


def test_step_rejects_unsupported_head_size(lib):
    assert _step(lib, N=32) == _lib.ERR_UNSUPPORTED
    assert _step(lib, N=128) == _lib.ERR_UNSUPPORTED


def test_step_rejects_bad_sizes_and_nulls(lib):
    assert _step(lib, B=-1) == _lib.ERR_INVALID_ARG
    assert _step(lib, H=0) == _lib.ERR_INVALID_ARG
    ptrs = [FAKE + i * (1 << 24) for i in range(8)]
    for i in range(8):
        bad = list(ptrs)
        bad[i] = 0
        assert _step(lib, ptrs=bad) == _lib.ERR_INVALID_ARG


def test_step_zero_batch_is_noop(lib):
    assert _step(lib, B=0) == _lib.OK


def test_step_rejects_misaligned(lib):
    ptrs = [FAKE + i * (1 << 24) for i in range(8)]
    for i in range(8):
        bad = list(ptrs)
        bad[i] += 4
        assert _step(lib, ptrs=bad) == _lib.ERR_ALIGNMENT


def test_step_rejects_state_aliasing_an_input(lib):
    ptrs = [FAKE + i * (1 << 24) for i in range(8)]
    ptrs[6] = ptrs[3]  # state over v
    assert _step(lib, ptrs=ptrs) == _lib.ERR_INVALID_ARG


def _prefill(lib, num_seqs=2, T=10, H=2, N=64, cu_host=None, dtype=_lib.BF16, ptrs=None,
             s0=None, sf=None, ws=None, ws_bytes=0):
    P = ctypes.c_void_p
    base = ptrs or [FAKE + i * (1 << 26) for i in range(8)]
    host = None
    if cu_host is not None:
        arr = (ctypes.c_int32 * len(cu_host))(*cu_host)
        host = ctypes.cast(arr, P)
    return lib.wkv7_prefill(num_seqs, T, H, N, P(base[0]), host, dtype,
                            *[P(p) for p in base[1:7]], P(s0), P(sf), P(base[7]),
                            P(ws), ws_bytes, P(0))


def test_prefill_rejects_unsupported(lib):
    assert _prefill(lib, N=48) == _lib.ERR_UNSUPPORTED
    assert _prefill(lib, dtype=7) == _lib.ERR_UNSUPPORTED
    assert _prefill(lib, dtype=_lib.F16) == _lib.ERR_UNSUPPORTED  # 16-bit inputs are bf16 only


def test_prefill_tf32_inputs_are_four_bytes(lib):
    """x_dtype WKV7_TF32 (fp32 inputs through the chunked kernel) passes the host
    checks with 4-byte elements: an output placed right after a bf16-sized r
    overlaps an fp32 r."""
    T, H = 10, 2
    ptrs = [FAKE + i * (1 << 26) for i in range(8)]
    ptrs[7] = ptrs[1] + T * H * 64 * 2  # o right after r's first T*H*64*2 bytes
    assert _prefill(lib, T=T, H=H, ptrs=ptrs, cu_host=[0, 4, 10], dtype=_lib.TF32) == _lib.ERR_INVALID_ARG
    assert _prefill(lib, T=T, H=H, ptrs=ptrs, cu_host=[0, 4, 10], dtype=_lib.F32) == _lib.ERR_INVALID_ARG
    assert _prefill(lib, T=T, H=H, ptrs=ptrs, cu_host=[0, 4, 10], dtype=_lib.BF16) != _lib.ERR_INVALID_ARG
    bad = [FAKE + i * (1 << 26) for i in range(8)]
    bad[3] += 4
    assert _prefill(lib, ptrs=bad, cu_host=[0, 4, 10], dtype=_lib.TF32) == _lib.ERR_ALIGNMENT


def test_prefill_rejects_malformed_host_cu_seqlens(lib):
    assert _prefill(lib, cu_host=[0, 6, 4]) == _lib.ERR_INVALID_ARG   # decreasing and wrong total
    assert _prefill(lib, cu_host=[1, 5, 10]) == _lib.ERR_INVALID_ARG  # does not start at 0
    assert _prefill(lib, cu_host=[0, 5, 9]) == _lib.ERR_INVALID_ARG   # does not end at T_total
    assert _prefill(lib, cu_host=[0, 7, 6, 10][:3] + [10], num_seqs=3) == _lib.ERR_INVALID_ARG


def test_prefill_rejects_misaligned_and_null(lib):
    ptrs = [FAKE + i * (1 << 26) for i in range(8)]
    for i in range(8):
        bad = list(ptrs)
        bad[i] += 2
        assert _prefill(lib, ptrs=bad, cu_host=[0, 4, 10]) == _lib.ERR_ALIGNMENT
    bad = list(ptrs)
    bad[0] = 0
    assert _prefill(lib, ptrs=bad) == _lib.ERR_INVALID_ARG


def test_prefill_rejects_partial_state_overlap(lib):
    s0 = FAKE + 40 * (1 << 26)
    assert _prefill(lib, cu_host=[0, 4, 10], s0=s0, sf=s0 + 256) == _lib.ERR_INVALID_ARG


def test_prefill_rejects_output_over_input(lib):
    ptrs = [FAKE + i * (1 << 26) for i in range(8)]
    ptrs[7] = ptrs[1]  # o over r
    assert _prefill(lib, ptrs=ptrs, cu_host=[0, 4, 10]) == _lib.ERR_INVALID_ARG


def test_prefill_empty_batch(lib):
    assert _prefill(lib, num_seqs=0, T=0) == _lib.OK
    assert _prefill(lib, num_seqs=0, T=5) == _lib.ERR_INVALID_ARG


def test_workspace_size_is_pure(lib):
    a = lib.wkv7_prefill_workspace_size(8, 32768, 40, 64)
    b = lib.wkv7_prefill_workspace_size(8, 32768, 40, 64)
    assert a == b
    assert lib.wkv7_prefill_workspace_size(8, 32768, 40, 32) == 0


def _backward(lib, num_seqs=2, T=10, H=2, N=64, cu_host=None, dtype=_lib.BF16, ptrs=None, ws_bytes=None):
    """wkv7_prefill_backward with fake, never-dereferenced device pointers.

    ptrs: cu, r, w, k, v, kk, a, s0, d_o, dsf, dr, dw, dk, dv, dkk, da, ds0, workspace."""
    P = ctypes.c_void_p
    base = ptrs or [FAKE + i * (1 << 26) for i in range(18)]
    host = None
    if cu_host is not None:
        arr = (ctypes.c_int32 * len(cu_host))(*cu_host)
        host = ctypes.cast(arr, P)
    need = lib.wkv7_prefill_backward_workspace_size(num_seqs, T, H, N)
    wsb = need if ws_bytes is None else ws_bytes
    return lib.wkv7_prefill_backward(num_seqs, T, H, N, P(base[0]), host, dtype, *[P(x) for x in base[1:17]],
                                     P(base[17]), wsb, P(0))


def test_backward_rejects_unsupported(lib):
    assert _backward(lib, N=32) == _lib.ERR_UNSUPPORTED
    assert _backward(lib, dtype=5) == _lib.ERR_UNSUPPORTED


def test_backward_rejects_bad_sizes_and_host_cu_seqlens(lib):
    assert _backward(lib, num_seqs=-1) == _lib.ERR_INVALID_ARG
    assert _backward(lib, H=0) == _lib.ERR_INVALID_ARG
    assert _backward(lib, num_seqs=0, T=0) == _lib.OK
    assert _backward(lib, num_seqs=0, T=4) == _lib.ERR_INVALID_ARG
    assert _backward(lib, cu_host=[0, 6, 4]) == _lib.ERR_INVALID_ARG
    assert _backward(lib, cu_host=[0, 4, 9]) == _lib.ERR_INVALID_ARG


def test_backward_rejects_nulls_and_misalignment(lib):
    good = [FAKE + i * (1 << 26) for i in range(18)]
    required = [0, 1, 2, 3, 4, 5, 6, 8, 10, 11, 12, 13, 14, 15]  # cu, inputs, d_o, the six gradients
    for i in required:
        bad = list(good)
        bad[i] = 0
        assert _backward(lib, ptrs=bad) == _lib.ERR_INVALID_ARG, i
    for i in range(17):
        bad = list(good)
        bad[i] += 4
        assert _backward(lib, ptrs=bad, cu_host=[0, 4, 10]) == _lib.ERR_ALIGNMENT, i


def test_backward_rejects_small_workspace_and_overlaps(lib):
    need = lib.wkv7_prefill_backward_workspace_size(2, 10, 2, 64)
    assert need > 0
    assert _backward(lib, ws_bytes=need - 16) == _lib.ERR_WORKSPACE
    ptrs = [FAKE + i * (1 << 26) for i in range(18)]
    over = list(ptrs)
    over[10] = ptrs[1]  # dr over r
    assert _backward(lib, ptrs=over, cu_host=[0, 4, 10]) == _lib.ERR_INVALID_ARG
    over = list(ptrs)
    over[17] = ptrs[12]  # workspace over dk
    assert _backward(lib, ptrs=over, cu_host=[0, 4, 10]) == _lib.ERR_INVALID_ARG


def test_backward_workspace_size(lib):
    # the state at every 64-token boundary plus A, F, E, T and the decay table per chunk: (6 chunks + seqs) 16 KB planes
    n, T, H = 8, 32768, 40
    nc = T // 64 + n
    table = ((n + 1) * 4 + 255) // 256 * 256
    assert lib.wkv7_prefill_backward_workspace_size(n, T, H, 64) == table + (6 * nc + n) * H * 16384
    assert lib.wkv7_prefill_backward_workspace_size(n, T, H, 32) == 0


def test_diag_bounded_wait_rejects_out_of_range_bound(lib):
    assert lib.wkv7_diag_bounded_wait(0, ctypes.c_void_p(0)) == _lib.ERR_INVALID_ARG
    assert lib.wkv7_diag_bounded_wait(2000001, ctypes.c_void_p(0)) == _lib.ERR_INVALID_ARG


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "rwkv_linear_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "wkv7_oracle" not in text, f


def test_binding_input_codes():
    """The binding's prefill input code: bf16 always takes the chunked kernel; fp32 the
    exact token-serial kernel unless tf32 contraction is asked for."""
    import torch
    import rwkv_linear_attention_gb300 as wkv7
    assert wkv7._x_code(torch.bfloat16, False) == _lib.BF16
    assert wkv7._x_code(torch.bfloat16, True) == _lib.BF16
    assert wkv7._x_code(torch.float32, False) == _lib.F32
    assert wkv7._x_code(torch.float32, True) == _lib.TF32
    assert (_lib.F32, _lib.BF16, _lib.F16, _lib.TF32) == (0, 1, 2, 3)


def test_size_limits_are_checked_before_anything_else(lib):
    """2^30 heads per call is the most the 32-bit index math allows.  One more is rejected
    before the pointers are looked at; exactly that many passes the size check, so the
    misaligned pointers given here are what is reported.  Every case is rejected on the
    host: nothing is launched."""
    mis = [FAKE + 4 + i * (1 << 24) for i in range(8)]
    assert _step(lib, B=1 << 15, H=(1 << 15) + 1, ptrs=mis) == _lib.ERR_INVALID_ARG
    assert _step(lib, B=1 << 15, H=1 << 15, ptrs=mis) == _lib.ERR_ALIGNMENT
    # the backward's grid holds the heads in its y dimension (at most 65535)
    bad = [FAKE + 4 + i * (1 << 26) for i in range(18)]
    assert _backward(lib, num_seqs=1, T=10, H=65536, ptrs=bad, ws_bytes=0) == _lib.ERR_INVALID_ARG
    assert _backward(lib, num_seqs=1, T=10, H=65535, ptrs=bad, ws_bytes=0) == _lib.ERR_ALIGNMENT
    # its workspace query answers 0 past the head limit
    assert lib.wkv7_prefill_backward_workspace_size(1 << 15, 64, (1 << 15) + 1, 64) == 0
    assert lib.wkv7_prefill_backward_workspace_size(1 << 15, 64, 1 << 15, 64) > 0
