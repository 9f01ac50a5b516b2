"""wkv7_prefill_noalloc, the prefill for callers that cannot allocate device
memory (a memory plan fixed up front, code recorded during stream capture, a
host that only holds pointers to someone else's buffers), against the
regular wkv7_prefill and against the fp64 oracle.

It runs the same kernels with its scratch in a fixed device array instead of
a caller workspace, so its outputs must match the regular entry point's
within the prefill tolerance -- on two calls in a row, the second reusing the
scratch the first one left behind -- and, since both share those kernels,
each call is also held to the oracle on its own.  The batches cover the
longest-first schedule (unequal lengths: the order is written into the fixed
array and read back) and the two cases that write no order at all (one
sequence; equal lengths).  Called through the C ABI.  This file is named to be
collected last.
"""
import ctypes

import pytest
import torch

import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import _lib, inputs
from tests.gpu_util import oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _noalloc(p, s0, sf, o):
    P = ctypes.c_void_p
    cu = p["cu_seqlens"]
    cu_dev = cu.to(p["r"].device)
    T, H, N = p["r"].shape
    lib = _lib.load()
    st = lib.wkv7_prefill_noalloc(
        cu.shape[0] - 1, T, H, N, P(cu_dev.data_ptr()), ctypes.cast(cu.numpy().ctypes.data, P), _lib.BF16,
        *[P(p[n].data_ptr()) for n in ("r", "w", "k", "v", "kk", "a")],
        P(s0.data_ptr()) if s0 is not None else None, P(sf.data_ptr()), P(o.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))
    _lib.check(st, "wkv7_prefill_noalloc")
    wkv7.check_device_status()
    return o, sf


# Two unequal-length batches (the longest-first order is written into the fixed
# array and read back on each call), one single-sequence batch and one batch of
# equal lengths (neither writes an order).
CASES = [([300, 5, 129, 64, 0, 700], 3, 31), ([17, 640, 2, 255], 2, 32), ([1000], 4, 33), ([130, 130, 130], 2, 34)]


@pytest.mark.parametrize("call", [0, 1])
def test_noalloc_matches_prefill_two_calls_in_a_row(dev, call):
    for lens, H, seed in CASES:
        p = inputs.prefill_inputs(lens, H, 64, seed=seed + call, device=dev)
        s0 = inputs.initial_state(len(lens), H, 64, seed=seed, device=dev)
        o_ref, sf_ref = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], p["cu_seqlens"].to(dev),
                                     initial_state=s0, cu_seqlens_host=p["cu_seqlens"])
        wkv7.check_device_status()
        o = torch.full_like(o_ref, float("nan"))
        sf = torch.full_like(sf_ref, float("nan"))
        _noalloc(p, s0, sf, o)
        assert rel_err(o, o_ref) <= TOL
        assert rel_err(sf, sf_ref) <= TOL
        # both entry points run the same kernels, so hold this one to the oracle too
        o_or, s_or = oracle_prefill(p, p["cu_seqlens"], s0=s0)
        assert rel_err(o, o_or) <= TOL, lens
        assert rel_err(sf, s_or) <= TOL, lens


def test_noalloc_rejects_batches_beyond_its_scratch(dev):
    n = 4097  # one more than WKV7_NOALLOC_MAX_SEQS
    p = inputs.prefill_inputs([1] * n, 1, 64, seed=1, device=dev)
    o = torch.empty(n, 1, 64, device=dev)
    sf = torch.empty(n, 1, 64, 64, device=dev)
    with pytest.raises(wkv7.WKV7Error) as e:
        _noalloc(p, None, sf, o)
    assert e.value.status == _lib.ERR_WORKSPACE
