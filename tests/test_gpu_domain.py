"""The chunked kernels' domain, w >= -1, at its bound and beyond it.

The chunked prefill and its backward take a chunk's decay factors relative to
the chunk's 32nd token, so a scaled operand carries a factor within
e^{+-32|w|} and the removal block C^T T Q of a chunk's transition, where a
strongly decaying channel meets a non-decaying one through the UT transform,
reaches e^{64|w|} (fp32 holds up to e^{88.7}).  An earlier stated bound of
-2.5 failed exactly there: w = -2.5 on even channels and 0 on odd ones gave a
NaN final state.  The tests below run at the bound against the fp64 oracle
(full 64-token chunks, a ragged tail, a random initial state; the bound on
every element, on alternate 32-token blocks, on alternate channels, and
uniform in [-1, 0]), and check that a w below the bound is reported by the
device as WKV7_ERR_INVALID_ARG without a fault (a check on the values, not a
trap).  The fp32-input prefill takes the token-serial kernel, which has no
such limit.
"""
import numpy as np
import pytest
import torch

import oracle
import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import _lib, inputs
from tests.gpu_util import NAMES, host_f32, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-3
TOL_FP32 = 1e-5
W_MIN = -1.0
LENS = [64, 101, 192, 0, 7]  # full chunks, a ragged tail, three chunks, an empty and a short sequence
H = 3


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _pattern(p, kind):
    w = p["w"]
    if kind == "all":
        w.fill_(W_MIN)
    elif kind == "halves":  # the bound on alternate 32-token blocks, no decay between
        t = torch.arange(w.shape[0], device=w.device)
        w.copy_(torch.where(((t // 32) % 2 == 0)[:, None, None], torch.full_like(w, W_MIN), torch.zeros_like(w)))
    elif kind == "channels":  # the bound on even channels, no decay on odd ones
        w.zero_()
        w[..., 0::2] = W_MIN
    elif kind == "uniform":  # uniform in [W_MIN, 0] per element
        g = torch.Generator(device=w.device).manual_seed(5)
        w.copy_(torch.rand(w.shape, generator=g, device=w.device) * W_MIN)
    return p


@pytest.mark.parametrize("kind", ["all", "halves", "channels", "uniform"])
def test_prefill_at_the_bound(dev, kind):
    p = _pattern(inputs.prefill_inputs(LENS, H, 64, seed=41, device=dev), kind)
    s0 = inputs.initial_state(len(LENS), H, 64, seed=41, device=dev)
    cu = p["cu_seqlens"]
    o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                         cu_seqlens_host=cu)
    wkv7.check_device_status()  # no domain report at the bound itself
    assert torch.isfinite(o).all() and torch.isfinite(sf).all()
    o_ref, s_ref = oracle_prefill(p, cu, s0=s0)
    e_o, e_s = rel_err(o, o_ref), rel_err(sf, s_ref)
    assert e_o <= TOL and e_s <= TOL, f"o {e_o:.3e}, state {e_s:.3e}"


@pytest.mark.parametrize("kind", ["all", "halves", "channels", "uniform"])
def test_backward_at_the_bound(dev, kind):
    p = _pattern(inputs.prefill_inputs(LENS, H, 64, seed=43, device=dev), kind)
    cu = p["cu_seqlens"]
    T = int(cu[-1])
    s0 = inputs.initial_state(len(LENS), H, 64, seed=43, device=dev)
    d_o, dsf = inputs.upstream_gradients(T, len(LENS), H, 64, seed=43, device=dev)
    got = wkv7.prefill_backward(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), d_o,
                                initial_state=s0, d_final_state=dsf, cu_seqlens_host=cu)
    wkv7.check_device_status()
    arrs = [host_f32(p[n]) for n in NAMES]
    ref = oracle.backward(*arrs, d_o.double().cpu().numpy(), cu_seqlens=cu.numpy().astype(np.int64),
                          s0=s0.double().cpu().numpy(), d_sfinal=dsf.double().cpu().numpy())
    errs = {n: rel_err(g, r) for n, g, r in zip(("dr", "dw", "dk", "dv", "dkk", "da", "ds0"), got, ref)}
    assert all(e <= TOL for e in errs.values()), errs


@pytest.mark.parametrize("bad", [W_MIN - 1e-3, float("-inf")], ids=["just_below", "minus_inf"])
def test_below_the_bound_is_reported(dev, bad):
    p = inputs.prefill_inputs(LENS, H, 64, seed=45, device=dev)
    p["w"][70, 1, 17] = bad  # one element of the second sequence
    cu = p["cu_seqlens"]
    with pytest.raises(wkv7.WKV7Error) as e:
        wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), cu_seqlens_host=cu)
        wkv7.check_device_status()
    assert e.value.status == _lib.ERR_INVALID_ARG
    d_o, _ = inputs.upstream_gradients(int(cu[-1]), len(LENS), H, 64, seed=45, device=dev)
    with pytest.raises(wkv7.WKV7Error) as e:
        wkv7.prefill_backward(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), d_o, cu_seqlens_host=cu)
        wkv7.check_device_status()
    assert e.value.status == _lib.ERR_INVALID_ARG
    # the report was read and cleared: the same call on in-domain inputs is clean
    p["w"][70, 1, 17] = W_MIN
    o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), cu_seqlens_host=cu)
    wkv7.check_device_status()
    o_ref, s_ref = oracle_prefill(p, cu)
    assert rel_err(o, o_ref) <= TOL and rel_err(sf, s_ref) <= TOL


def test_fp32_prefill_has_no_bound(dev):
    """fp32 inputs take the token-serial kernel: w far below -2.5 is fine there."""
    p = inputs.prefill_inputs([150, 64], H, 64, seed=47, device=dev, x_dtype=torch.float32)
    p["w"][:75] = -6.0
    p["w"][75:150, :, 0::2] = -3.0  # strong decay on some channels, mild on the others
    s0 = inputs.initial_state(2, H, 64, seed=47, device=dev)
    cu = p["cu_seqlens"]
    o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                         cu_seqlens_host=cu)
    wkv7.check_device_status()
    o_ref, s_ref = oracle_prefill(p, cu, s0=s0)
    assert rel_err(o, o_ref) <= TOL_FP32 and rel_err(sf, s_ref) <= TOL_FP32
