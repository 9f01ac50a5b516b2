"""16-bit recurrent state (wkv7_step_state, wkv7_prefill_state) against the fp64 oracle.

The Core AI model zoo note (section 5) runs an fp16 export with fp16 state
arrays.  Here the state is stored in fp16 or bf16, widened to fp32 exactly on
load, updated in fp32 and rounded to nearest even on store.  The oracle runs
from the same 16-bit state widened to double ("the same rounded states"), so
the only difference besides fp32 arithmetic is the final rounding of the state:

* o is computed from the fp32 state before rounding: the fp32 bound, 1e-5
  (decode) or 2e-3 (bf16-input prefill);
* the stored state differs from the exact result by at most half a 16-bit ulp,
  i.e. 2^-11 |S| (fp16, 11 significant bits) or 2^-8 |S| (bf16, 8 bits), plus
  the fp32 error: bound = 2^-11 + 1e-5 resp. 2^-8 + 1e-5 of max|S| for the
  step; the prefill adds its 2e-3.

Besides the oracle, the 16-bit paths are checked for consistency with the fp32
paths: the prefill's 16-bit final state is bit-identical to its fp32 final state
rounded (same kernels and arithmetic, only the store differs), and the step's
16-bit result equals the fp32 step's result rounded except where the two fp32
summation orders straddle a rounding boundary (at most one 16-bit ulp).
"""
import pytest
import torch

import oracle
import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import inputs
from tests.gpu_util import NAMES, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

DTYPES = {"f16": (torch.float16, 2.0 ** -11), "bf16": (torch.bfloat16, 2.0 ** -8)}
TOL_O = 1e-5
TOL_PREFILL = 2e-3


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _oracle_step(x, state16):
    return oracle.step(*(x[n].cpu() for n in NAMES), state=state16.double().cpu())


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("B,H", [(1, 40), (8, 40), (32, 40), (256, 64)], ids=["2.9B-B1", "2.9B-B8", "2.9B-B32", "7.2B-B256"])
def test_step_state16_against_oracle(dev, dt, B, H):
    dtype, half_ulp = DTYPES[dt]
    x = {n: t[0].contiguous() for n, t in inputs.decode_inputs(B, H, 64, steps=1, seed=301 + B, device=dev).items()}
    s0 = inputs.initial_state(B, H, 64, seed=301, std=0.1, device=dev).to(dtype)
    state = s0.clone()
    o = wkv7.step(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], state)
    wkv7.check_device_status()
    o_ref, s_ref = _oracle_step(x, s0)
    assert rel_err(o, o_ref) <= TOL_O
    e_s = rel_err(state.float(), s_ref)
    assert e_s <= half_ulp + 1e-5, f"state {e_s:.3e} (bound {half_ulp + 1e-5:.3e})"


@pytest.mark.parametrize("dt", list(DTYPES))
def test_step_state16_64_steps_each_against_oracle(dev, dt):
    """64 consecutive steps; each checked against the oracle run from the GPU's
    own (rounded) state before that step."""
    dtype, half_ulp = DTYPES[dt]
    B, H, T = 4, 40, 64
    xs = inputs.decode_inputs(B, H, 64, steps=T, seed=311, device=dev)
    state = inputs.initial_state(B, H, 64, seed=311, std=0.1, device=dev).to(dtype)
    for t in range(T):
        x = {n: xs[n][t].contiguous() for n in NAMES}
        before = state.clone()
        o = wkv7.step(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], state)
        o_ref, s_ref = _oracle_step(x, before)
        assert rel_err(o, o_ref) <= TOL_O, t
        assert rel_err(state.float(), s_ref) <= half_ulp + 1e-5, t
    wkv7.check_device_status()


@pytest.mark.parametrize("dt", list(DTYPES))
def test_step_state16_matches_fp32_step_rounded(dev, dt):
    dtype, _ = DTYPES[dt]
    B, H = 32, 40
    x = {n: t[0].contiguous() for n, t in inputs.decode_inputs(B, H, 64, steps=1, seed=321, device=dev).items()}
    s16 = inputs.initial_state(B, H, 64, seed=321, std=0.1, device=dev).to(dtype)
    s32 = s16.float()
    o16 = wkv7.step(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], s16)
    o32 = wkv7.step(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], s32)
    wkv7.check_device_status()
    assert rel_err(o16, o32) <= 1e-6
    ref = s32.to(dtype)
    differ = (s16 != ref)
    assert differ.float().mean().item() <= 1e-3
    # where they differ, by one 16-bit ulp at most
    ulp = (ref.float().abs() * (2.0 ** -10 if dtype == torch.float16 else 2.0 ** -7)).clamp_min(2.0 ** -24)
    assert ((s16.float() - ref.float()).abs() <= ulp + 1e-12).all()


def test_step_state16_rejects_overlap_and_bad_dtype(dev):
    B, H = 2, 3
    x = {n: t[0].contiguous() for n, t in inputs.decode_inputs(B, H, 64, steps=1, seed=1, device=dev).items()}
    with pytest.raises(TypeError):
        wkv7.step(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], torch.zeros(B, H, 64, 64, device=dev,
                                                                                 dtype=torch.float64))


PREFILL_CASES = [([64, 101, 0, 7], 3, torch.bfloat16), ([3000], 8, torch.bfloat16), ([150, 33], 3, torch.float32)]


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("lens,H,xdt", PREFILL_CASES, ids=["ragged-bf16", "tail-split-bf16", "token-serial-fp32"])
def test_prefill_state16_against_oracle(dev, dt, lens, H, xdt):
    dtype, half_ulp = DTYPES[dt]
    p = inputs.prefill_inputs(lens, H, 64, seed=331, device=dev, x_dtype=xdt)
    cu = p["cu_seqlens"]
    s0 = inputs.initial_state(len(lens), H, 64, seed=331, std=0.1, device=dev).to(dtype)
    need = wkv7.prefill_workspace_size(len(lens), int(cu[-1]), H)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                         cu_seqlens_host=cu, workspace=ws)
    wkv7.check_device_status()
    assert sf.dtype == dtype
    o_ref, s_ref = oracle_prefill(p, cu, s0=s0.float())
    tol = TOL_PREFILL if xdt == torch.bfloat16 else 1e-5
    assert rel_err(o, o_ref) <= tol
    e_s = rel_err(sf.float(), s_ref)
    assert e_s <= tol + half_ulp, f"state {e_s:.3e} (bound {tol + half_ulp:.3e})"
    # the same call with fp32 states (the 16-bit initial state widened): same kernels, so the
    # 16-bit final state is exactly the fp32 one rounded once
    o32, sf32 = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0.float(),
                             cu_seqlens_host=cu, workspace=ws)
    wkv7.check_device_status()
    assert torch.equal(o, o32)
    assert torch.equal(sf, sf32.to(dtype))
