"""The time-mix tail after WKV on the GPU, against the fp64 oracle:
y = (GroupNorm_head(o) * ln_w + ln_b + (sum_i r_i k_i r_k_i) v) * g.

* wkv7_step_tail: the decode step with the tail fused (both kernel forms: the
  shared-memory ring below 8192 heads and the register form from 8192), bound
  1e-5 on o, y and the state.
* wkv7_tmix_tail: the tail over packed rows, fp32 (1e-5) and bf16 row inputs
  (exact inputs, fp32 arithmetic: 1e-5), in place and out of place.
* prefill followed by the row tail on the prefill's outputs: the prefill bound
  2e-3 on y.
Called through the C ABI (the package binding)."""
import pytest
import torch

import oracle
import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import _lib, inputs
from tests.gpu_util import rel_err, oracle_prefill

pytestmark = pytest.mark.gpu

EPS = 64e-5


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _params(H, N, seed, dev):
    g = torch.Generator(device="cpu").manual_seed(seed)
    rk = (0.5 * torch.randn(H, N, generator=g)).to(dev)
    ln_w = (1.0 + 0.2 * torch.randn(H, N, generator=g)).to(dev)
    ln_b = (0.1 * torch.randn(H, N, generator=g)).to(dev)
    return rk, ln_w, ln_b


def _gate(shape, seed, dev, dtype=torch.float32):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.sigmoid(torch.randn(*shape, generator=g)).to(dev).to(dtype)


@pytest.mark.parametrize("B,H", [(2, 12), (32, 40), (128, 64)], ids=["B2-H12", "B32-H40", "B128-H64-register-form"])
def test_step_tail_matches_oracle(dev, B, H):
    N = 64
    x = inputs.decode_inputs(B, H, N, steps=1, seed=50 + B, device=dev)
    x = {n: t[0].contiguous() for n, t in x.items()}
    s0 = inputs.initial_state(B, H, N, seed=51 + B, device=dev)
    rk, ln_w, ln_b = _params(H, N, 52 + B, dev)
    gate = _gate((B, H, N), 53 + B, dev)
    state = s0.clone()
    y, o = wkv7.step_tail(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], state, rk, ln_w, ln_b, gate, EPS,
                          want_o=True)
    wkv7.check_device_status()
    cpu = {n: t.cpu() for n, t in x.items()}
    o_ref, s_ref = oracle.step(*(cpu[n] for n in ("r", "w", "k", "v", "kk", "a")), state=s0.cpu().double())
    y_ref = oracle.tail(o_ref, cpu["r"], cpu["k"], cpu["v"], rk.cpu(), ln_w.cpu(), ln_b.cpu(), gate.cpu(), EPS)
    assert rel_err(o, o_ref) <= 1e-5
    assert rel_err(state, s_ref) <= 1e-5
    assert rel_err(y, y_ref) <= 1e-5


def test_step_tail_without_o_equals_step_then_row_tail(dev):
    """o = NULL: only y is written; it equals wkv7_step followed by wkv7_tmix_tail."""
    B, H, N = 8, 40, 64
    x = inputs.decode_inputs(B, H, N, steps=1, seed=60, device=dev)
    x = {n: t[0].contiguous() for n, t in x.items()}
    s0 = inputs.initial_state(B, H, N, seed=61, device=dev)
    rk, ln_w, ln_b = _params(H, N, 62, dev)
    gate = _gate((B, H, N), 63, dev)
    s1, s2 = s0.clone(), s0.clone()
    y1 = wkv7.step_tail(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], s1, rk, ln_w, ln_b, gate, EPS)
    o2 = wkv7.step(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], s2)
    y2 = wkv7.tmix_tail(o2, x["r"], x["k"], x["v"], gate, rk, ln_w, ln_b, EPS)
    wkv7.check_device_status()
    assert torch.equal(s1, s2)
    assert rel_err(y1, y2) <= 1e-6


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("in_place", [False, True], ids=["out", "in-place"])
def test_row_tail_matches_oracle(dev, dtype, in_place):
    rows, H, N = 333, 12, 64
    g = torch.Generator(device="cpu").manual_seed(70)
    o = torch.randn(rows, H, N, generator=g).to(dev)
    r, k, v = (torch.randn(rows, H, N, generator=g).to(dev).to(dtype) for _ in range(3))
    gate = _gate((rows, H, N), 71, dev, dtype)
    rk, ln_w, ln_b = _params(H, N, 72, dev)
    y_ref = oracle.tail(o.cpu().double(), r.float().cpu(), k.float().cpu(), v.float().cpu(), rk.cpu(), ln_w.cpu(),
                        ln_b.cpu(), gate.float().cpu(), EPS)
    y = wkv7.tmix_tail(o, r, k, v, gate, rk, ln_w, ln_b, EPS, y=o if in_place else None)
    wkv7.check_device_status()
    if in_place:
        assert y.data_ptr() == o.data_ptr()
    assert rel_err(y, y_ref) <= 1e-5


def test_prefill_then_row_tail_matches_oracle(dev):
    lens, H, N = [300, 0, 129, 64], 12, 64
    p = inputs.prefill_inputs(lens, H, N, seed=80, device=dev)
    s0 = inputs.initial_state(len(lens), H, N, seed=81, device=dev)
    cu = p["cu_seqlens"]
    rk, ln_w, ln_b = _params(H, N, 82, dev)
    gate = _gate(tuple(p["r"].shape), 83, dev, torch.bfloat16)
    o, _ = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                        cu_seqlens_host=cu)
    y = wkv7.tmix_tail(o, p["r"], p["k"], p["v"], gate, rk, ln_w, ln_b, EPS)
    wkv7.check_device_status()
    o_ref, _ = oracle_prefill(p, cu, s0=s0)
    y_ref = oracle.tail(o_ref, p["r"].float().cpu(), p["k"].float().cpu(), p["v"].float().cpu(), rk.cpu(),
                        ln_w.cpu(), ln_b.cpu(), gate.float().cpu(), EPS)
    assert rel_err(y, y_ref) <= 2e-3


def test_tail_argument_errors(dev):
    B, H, N = 2, 4, 64
    x = inputs.decode_inputs(B, H, N, steps=1, seed=90, device=dev)
    x = {n: t[0].contiguous() for n, t in x.items()}
    state = inputs.initial_state(B, H, N, seed=91, device=dev)
    rk, ln_w, ln_b = _params(H, N, 92, dev)
    gate = _gate((B, H, N), 93, dev)
    args = (x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], state, rk, ln_w, ln_b, gate)
    for eps in (-1.0, float("nan"), float("inf")):
        with pytest.raises(wkv7.WKV7Error) as e:
            wkv7.step_tail(*args, eps)
        assert e.value.status == _lib.ERR_INVALID_ARG
    with pytest.raises(wkv7.WKV7Error) as e:  # y aliasing an input
        wkv7.step_tail(*args, EPS, y=x["v"])
    assert e.value.status == _lib.ERR_INVALID_ARG
    o = torch.randn(5, H, N, device=dev)
    with pytest.raises(wkv7.WKV7Error) as e:  # y partially overlapping o
        wkv7.tmix_tail(o[1:], o[1:], o[1:], o[1:], o[1:], rk, ln_w, ln_b, EPS, y=o[:4])
    assert e.value.status in (_lib.ERR_INVALID_ARG, _lib.ERR_ALIGNMENT)
    assert wkv7.tmix_tail(o[:0], o[:0], o[:0], o[:0], o[:0], rk, ln_w, ln_b, EPS).shape == (0, H, N)
