"""Prefill over a right-padded batch (wkv7_prefill_padded): row b of the
[B, T_max, H, N] inputs holds lens[b] real tokens.  Each row must give exactly
what the packed prefill gives for its real tokens (bit for bit: the same
kernels and arithmetic, with every pair run whole in both), match the oracle,
and leave o past each row's length untouched.  Called through the C ABI."""
import pytest
import torch

import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import _lib, inputs
from tests.gpu_util import oracle_prefill, rel_err

pytestmark = pytest.mark.gpu
NAMES = ("r", "w", "k", "v", "kk", "a")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _pad(p, lens, T_max):
    """Packed [T, H, N] inputs -> right-padded [B, T_max, H, N] (padding filled with noise)."""
    B = len(lens)
    out = {}
    for n in NAMES:
        x = p[n]
        pad = torch.randn(B, T_max, *x.shape[1:], device=x.device).to(x.dtype)
        if n == "w":
            pad = -torch.rand_like(pad)
        start = 0
        for b, L in enumerate(lens):
            pad[b, :L] = x[start:start + L]
            start += L
        out[n] = pad.contiguous()
    return out


@pytest.mark.parametrize("lens,T_max,H,dtype", [([300, 0, 129, 64], 320, 12, torch.bfloat16),
                                                ([5, 70, 64], 72, 4, torch.float32),
                                                ([1000, 700, 1000, 3], 1000, 40, torch.bfloat16)],
                         ids=["bf16-ragged", "fp32-token-serial", "bf16-40-heads"])
def test_padded_equals_packed(dev, lens, T_max, H, dtype):
    p = inputs.prefill_inputs(lens, H, 64, seed=180 + H, device=dev, x_dtype=dtype)
    s0 = inputs.initial_state(len(lens), H, 64, seed=181, device=dev)
    cu = p["cu_seqlens"]
    small = torch.empty(256, dtype=torch.uint8, device=dev)
    o_pk, f_pk = wkv7.prefill(*(p[n] for n in NAMES), cu.to(dev), initial_state=s0, cu_seqlens_host=cu,
                              workspace=small)
    x = _pad(p, lens, T_max)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    o = torch.full((len(lens), T_max, H, 64), float("nan"), device=dev)
    o_pd, f_pd = wkv7.prefill_padded(*(x[n] for n in NAMES), lens_t.to(dev), initial_state=s0, o=o,
                                     lens_host=lens_t, workspace=small)
    wkv7.check_device_status()
    assert torch.equal(f_pd, f_pk)
    start = 0
    for b, L in enumerate(lens):
        assert torch.equal(o_pd[b, :L], o_pk[start:start + L]), f"row {b}"
        assert torch.isnan(o_pd[b, L:]).all(), f"row {b}: padding was written"
        start += L
    o_ref, s_ref = oracle_prefill(p, cu, s0=s0)
    tol = 1e-5 if dtype == torch.float32 else 2e-3
    assert rel_err(f_pd, s_ref) <= tol


def test_padded_with_full_workspace_and_no_host_lengths(dev):
    """The default workspace (tail split allowed when the host lengths are given)
    and no host copy at all (lengths sorted on the device): both match the oracle."""
    lens, T_max, H = [1000, 700, 1000, 3], 1000, 40
    p = inputs.prefill_inputs(lens, H, 64, seed=190, device=dev)
    s0 = inputs.initial_state(len(lens), H, 64, seed=191, device=dev)
    x = _pad(p, lens, T_max)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    o_ref, s_ref = oracle_prefill(p, p["cu_seqlens"], s0=s0)
    for host in (lens_t, None):
        o, f = wkv7.prefill_padded(*(x[n] for n in NAMES), lens_t.to(dev), initial_state=s0, lens_host=host)
        wkv7.check_device_status()
        start = 0
        got = torch.cat([o[b, :L] for b, L in enumerate(lens)])
        assert rel_err(got, o_ref) <= 2e-3
        assert rel_err(f, s_ref) <= 2e-3


def test_padded_length_errors(dev):
    B, T_max, H = 2, 64, 4
    x = {n: torch.zeros(B, T_max, H, 64, device=dev) for n in NAMES}
    with pytest.raises(wkv7.WKV7Error) as e:  # host length past T_max
        wkv7.prefill_padded(*(x[n] for n in NAMES), torch.tensor([3, 65], dtype=torch.int32, device=dev),
                            lens_host=torch.tensor([3, 65], dtype=torch.int32))
    assert e.value.status == _lib.ERR_INVALID_ARG
    # the same length only on the device: reported by the kernel, nothing faults
    wkv7.prefill_padded(*(x[n] for n in NAMES), torch.tensor([3, 65], dtype=torch.int32, device=dev))
    with pytest.raises(wkv7.WKV7Error) as e:
        wkv7.check_device_status()
    assert e.value.status == _lib.ERR_INVALID_ARG or e.value.status == _lib.ERR_DEVICE_BOUNDS
