"""The WKV output cast to bf16 (wkv7_step_cast, wkv7_prefill_cast): the bf16
o must equal the fp32 path's o rounded to nearest even, bit for bit (the same
arithmetic, one rounding at the store), with the state identical; against the
oracle it is within the path's bound plus one bf16 rounding (2^-8 of the
largest output: bf16 keeps 8 significant bits).  Called
through the C ABI (the package binding)."""
import pytest
import torch

import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import inputs
from tests.gpu_util import oracle_prefill, rel_err

pytestmark = pytest.mark.gpu
NAMES = ("r", "w", "k", "v", "kk", "a")
BF16_ROUND = 2.0 ** -8


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("B,H", [(32, 40), (128, 64)], ids=["ring-form", "register-form"])
def test_step_bf16_output_is_the_rounded_fp32_output(dev, B, H):
    x = inputs.decode_inputs(B, H, 64, steps=1, seed=150 + B, device=dev)
    x = {n: t[0].contiguous() for n, t in x.items()}
    s0 = inputs.initial_state(B, H, 64, seed=151, device=dev)
    s32, s16 = s0.clone(), s0.clone()
    o32 = wkv7.step(*(x[n] for n in NAMES), s32)
    o16 = wkv7.step(*(x[n] for n in NAMES), s16, out_dtype=torch.bfloat16)
    wkv7.check_device_status()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(s16, s32)


@pytest.mark.parametrize("lens,dtype", [([300, 0, 129, 64], torch.bfloat16), ([4096] * 8, torch.bfloat16),
                                        ([70, 5], torch.float32)],
                         ids=["chunked-ragged", "chunked-2.9B", "token-serial-fp32-inputs"])
def test_prefill_bf16_output_is_the_rounded_fp32_output(dev, lens, dtype):
    H = 40 if len(lens) == 8 else 12
    p = inputs.prefill_inputs(lens, H, 64, seed=160 + len(lens), device=dev, x_dtype=dtype)
    s0 = inputs.initial_state(len(lens), H, 64, seed=161, device=dev)
    cu = p["cu_seqlens"]
    # a workspace holding only the sequence order: every pair runs whole in both calls
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    o32, f32 = wkv7.prefill(*(p[n] for n in NAMES), cu.to(dev), initial_state=s0, cu_seqlens_host=cu, workspace=ws)
    o16, f16 = wkv7.prefill(*(p[n] for n in NAMES), cu.to(dev), initial_state=s0, cu_seqlens_host=cu, workspace=ws,
                            out_dtype=torch.bfloat16)
    wkv7.check_device_status()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(f16, f32)
    if len(lens) < 8:
        o_ref, _ = oracle_prefill(p, cu, s0=s0)
        tol = (1e-5 if dtype == torch.float32 else 2e-3) + BF16_ROUND
        assert rel_err(o16.float(), o_ref) <= tol


def test_prefill_bf16_output_with_the_tail_split(dev):
    """With the full workspace a bf16 output takes the tail split when the plan's
    scratch fits (the part items' outputs go to fp32 rows and are rounded once,
    after the correction): it matches the oracle and the whole-pair bf16 result
    within one bf16 rounding."""
    lens, H = [1000] * 4, 40  # 160 pairs: on 152 SMs an 8-pair tail in 8 segments
    p = inputs.prefill_inputs(lens, H, 64, seed=170, device=dev)
    s0 = inputs.initial_state(len(lens), H, 64, seed=171, device=dev)
    cu = p["cu_seqlens"]
    need = wkv7.prefill_workspace_size(len(lens), sum(lens), H)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)
    o16, f16 = wkv7.prefill(*(p[n] for n in NAMES), cu.to(dev), initial_state=s0, cu_seqlens_host=cu, workspace=ws,
                            out_dtype=torch.bfloat16)
    small = torch.empty(256, dtype=torch.uint8, device=dev)
    o_whole, f_whole = wkv7.prefill(*(p[n] for n in NAMES), cu.to(dev), initial_state=s0, cu_seqlens_host=cu,
                                    workspace=small, out_dtype=torch.bfloat16)
    wkv7.check_device_status()
    S = torch.cuda.get_device_properties(0).multi_processor_count
    if 0 < (len(lens) * H) % S <= min(S // 2, 80):
        # the split ran: its state slots (after the 256-byte sequence order) were written
        assert bool((ws[256:256 + 16384] != 0xFF).any())
    o_ref, s_ref = oracle_prefill(p, cu, s0=s0)
    assert rel_err(o16.float(), o_ref) <= 2e-3 + BF16_ROUND
    assert rel_err(f16, s_ref) <= 2e-3
    assert rel_err(o16.float(), o_whole.float()) <= 2e-3 + BF16_ROUND
    assert rel_err(f16, f_whole) <= 2e-3


def test_prefill_bf16_output_with_a_rounds_split(dev):
    """A tail of 64 pairs (one sequence of 64 heads) is cut into more items than SMs:
    a longer first segment with the short part and transfer items in rounds.  With a
    bf16 output the part items' fp32 rows sit beside the transfer rows in the
    scratch; the result matches the oracle and the fp32-output call rounded once."""
    lens, H = [2500], 64
    p = inputs.prefill_inputs(lens, H, 64, seed=172, device=dev)
    s0 = inputs.initial_state(1, H, 64, seed=173, device=dev)
    cu = p["cu_seqlens"]
    o16, f16 = wkv7.prefill(*(p[n] for n in NAMES), cu.to(dev), initial_state=s0, cu_seqlens_host=cu,
                            out_dtype=torch.bfloat16)
    o32, f32 = wkv7.prefill(*(p[n] for n in NAMES), cu.to(dev), initial_state=s0, cu_seqlens_host=cu)
    wkv7.check_device_status()
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(f16, f32)
    o_ref, s_ref = oracle_prefill(p, cu, s0=s0)
    assert rel_err(o16.float(), o_ref) <= 2e-3 + BF16_ROUND
    assert rel_err(f16, s_ref) <= 2e-3
