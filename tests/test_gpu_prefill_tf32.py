"""fp32 inputs through the chunked tensor-core prefill (x_dtype WKV7_TF32).

The chunked WY/UT kernel contracts at tf32 with fp32 accumulation whatever the
input type, so fp32 inputs taken through it are held to the bound of the
bf16-input prefill, max|gpu - oracle| / max|oracle| <= 2e-3, on o and on the
final state; its domain is the same (w >= -1).  The oracle runs on the same
fp32 inputs in fp64.

Besides the oracle:
* fp32 inputs that are exactly bf16 values give results bit-identical to the
  bf16-input call (the same kernel arithmetic on the same values; only the
  loads differ), at one chunk, over ragged multi-chunk sequences with initial
  states, and through the tail split;
* the recurrent path (wkv7_step token by token on the same fp32 inputs) and
  the exact token-serial prefill agree with it within 2e-3 (the pages'
  parallel-vs-recurrent check, at fp32 inputs);
* the bf16 output cast, 16-bit states, the right-padded layout and the
  backward accept the same input code.
"""
import pytest
import torch

import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import _lib, inputs
from tests.gpu_util import NAMES, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _run(p, dev, s0=None, tf32=True, ws=None, **kw):
    cu = p["cu_seqlens"]
    o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                         cu_seqlens_host=cu, tf32=tf32, workspace=ws, **kw)
    wkv7.check_device_status()
    return o, sf


def _check(p, o, sf, s0=None):
    o_ref, s_ref = oracle_prefill(p, p["cu_seqlens"], s0=s0)
    e_o, e_s = rel_err(o, o_ref), rel_err(sf, s_ref)
    assert e_o <= TOL and e_s <= TOL, f"o {e_o:.3e}, state {e_s:.3e} (bound {TOL:.0e})"


def _widened(p):
    """The same inputs as fp32 tensors holding exactly the bf16 values."""
    q = {n: p[n].float().contiguous() for n in NAMES}
    q["cu_seqlens"] = p["cu_seqlens"]
    return q


def _step_loop(p, s0):
    state = s0.clone()
    outs = []
    for t in range(p["r"].shape[0]):
        outs.append(wkv7.step(*(p[n][t:t + 1].contiguous() for n in NAMES), state).clone())
    return torch.cat(outs), state


def test_small_0p1b(dev):
    """The 0.1B case (1 x 64 tokens, 12 heads, fp32 inputs, zero initial state) through
    the chunked kernel, against the oracle, the token-serial kernel and the step loop."""
    cfg = inputs.SMALL_0P1B
    p = inputs.prefill_inputs([cfg["T"]], cfg["H"], cfg["N"], seed=1000, device=dev, x_dtype=torch.float32)
    o, sf = _run(p, dev)
    _check(p, o, sf)
    o_x, s_x = _run(p, dev, tf32=False)
    assert rel_err(o, o_x) <= TOL and rel_err(sf, s_x) <= TOL
    o_s, s_s = _step_loop(p, torch.zeros_like(sf))
    assert rel_err(o, o_s) <= TOL and rel_err(sf, s_s) <= TOL
    # the chunked kernel really ran: its tf32 results differ from the exact kernel's
    assert not torch.equal(o, o_x)


EDGE_LENGTHS = [[1], [63], [64], [65], [130, 3, 191], [1, 63, 64, 65, 0, 127, 200], [0, 0, 5], [3, 0]]


@pytest.mark.parametrize("lens", EDGE_LENGTHS, ids=lambda x: "-".join(map(str, x)))
@pytest.mark.parametrize("with_s0", [False, True], ids=["zero_s0", "s0"])
def test_varlen_edges(dev, lens, with_s0):
    H = 3
    p = inputs.prefill_inputs(lens, H, 64, seed=len(lens) * 37 + sum(lens), device=dev, x_dtype=torch.float32)
    s0 = inputs.initial_state(len(lens), H, 64, seed=19, device=dev) if with_s0 else None
    o, sf = _run(p, dev, s0=s0)
    _check(p, o, sf, s0=s0)
    for b, n in enumerate(lens):
        if n == 0:
            ref = s0[b] if s0 is not None else torch.zeros_like(sf[b])
            assert torch.equal(sf[b], ref)


@pytest.mark.parametrize("lens,H", [([64], 12), ([130, 3, 191, 0, 64], 5), ([3000], 8), ([2500], 64)],
                         ids=["one-chunk", "ragged", "split-1x3000-H8", "split-1x2500-H64"])
def test_bf16_values_bit_identical(dev, lens, H):
    p = inputs.prefill_inputs(lens, H, 64, seed=61 + H, device=dev, x_dtype=torch.bfloat16)
    s0 = inputs.initial_state(len(lens), H, 64, seed=61, device=dev)
    cu = p["cu_seqlens"]
    ws = torch.empty(max(wkv7.prefill_workspace_size(len(lens), int(cu[-1]), H), 16), dtype=torch.uint8, device=dev)
    o_b, s_b = _run(p, dev, s0=s0, ws=ws)
    o_f, s_f = _run(_widened(p), dev, s0=s0, ws=ws)
    assert torch.equal(o_b, o_f)
    assert torch.equal(s_b, s_f)


@pytest.mark.parametrize("lens,H,seed", [([3000], 8, 71), ([2000, 1500, 700], 10, 72), ([2500], 64, 74)],
                         ids=["1x3000-H8", "unequal-H10", "1x2500-H64-rounds"])
def test_tail_split_against_oracle(dev, lens, H, seed):
    p = inputs.prefill_inputs(lens, H, 64, seed=seed, device=dev, x_dtype=torch.float32)
    s0 = inputs.initial_state(len(lens), H, 64, seed=seed, device=dev)
    o, sf = _run(p, dev, s0=s0)
    _check(p, o, sf, s0=s0)


def test_step_and_chunked_prefill_agree(dev):
    T, H = 333, 4
    p = inputs.prefill_inputs([T], H, 64, seed=76, device=dev, x_dtype=torch.float32)
    s0 = inputs.initial_state(1, H, 64, seed=76, device=dev)
    o_p, s_p = _run(p, dev, s0=s0)
    o_s, s_s = _step_loop(p, s0)
    assert rel_err(o_p, o_s) <= TOL
    assert rel_err(s_p, s_s) <= TOL


@pytest.mark.parametrize("kind", ["all", "channels"])
def test_at_the_domain_bound(dev, kind):
    lens, H = [64, 101, 192, 0, 7], 3
    p = inputs.prefill_inputs(lens, H, 64, seed=78, device=dev, x_dtype=torch.float32)
    if kind == "all":
        p["w"].fill_(-1.0)
    else:
        p["w"].zero_()
        p["w"][..., 0::2] = -1.0
    s0 = inputs.initial_state(len(lens), H, 64, seed=78, device=dev)
    o, sf = _run(p, dev, s0=s0)
    _check(p, o, sf, s0=s0)


def test_below_the_bound_is_reported(dev):
    lens, H = [64, 101], 3
    p = inputs.prefill_inputs(lens, H, 64, seed=79, device=dev, x_dtype=torch.float32)
    p["w"][70, 1, 17] = -1.001
    cu = p["cu_seqlens"]
    with pytest.raises(wkv7.WKV7Error) as e:
        wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), cu_seqlens_host=cu, tf32=True)
        wkv7.check_device_status()
    assert e.value.status == _lib.ERR_INVALID_ARG
    # the exact kernel has no such limit
    o, sf = _run(p, dev, tf32=False)
    o_ref, s_ref = oracle_prefill(p, cu)
    assert rel_err(o, o_ref) <= 1e-5 and rel_err(sf, s_ref) <= 1e-5


def test_cast_and_16bit_state(dev):
    """bf16 o and an fp16 state from fp32 inputs: the same kernels, so each equals the
    fp32 result rounded once."""
    lens, H = [200, 64, 5], 4
    p = inputs.prefill_inputs(lens, H, 64, seed=81, device=dev, x_dtype=torch.float32)
    s0 = inputs.initial_state(len(lens), H, 64, seed=81, device=dev).half()
    o32, s32 = _run(p, dev, s0=s0.float())
    o16, s16 = _run(p, dev, s0=s0, out_dtype=torch.bfloat16)
    assert s16.dtype == torch.float16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(s16, s32.to(torch.float16))
    _check(p, o32, s32, s0=s0.float())


def test_padded_layout(dev):
    B, T_max, H = 3, 150, 4
    lens = [150, 37, 0]
    p = inputs.prefill_inputs([T_max] * B, H, 64, seed=83, device=dev, x_dtype=torch.float32)
    x = {n: p[n].view(B, T_max, H, 64) for n in NAMES}
    s0 = inputs.initial_state(B, H, 64, seed=83, device=dev)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    o, sf = wkv7.prefill_padded(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], lens_t.to(dev), initial_state=s0,
                                lens_host=lens_t, tf32=True)
    wkv7.check_device_status()
    # the same rows packed
    packed = {n: torch.cat([x[n][b, :lens[b]] for b in range(B)]).contiguous() for n in NAMES}
    packed["cu_seqlens"] = inputs.cu_seqlens_of(lens)
    o_p, s_p = _run(packed, dev, s0=s0)
    assert torch.equal(sf, s_p)
    assert torch.equal(torch.cat([o[b, :lens[b]] for b in range(B)]), o_p)
    _check(packed, o_p, s_p, s0=s0)


def test_backward_accepts_the_code(dev):
    lens, H = [100, 30], 2
    p = inputs.prefill_inputs(lens, H, 64, seed=85, device=dev, x_dtype=torch.float32)
    cu = p["cu_seqlens"]
    d_o, d_sf = inputs.upstream_gradients(int(cu[-1]), len(lens), H, 64, seed=85, device=dev)
    args = (p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), d_o)
    g1 = wkv7.prefill_backward(*args, d_final_state=d_sf, cu_seqlens_host=cu, tf32=True)
    g2 = wkv7.prefill_backward(*args, d_final_state=d_sf, cu_seqlens_host=cu)
    wkv7.check_device_status()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
