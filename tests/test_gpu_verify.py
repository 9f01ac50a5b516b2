"""Multi-token verify and rollback (speculative decoding) on the GPU.

wkv7_verify runs T tokens per row from a read-only state and keeps every
position's state; wkv7_verify_commit rolls the state to each row's accepted
length.  Checked against the oracle (position t's state is the final state of
a (t+1)-token run; bound 1e-5), against T sequential wkv7_step calls (the same
arithmetic: bit-exact), and for the argument and device checks.  Called
through the C ABI (the package binding)."""
import numpy as np
import pytest
import torch

import oracle
import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import _lib, inputs
from tests.gpu_util import rel_err

pytestmark = pytest.mark.gpu
NAMES = ("r", "w", "k", "v", "kk", "a")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _draw(B, T, H, seed, dev):
    x = inputs.draw_rwkkva((B, T, H, 64), seed=seed, device=dev)
    return {n: x[n].contiguous() for n in NAMES}


def _oracle_prefix(x, s0, t):
    """o and the final state of the first t tokens of every row, in double."""
    B, T, H, N = x["r"].shape
    arrs = [x[n][:, :t].reshape(B * t, H, N).cpu() for n in NAMES]
    return oracle.run(*arrs, cu_seqlens=np.arange(0, B * t + 1, t), s0=s0.cpu().double())


@pytest.mark.parametrize("B,T,H", [(3, 1, 12), (4, 4, 40), (16, 3, 40), (2, 8, 64)],
                         ids=["B3-T1", "B4-T4-2.9B", "B16-T3-2.9B", "B2-T8"])
def test_verify_matches_oracle(dev, B, T, H):
    x = _draw(B, T, H, 100 + T, dev)
    s0 = inputs.initial_state(B, H, 64, seed=101 + T, device=dev)
    keep = s0.clone()
    o, states = wkv7.verify(*(x[n] for n in NAMES), s0)
    wkv7.check_device_status()
    assert torch.equal(s0, keep), "the input state must not change"
    o_ref, _ = _oracle_prefix(x, s0, T)
    assert rel_err(o, o_ref.reshape(B, T, H, 64)) <= 1e-5
    for t in range(1, T + 1):
        _, s_ref = _oracle_prefix(x, s0, t)
        assert rel_err(states[t - 1], s_ref) <= 1e-5, f"state after {t} tokens"


def test_verify_equals_sequential_steps(dev):
    B, T, H = 8, 5, 40
    x = _draw(B, T, H, 110, dev)
    s0 = inputs.initial_state(B, H, 64, seed=111, device=dev)
    o, states = wkv7.verify(*(x[n] for n in NAMES), s0)
    state = s0.clone()
    for t in range(T):
        ot = wkv7.step(*(x[n][:, t].contiguous() for n in NAMES), state)
        assert torch.equal(ot, o[:, t]), f"o at position {t}"
        assert torch.equal(state, states[t]), f"state at position {t}"
    wkv7.check_device_status()


def test_commit_rolls_back_to_each_rows_accepted_length(dev):
    B, T, H = 6, 4, 12
    x = _draw(B, T, H, 120, dev)
    s0 = inputs.initial_state(B, H, 64, seed=121, device=dev)
    _, states = wkv7.verify(*(x[n] for n in NAMES), s0)
    acc = torch.tensor([0, 1, 2, 3, 4, 2], dtype=torch.int32, device=dev)
    state = s0.clone()
    wkv7.verify_commit(states, acc, state)
    wkv7.check_device_status()
    for b, a in enumerate(acc.tolist()):
        want = s0[b] if a == 0 else states[a - 1, b]
        assert torch.equal(state[b], want), f"row {b} accepted {a}"


def test_commit_rejects_out_of_range_lengths_on_the_device(dev):
    B, T, H = 3, 2, 4
    x = _draw(B, T, H, 130, dev)
    s0 = inputs.initial_state(B, H, 64, seed=131, device=dev)
    _, states = wkv7.verify(*(x[n] for n in NAMES), s0)
    state = s0.clone()
    wkv7.verify_commit(states, torch.tensor([1, 7, -1], dtype=torch.int32, device=dev), state)
    with pytest.raises(wkv7.WKV7Error) as e:
        wkv7.check_device_status()
    assert e.value.status == _lib.ERR_DEVICE_BOUNDS
    assert torch.equal(state[0], states[0, 0])
    assert torch.equal(state[1:], s0[1:]), "rows with an invalid length stay unchanged"


def test_verify_argument_errors(dev):
    B, H = 2, 4
    x = _draw(B, 9, H, 140, dev)
    s0 = inputs.initial_state(B, H, 64, seed=141, device=dev)
    with pytest.raises(wkv7.WKV7Error) as e:  # T = 9 > 8
        wkv7.verify(*(x[n] for n in NAMES), s0)
    assert e.value.status == _lib.ERR_INVALID_ARG
    x = _draw(B, 2, H, 142, dev)
    lib = _lib.load()
    import ctypes
    P = ctypes.c_void_p
    o = torch.empty(B, 2, H, 64, device=dev)
    # states aliasing an input
    st = lib.wkv7_verify(B, 2, H, 64, *[P(x[n].data_ptr()) for n in NAMES], P(s0.data_ptr()), P(o.data_ptr()),
                         P(x["r"].data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.ERR_INVALID_ARG
    assert wkv7.verify(*(t[:0] for t in (x[n] for n in NAMES)), s0[:0])[0].shape == (0, 2, H, 64)
