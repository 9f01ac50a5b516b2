"""Decode step (wkv7_step) against the fp64 oracle, element by element.

Bound: max|gpu - oracle| / max|oracle| <= 1e-5 for o and for the state, the
fp32-decode tolerance.  Inputs and initial states are seeded and synthetic;
the oracle always starts from the exact fp32 values the GPU holds.
"""
import numpy as np
import pytest
import torch

import oracle
import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import inputs
from tests.gpu_util import NAMES, host_f32, rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _step(x, state, o=None):
    return wkv7.step(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], state, o)


def test_small_0p1b_step_loop_from_zero(dev):
    """B=1, T=64, H=12, zero state: 64 consecutive wkv7_step calls."""
    cfg = inputs.SMALL_0P1B
    T, H, N = cfg["T"], cfg["H"], cfg["N"]
    x = inputs.draw_rwkkva((T, 1, H, N), seed=1000, device=dev)
    state = torch.zeros(1, H, N, N, device=dev)
    outs = []
    for t in range(T):
        outs.append(_step({n: x[n][t] for n in NAMES}, state).clone())
    wkv7.check_device_status()
    o = torch.stack(outs)[:, 0]
    o_ref, s_ref = oracle.run(*(host_f32(x[n][:, 0]) for n in NAMES))
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(state, s_ref) <= TOL


@pytest.mark.parametrize("B", [1, 3, 8])
def test_step_random_state(dev, B):
    H, N = 5, 64
    x = inputs.decode_inputs(B, H, N, steps=1, seed=77 + B, device=dev)
    x = {n: t[0].contiguous() for n, t in x.items()}
    s0 = inputs.initial_state(B, H, N, seed=77, device=dev)
    state = s0.clone()
    o = _step(x, state)
    wkv7.check_device_status()
    o_ref, s_ref = oracle.step(*(x[n] for n in NAMES), state=s0.double().cpu())
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(state, s_ref) <= TOL


def test_step_projector_and_decay_bound(dev):
    """Degenerate inputs: a = 1 with unit kk and w = 0 (the projector), and the
    log-decay at its bound -0.606531 on every channel."""
    B, H, N = 2, 4, 64
    x = inputs.decode_inputs(B, H, N, steps=1, seed=5, device=dev)
    x = {n: t[0].contiguous() for n, t in x.items()}
    x["a"] = torch.ones_like(x["a"])
    x["w"] = torch.zeros_like(x["w"])
    x["w"][1] = -0.606531
    s0 = inputs.initial_state(B, H, N, seed=5, device=dev)
    state = s0.clone()
    o = _step(x, state)
    o_ref, s_ref = oracle.step(*(x[n] for n in NAMES), state=s0.double().cpu())
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(state, s_ref) <= TOL


def _warm_state(L, B, H, N, warm, seed, dev):
    """The oracle's state after ``warm`` random tokens from zero, per (layer, b)."""
    out = []
    for layer in range(L):
        x = inputs.draw_rwkkva((B * warm, H, N), seed=seed + 7 * layer, device=dev)
        cu = np.arange(B + 1, dtype=np.int64) * warm
        _, s = oracle.run(*(host_f32(x[n]) for n in NAMES), cu_seqlens=cu)
        out.append(torch.from_numpy(s).float())
    return torch.stack(out)


@pytest.mark.parametrize("B", [1, 8, 32])
def test_decode_2p9b_geometry(dev, B):
    """2.9B geometry: 32 layers x 40 heads, states = oracle state after 256
    tokens, a pool of 16 input sets per layer cycled.  Steps 1-8 are checked on
    every slab; then 1024 steps on 64 sampled (layer, b, head) slabs."""
    cfg = inputs.DECODE_2P9B
    L, H, N, P = cfg["layers"], cfg["H"], cfg["N"], cfg["pool"]
    steps = cfg["steps"]
    s0 = _warm_state(L, B, H, N, cfg["warm_tokens"], seed=2001 + B, dev=dev)
    state = s0.to(dev)
    pool = inputs.draw_rwkkva((L, P, B, H, N), seed=1001 + B, device=dev)
    g = np.random.default_rng(B)
    n_samp = 64
    sl, sb, sh = g.integers(0, L, n_samp), g.integers(0, B, n_samp), g.integers(0, H, n_samp)
    sl_t, sb_t, sh_t = (torch.from_numpy(x).to(dev) for x in (sl, sb, sh))
    o_step = torch.empty(L, B, H, N, device=dev)
    o_first = torch.empty(8, L, B, H, N, device=dev)
    o_samp = torch.empty(steps, n_samp, N, device=dev)
    for s in range(steps):
        for layer in range(L):
            _step({n: pool[n][layer, s % P] for n in NAMES}, state[layer], o_step[layer])
        if s < 8:
            o_first[s] = o_step
        o_samp[s] = o_step[sl_t, sb_t, sh_t]
        if s == 7:
            state8 = state.clone()
    wkv7.check_device_status()

    # steps 1-8, every slab: sequences = (layer, b), 8 tokens each
    packed = {n: pool[n][:, :8].permute(0, 2, 1, 3, 4).reshape(L * B * 8, H, N) for n in NAMES}
    cu = np.arange(L * B + 1, dtype=np.int64) * 8
    o_ref, s_ref = oracle.run(*(host_f32(packed[n]) for n in NAMES), cu_seqlens=cu,
                              s0=s0.double().reshape(L * B, H, N, N).numpy())
    o_ref = o_ref.reshape(L, B, 8, H, N).transpose(2, 0, 1, 3, 4)
    assert rel_err(o_first, o_ref) <= TOL
    assert rel_err(state8.reshape(L * B, H, N, N), s_ref) <= TOL

    # all 1024 steps on the sampled slabs
    idx = torch.arange(steps, device=dev) % P
    seq = {n: pool[n][sl_t, :, sb_t, sh_t][:, idx] for n in NAMES}  # [S, steps, N]
    arrs = [host_f32(seq[n]).reshape(n_samp * steps, 1, N) for n in NAMES]
    s0s = s0.double().numpy()[sl, sb, sh].reshape(n_samp, 1, N, N)
    o_ref, s_ref = oracle.run(*arrs, cu_seqlens=np.arange(n_samp + 1, dtype=np.int64) * steps, s0=s0s)
    o_ref = o_ref.reshape(n_samp, steps, N).transpose(1, 0, 2)
    assert rel_err(o_samp, o_ref) <= TOL
    assert rel_err(state[sl_t, sb_t, sh_t], s_ref[:, 0]) <= TOL


def test_decode_7p2b_serving_batch(dev):
    """7.2B geometry at B=256: per layer, 8 steps on all 16384 heads from a
    seeded N(0, 0.1) state; on two layers, 1024 steps for 16 sampled heads."""
    cfg = inputs.DECODE_7P2B
    L, H, N, B, P = cfg["layers"], cfg["H"], cfg["N"], cfg["B"], cfg["pool"]
    g = np.random.default_rng(3)
    for layer in range(L):
        s0 = inputs.initial_state(B, H, N, seed=3000 + layer, std=cfg["state_std"], device=dev)
        pool = inputs.draw_rwkkva((P, B, H, N), seed=1003 + 17 * layer, device=dev)
        state = s0.clone()
        long_run = layer in (0, L - 1)
        steps = cfg["steps"] if long_run else 8
        o8 = torch.empty(8, B, H, N, device=dev)
        if long_run:
            sb, sh = g.integers(0, B, 16), g.integers(0, H, 16)
            sb_t, sh_t = torch.from_numpy(sb).to(dev), torch.from_numpy(sh).to(dev)
            o_samp = torch.empty(steps, 16, N, device=dev)
        o = torch.empty(B, H, N, device=dev)
        for s in range(steps):
            _step({n: pool[n][s % P] for n in NAMES}, state, o)
            if s < 8:
                o8[s] = o
            if s == 7:
                state8 = state.clone()
            if long_run:
                o_samp[s] = o[sb_t, sh_t]
        wkv7.check_device_status()
        packed = {n: pool[n][:8].transpose(0, 1).reshape(B * 8, H, N) for n in NAMES}
        o_ref, s_ref = oracle.run(*(host_f32(packed[n]) for n in NAMES),
                                  cu_seqlens=np.arange(B + 1, dtype=np.int64) * 8,
                                  s0=s0.double().cpu().numpy())
        assert rel_err(o8, o_ref.reshape(B, 8, H, N).transpose(1, 0, 2, 3)) <= TOL, layer
        assert rel_err(state8, s_ref) <= TOL, layer
        if long_run:
            idx = torch.arange(steps, device=dev) % P
            seq = {n: pool[n][:, sb_t, sh_t][idx].transpose(0, 1) for n in NAMES}  # [16, steps, N]
            arrs = [host_f32(seq[n]).reshape(16 * steps, 1, N) for n in NAMES]
            s0s = s0.double().cpu().numpy()[sb, sh].reshape(16, 1, N, N)
            o_ref, s_ref = oracle.run(*arrs, cu_seqlens=np.arange(17, dtype=np.int64) * steps, s0=s0s)
            assert rel_err(o_samp, o_ref.reshape(16, steps, N).transpose(1, 0, 2)) <= TOL
            assert rel_err(state[sb_t, sh_t], s_ref[:, 0]) <= TOL
        del pool, state, s0


def test_step_rejects_bad_arguments_on_gpu(dev):
    B, H, N = 2, 3, 64
    x = {n: torch.zeros(B, H, N, device=dev) for n in NAMES}
    state = torch.zeros(B, H, N, N, device=dev)
    with pytest.raises(wkv7.WKV7Error) as e:
        # state aliasing an input
        wkv7._lib.check(wkv7._lib.load().wkv7_step(
            B, H, N, *[wkv7._ptr(x[n]) for n in NAMES], wkv7._ptr(x["v"]), wkv7._ptr(x["r"]),
            wkv7._stream()), "aliasing")
    assert e.value.status == wkv7._lib.ERR_INVALID_ARG
    big = torch.zeros(B * H * N + 4, device=dev)
    with pytest.raises(wkv7.WKV7Error) as e:
        wkv7._lib.check(wkv7._lib.load().wkv7_step(
            B, H, N, *[wkv7._ptr(x[n]) for n in NAMES], wkv7._ptr(state),
            wkv7._ptr(big[1:]), wkv7._stream()), "misaligned o")
    assert e.value.status == wkv7._lib.ERR_ALIGNMENT


@pytest.mark.parametrize("B,H", [(24, 38), (1, 913), (8191, 1), (128, 64)],
                         ids=["912-heads", "913-heads", "8191-heads", "8192-heads"])
def test_step_either_side_of_the_large_batch_form(dev, B, H):
    """Both decode forms against the oracle, from a random state, either side of
    each switch: the register form up to one wave of it (912 heads on a GB300)
    and from 8192 heads, the shared-memory ring in between."""
    N = 64
    x = inputs.decode_inputs(B, H, N, steps=1, seed=B + H, device=dev)
    x = {n: t[0].contiguous() for n, t in x.items()}
    s0 = inputs.initial_state(B, H, N, seed=B, device=dev)
    state = s0.clone()
    o = _step(x, state)
    wkv7.check_device_status()
    o_ref, s_ref = oracle.step(*(x[n] for n in NAMES), state=s0.double().cpu())
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(state, s_ref) <= TOL
