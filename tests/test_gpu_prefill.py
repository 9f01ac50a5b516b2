"""Packed varlen prefill (wkv7_prefill) against the fp64 oracle.

Bound: max|gpu - oracle| / max|oracle| <= 2e-3 for o and for the final state
with bf16 inputs (the chunked tensor-core kernel: tf32 operands), and <= 1e-5
with fp32 inputs, which take the token-serial kernel (the decode step's fp32
arithmetic run over the tokens; the fp32 decode bound).  The oracle consumes
exactly the values the GPU sees (bf16 inputs widened to fp32 exactly).
"""
import numpy as np
import pytest
import torch

import oracle
import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import inputs
from tests.gpu_util import NAMES, host_f32, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-3
TOL_FP32 = 1e-5


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _run(p, dev, s0=None, final=None, want_final=True, host_cu=True):
    cu = p["cu_seqlens"]
    o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev),
                         initial_state=s0, final_state=final, want_final_state=want_final,
                         cu_seqlens_host=cu if host_cu else None)
    wkv7.check_device_status()
    return o, sf


def _check(p, o, sf, s0=None, heads=None):
    o_ref, s_ref = oracle_prefill(p, p["cu_seqlens"], s0=s0, heads=heads)
    sel = slice(None) if heads is None else list(heads)
    e_o = rel_err(o[:, sel], o_ref)
    e_s = rel_err(sf[:, sel], s_ref) if sf is not None else 0.0
    tol = TOL_FP32 if p["r"].dtype == torch.float32 else TOL
    assert e_o <= tol and e_s <= tol, f"o {e_o:.3e}, state {e_s:.3e} (bound {tol:.0e})"
    return e_o, e_s


def test_small_0p1b_fp32_inputs(dev):
    cfg = inputs.SMALL_0P1B
    p = inputs.prefill_inputs([cfg["T"]], cfg["H"], cfg["N"], seed=1000, device=dev, x_dtype=torch.float32)
    o, sf = _run(p, dev)
    _check(p, o, sf)


EDGE_LENGTHS = [[1], [63], [64], [65], [128], [192], [130, 3, 191], [1, 63, 64, 65, 0, 127, 200], [0, 0, 5], [0],
                [3, 0]]


@pytest.mark.parametrize("lens", EDGE_LENGTHS, ids=lambda x: "-".join(map(str, x)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("with_s0", [False, True], ids=["zero_s0", "s0"])
def test_varlen_edges(dev, lens, dtype, with_s0):
    H, N = 3, 64
    p = inputs.prefill_inputs(lens, H, N, seed=len(lens) * 31 + sum(lens), device=dev, x_dtype=dtype)
    s0 = inputs.initial_state(len(lens), H, N, seed=9, device=dev) if with_s0 else None
    o, sf = _run(p, dev, s0=s0)
    _check(p, o, sf, s0=s0)
    # a zero-length sequence returns its initial state exactly
    for b, n in enumerate(lens):
        if n == 0:
            ref = s0[b] if s0 is not None else torch.zeros_like(sf[b])
            assert torch.equal(sf[b], ref)


def test_many_short_sequences(dev):
    """Hundreds of short sequences (seeded lengths 1..200, several waves of pairs, most
    chunks partial) with initial states, against the oracle."""
    lens = inputs.seqlens_uniform(300, 1, 200, seed=31)
    p = inputs.prefill_inputs(lens, 2, 64, seed=31, device=dev)
    s0 = inputs.initial_state(len(lens), 2, 64, seed=31, device=dev)
    o, sf = _run(p, dev, s0=s0)
    _check(p, o, sf, s0=s0)


def test_no_host_cu_seqlens(dev):
    p = inputs.prefill_inputs([5, 70, 0, 33], 4, 64, seed=3, device=dev)
    s0 = inputs.initial_state(4, 4, 64, seed=3, device=dev)
    o, sf = _run(p, dev, s0=s0, host_cu=False)
    _check(p, o, sf, s0=s0)


def test_null_initial_state_equals_zeros(dev):
    p = inputs.prefill_inputs([40, 90], 2, 64, seed=4, device=dev)
    o1, s1 = _run(p, dev)
    o2, s2 = _run(p, dev, s0=torch.zeros(2, 2, 64, 64, device=dev))
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_in_place_state_carry(dev):
    p = inputs.prefill_inputs([77, 13, 130], 2, 64, seed=5, device=dev)
    s0 = inputs.initial_state(3, 2, 64, seed=5, device=dev)
    buf = s0.clone()
    o, sf = _run(p, dev, s0=buf, final=buf)
    assert sf.data_ptr() == buf.data_ptr()
    _check(p, o, buf, s0=s0)


def test_final_state_not_requested(dev):
    p = inputs.prefill_inputs([100], 2, 64, seed=6, device=dev)
    o, sf = _run(p, dev, want_final=False)
    assert sf is None
    _check(p, o, None)


def test_split_resume_equals_whole(dev):
    """Prefill [0, T1) then [T1, T) from the carried state equals one prefill."""
    T, T1, H = 300, 130, 3
    p = inputs.prefill_inputs([T], H, 64, seed=7, device=dev)
    o, sf = _run(p, dev)
    pa = {n: p[n][:T1].contiguous() for n in NAMES}
    pa["cu_seqlens"] = torch.tensor([0, T1], dtype=torch.int32)
    pb = {n: p[n][T1:].contiguous() for n in NAMES}
    pb["cu_seqlens"] = torch.tensor([0, T - T1], dtype=torch.int32)
    oa, sa = _run(pa, dev)
    ob, sb = _run(pb, dev, s0=sa)
    o_ref, s_ref = oracle_prefill(p, p["cu_seqlens"])
    assert rel_err(torch.cat([oa, ob]), o_ref) <= TOL
    assert rel_err(sb, s_ref) <= TOL
    assert rel_err(torch.cat([oa, ob]), o) <= TOL


def test_degenerate_inputs(dev):
    """a = 1 with unit kk and w = 0 on one sequence (the projector); log-decay at
    its bound -0.606531 on every token of another."""
    H = 2
    p = inputs.prefill_inputs([96, 96], H, 64, seed=8, device=dev)
    p["a"][:96] = 1.0
    p["w"][:96] = 0.0
    p["w"][96:] = -0.606531
    s0 = inputs.initial_state(2, H, 64, seed=8, device=dev)
    o, sf = _run(p, dev, s0=s0)
    _check(p, o, sf, s0=s0)


def test_prefill_2p9b(dev):
    """2.9B geometry: 8 x 4096 tokens, 40 heads, bf16 inputs, zero state."""
    cfg = inputs.PREFILL_2P9B
    p = inputs.prefill_inputs([cfg["T"]] * cfg["num_seqs"], cfg["H"], cfg["N"], seed=1002, device=dev)
    o, sf = _run(p, dev)
    _check(p, o, sf)


def test_prefill_7p2b_varlen(dev):
    """7.2B geometry: 16 sequences of U[1, 32768] tokens, 64 heads, bf16, random
    initial states; every head checked, 16 heads per oracle call."""
    cfg = inputs.VARLEN_7P2B
    lens = inputs.seqlens_uniform(cfg["num_seqs"], cfg["lo"], cfg["hi"], seed=1004)
    H, N = cfg["H"], cfg["N"]
    p = inputs.prefill_inputs(lens, H, N, seed=1004, device=dev)
    s0 = inputs.initial_state(len(lens), H, N, seed=1004, std=cfg["state_std"], device=dev)
    o, sf = _run(p, dev, s0=s0)
    for h0 in range(0, H, 16):
        _check(p, o, sf, s0=s0, heads=range(h0, h0 + 16))


def test_prefill_7p2b_single_32768(dev):
    cfg = inputs.VARLEN_7P2B
    H, N = cfg["H"], cfg["N"]
    p = inputs.prefill_inputs([cfg["single_T"]], H, N, seed=1005, device=dev)
    s0 = inputs.initial_state(1, H, N, seed=1005, std=cfg["state_std"], device=dev)
    o, sf = _run(p, dev, s0=s0)
    for h0 in range(0, H, 32):
        _check(p, o, sf, s0=s0, heads=range(h0, h0 + 32))


# Tail split: with P (sequence, head) pairs on S SMs, the last r = P mod S pairs are
# cut into segments when 0 < r <= S/2 (and r <= 80), k of them with a first segment
# of a chosen length (the host's list schedule).  These shapes split on a GB300
# (S = 152): one ragged sequence of 8 heads (10 equal segments per pair), three
# unequal sequences of 10 heads (the schedule's longest-first order), one sequence of
# 64 heads and two unequal sequences of 30 heads (more items than SMs: a longer first
# segment, the short items in rounds).
SPLIT_CASES = [([3000], 8, 21), ([2000, 1500, 700], 10, 22), ([2500], 64, 24), ([1500, 900], 30, 25)]
SPLIT_IDS = ["1x3000-H8", "unequal-H10", "1x2500-H64-rounds", "unequal-H30-rounds"]


def _expect_split(num_seqs, H):
    S = torch.cuda.get_device_properties(0).multi_processor_count
    r = (num_seqs * H) % S
    return 0 < r and 2 * r <= S and r <= 80


@pytest.mark.parametrize("lens,H,seed", SPLIT_CASES, ids=SPLIT_IDS)
def test_tail_split_against_oracle(dev, lens, H, seed):
    p = inputs.prefill_inputs(lens, H, 64, seed=seed, device=dev)
    s0 = inputs.initial_state(len(lens), H, 64, seed=seed, device=dev)
    cu = p["cu_seqlens"]
    need = wkv7.prefill_workspace_size(len(lens), cu[-1].item(), H)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)
    o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                         cu_seqlens_host=cu, workspace=ws)
    wkv7.check_device_status()
    _check(p, o, sf, s0=s0)
    # the split scratch (after the 256-byte-rounded sequence order) holds boundary states iff it ran
    head = 0 if len(lens) < 2 else 256
    touched = bool((ws[head:head + 16384] != 0xFF).any())
    assert touched == _expect_split(len(lens), H)


@pytest.mark.parametrize("lens,H,seed", SPLIT_CASES, ids=SPLIT_IDS)
def test_tail_split_matches_whole_pairs(dev, lens, H, seed):
    """The same batch with a workspace that only holds the sequence order, so every
    pair runs whole: both schedules agree within the prefill bound."""
    p = inputs.prefill_inputs(lens, H, 64, seed=seed, device=dev)
    s0 = inputs.initial_state(len(lens), H, 64, seed=seed, device=dev)
    o1, s1 = _run(p, dev, s0=s0)
    cu = p["cu_seqlens"]
    small = torch.empty(256, dtype=torch.uint8, device=dev)
    o2, s2 = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                          cu_seqlens_host=cu, workspace=small)
    wkv7.check_device_status()
    assert rel_err(o1, o2) <= TOL
    assert rel_err(s1, s2) <= TOL


def test_tail_split_in_place_state(dev):
    lens, H = [3000], 8
    p = inputs.prefill_inputs(lens, H, 64, seed=23, device=dev)
    s0 = inputs.initial_state(1, H, 64, seed=23, device=dev)
    s = s0.clone()
    o, sf = _run(p, dev, s0=s, final=s)
    assert sf.data_ptr() == s.data_ptr()
    _check(p, o, sf, s0=s0)


def _step_loop(p, s0):
    state = s0.clone()
    outs = []
    for t in range(p["r"].shape[0]):
        outs.append(wkv7.step(*(p[n][t:t + 1].float().contiguous() for n in NAMES), state).clone())
    return torch.cat(outs), state


def test_step_and_prefill_agree(dev):
    """The recurrent path (wkv7_step token by token) and the token-serial
    prefill agree within the fp32 bound on the same fp32 inputs."""
    T, H, N = 200, 4, 64
    p = inputs.prefill_inputs([T], H, N, seed=10, device=dev, x_dtype=torch.float32)
    s0 = inputs.initial_state(1, H, N, seed=10, device=dev)
    o_p, s_p = _run(p, dev, s0=s0)
    o_s, state = _step_loop(p, s0)
    assert rel_err(o_p, o_s) <= TOL_FP32
    assert rel_err(s_p, state) <= TOL_FP32


def test_step_and_chunked_prefill_agree(dev):
    """The recurrent path (wkv7_step on the bf16 inputs widened to fp32) and the
    chunked tensor-core prefill agree within the bf16-input prefill bound, over
    several chunks and a ragged tail."""
    T, H, N = 333, 4, 64
    p = inputs.prefill_inputs([T], H, N, seed=12, device=dev, x_dtype=torch.bfloat16)
    s0 = inputs.initial_state(1, H, N, seed=12, device=dev)
    o_p, s_p = _run(p, dev, s0=s0)
    o_s, state = _step_loop(p, s0)
    assert rel_err(o_p, o_s) <= TOL
    assert rel_err(s_p, state) <= TOL


def test_device_detects_malformed_cu_seqlens(dev):
    """Without a host copy the device validates cu_seqlens and reports through
    the status word; no out-of-range index is ever used."""
    H, N, T = 2, 64, 10
    p = inputs.prefill_inputs([T], H, N, seed=11, device=dev)
    for bad in ([0, 5, 3, 10], [0, 4, 12, 10]):
        cu = torch.tensor(bad, dtype=torch.int32, device=dev)
        with pytest.raises(wkv7.WKV7Error) as e:
            wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu)
            wkv7.check_device_status()
        assert e.value.status == wkv7._lib.ERR_INVALID_ARG
    # the status word was cleared: a good call afterwards reports OK
    o, sf = _run(p, dev)
    _check(p, o, sf)


def test_host_rejects_malformed_cu_seqlens(dev):
    p = inputs.prefill_inputs([10], 2, 64, seed=12, device=dev)
    bad = torch.tensor([0, 6, 4, 10], dtype=torch.int32)
    with pytest.raises(wkv7.WKV7Error) as e:
        wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], bad.to(dev), cu_seqlens_host=bad)
    assert e.value.status == wkv7._lib.ERR_INVALID_ARG


def test_concurrent_calls_on_two_streams(dev):
    """Two calls with distinct workspaces, outputs and states, issued on two streams
    so that they overlap on the GPU (one of them tail-split, so its fix-up kernels and
    scratch are in flight too): each result is bit-identical to the same call run
    alone (the kernels are deterministic), and within the bound of the oracle."""
    cases = [([3000], 8, 91), ([64, 101, 0, 7, 700], 3, 92)]
    runs = []
    for lens, H, seed in cases:
        p = inputs.prefill_inputs(lens, H, 64, seed=seed, device=dev)
        s0 = inputs.initial_state(len(lens), H, 64, seed=seed, device=dev)
        cu = p["cu_seqlens"]
        ws = torch.empty(max(wkv7.prefill_workspace_size(len(lens), int(cu[-1]), H), 16), dtype=torch.uint8,
                         device=dev)
        o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                             cu_seqlens_host=cu, workspace=ws)
        runs.append((p, s0, cu, ws, o.clone(), sf.clone()))
    torch.cuda.synchronize()
    wkv7.check_device_status()
    streams = [torch.cuda.Stream(device=dev) for _ in runs]
    for _ in range(4):
        outs = []
        for (p, s0, cu, ws, o_ref, sf_ref), st in zip(runs, streams):
            o = torch.full_like(o_ref, float("nan"))
            sf = torch.full_like(sf_ref, float("nan"))
            st.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(st):
                wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                             final_state=sf, o=o, cu_seqlens_host=cu, workspace=ws, stream=st)
            outs.append((o, sf))
        torch.cuda.synchronize()
        wkv7.check_device_status()
        for (o, sf), (_, _, _, _, o_ref, sf_ref) in zip(outs, runs):
            assert torch.equal(o, o_ref)
            assert torch.equal(sf, sf_ref)
    for p, s0, cu, _, o_ref, sf_ref in runs:
        _check(p, o_ref, sf_ref, s0=s0)


# Randomised schedules: batches whose last wave of pairs is split in many different
# ways (equal segments, a longer first segment with the short items in rounds, pairs
# too short to split beside long ones), each checked on sampled heads against the
# oracle and against the same call with every pair whole.  Heads H - 1 and H - 2
# belong to the last sequence in the schedule, whose pairs form the tail.
RANDOM_SCHEDULES = [
    (1, 8, 9001), (1, 40, 9002), (1, 64, 9003), (2, 30, 9004), (2, 38, 9005), (3, 13, 9006),
    (3, 25, 9007), (4, 19, 9008), (5, 7, 9009), (6, 12, 9010), (1, 76, 9011), (2, 76, 9012),
]


@pytest.mark.parametrize("num_seqs,H,seed", RANDOM_SCHEDULES, ids=lambda x: str(x))
def test_random_split_schedules(dev, num_seqs, H, seed):
    g = torch.Generator().manual_seed(seed)
    lens = (torch.randint(3, 5000, (num_seqs,), generator=g)).tolist()
    if sum(lens) < 1024:  # the split needs at least 1024 tokens of scratch
        lens[0] += 1024
    p = inputs.prefill_inputs(lens, H, 64, seed=seed, device=dev)
    s0 = inputs.initial_state(num_seqs, H, 64, seed=seed, device=dev)
    cu = p["cu_seqlens"]
    o, sf = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                         cu_seqlens_host=cu)
    small = torch.empty(max(256, wkv7.prefill_workspace_size(num_seqs, 0, H)), dtype=torch.uint8, device=dev)
    o_w, sf_w = wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), initial_state=s0,
                             cu_seqlens_host=cu, workspace=small)
    wkv7.check_device_status()
    assert rel_err(o, o_w) <= TOL and rel_err(sf, sf_w) <= TOL
    heads = sorted({0, H - 2, H - 1})
    o_ref, s_ref = oracle_prefill(p, cu, s0=s0, heads=heads)
    e_o, e_s = rel_err(o[:, heads], o_ref), rel_err(sf[:, heads], s_ref)
    assert e_o <= TOL and e_s <= TOL, f"o {e_o:.3e}, state {e_s:.3e}"
