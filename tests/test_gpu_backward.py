"""Backward of the packed prefill (wkv7_prefill_backward) against the fp64 oracle.

The oracle is the token-serial reverse-mode derivative of the recurrence
(``oracle.backward``), pinned by finite differences of the forward oracle.  It
sees exactly the values the GPU sees (bf16 inputs widened exactly; d_o and the
states in fp32).

Bound: max|gpu - oracle| / max|oracle| <= 2e-3 per gradient tensor.  The
chunk summaries and the per-chunk gradients run their products on the tensor
cores with tf32 operands (each rounded to 11 significant bits, relative error
<= 2^-12) and fp32 accumulation; the two chains over the chunks are fp32.  A
gradient passes through at most four rounded products (Gram -> Y -> Z -> P ->
final), and the carried states and adjoints through one rounded transition
per chunk in a contracting chain, so the error is a few times 2^-12 of the
largest term: about 1e-3, the same order as the bf16-input forward bound.  The
measured maximum over every case below, the 2.9B and 7.2B full-size samples
included (512 chained chunks in the 32768-token sequence), is 1.08e-3 (dw);
d_initial_state stays near 5e-4.
"""
import numpy as np
import pytest
import torch

import oracle
import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import inputs
from tests.gpu_util import NAMES, host_f32, rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-3
GRADS = ("dr", "dw", "dk", "dv", "dkk", "da")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _case(lens, H, dtype, dev, seed, with_s0=True, with_dsf=True):
    p = inputs.prefill_inputs(lens, H, 64, seed=seed, device=dev, x_dtype=dtype)
    cu = p["cu_seqlens"]
    T_total, ns = int(cu[-1]), len(lens)
    d_o, dsf = inputs.upstream_gradients(T_total, ns, H, 64, seed=seed, device=dev)
    s0 = inputs.initial_state(ns, H, 64, seed=seed, device=dev) if with_s0 else None
    return p, cu, d_o, (dsf if with_dsf else None), s0


def _gpu(p, cu, d_o, dsf, s0, dev, host_cu=True):
    out = wkv7.prefill_backward(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), d_o,
                                initial_state=s0, d_final_state=dsf, cu_seqlens_host=cu if host_cu else None)
    wkv7.check_device_status()
    return out


def _oracle(p, cu, d_o, dsf, s0, heads=None):
    sel = slice(None) if heads is None else list(heads)
    arrs = [host_f32(p[n][:, sel]) for n in NAMES]
    f64 = lambda t: None if t is None else t[:, sel].detach().double().cpu().numpy()  # noqa: E731
    return oracle.backward(*arrs, f64(d_o), cu_seqlens=cu.numpy().astype(np.int64), s0=f64(s0), d_sfinal=f64(dsf))


def _compare(got, ref, heads=None):
    sel = slice(None) if heads is None else list(heads)
    errs = {}
    for name, x, y in zip(GRADS, got[:6], ref[:6]):
        errs[name] = rel_err(x[:, sel], y)
    if got[6] is not None:
        errs["ds0"] = rel_err(got[6][:, sel], ref[6])
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    print("backward errors", {k: f"{v:.2e}" for k, v in errs.items()})
    assert not bad, f"gradients off: {errs}"
    return errs


CASES = [
    ([64], 2, torch.float32),
    ([1, 63, 64, 65, 130, 0, 200], 3, torch.float32),
    ([300, 77], 4, torch.bfloat16),
    ([0, 0, 5], 2, torch.bfloat16),
    ([2048], 2, torch.float32),
    ([1, 100, 63], 1, torch.bfloat16),  # one head: the token tiles' maps are 64 wide
    ([65, 3, 128], 5, torch.float32),   # an odd head count, fp32 inputs (two boxes per tile)
]


@pytest.mark.parametrize("lens,H,dtype", CASES, ids=lambda x: str(x).replace(" ", ""))
def test_backward_matches_oracle(lens, H, dtype, dev):
    p, cu, d_o, dsf, s0 = _case(lens, H, dtype, dev, seed=2000 + sum(lens))
    got = _gpu(p, cu, d_o, dsf, s0, dev)
    _compare(got, _oracle(p, cu, d_o, dsf, s0))


def test_backward_without_states(dev):
    """No initial state and no final-state gradient (both zeros)."""
    p, cu, d_o, dsf, s0 = _case([129, 64], 2, torch.bfloat16, dev, seed=2100, with_s0=False, with_dsf=False)
    got = _gpu(p, cu, d_o, dsf, s0, dev)
    _compare(got, _oracle(p, cu, d_o, dsf, s0))


def test_backward_device_cu_seqlens_only(dev):
    """Without the host copy of cu_seqlens the chunk table is built on the device alone."""
    p, cu, d_o, dsf, s0 = _case([65, 0, 191], 2, torch.float32, dev, seed=2200)
    got = _gpu(p, cu, d_o, dsf, s0, dev, host_cu=False)
    _compare(got, _oracle(p, cu, d_o, dsf, s0))


def test_zero_length_passes_final_gradient(dev):
    p, cu, d_o, dsf, s0 = _case([0, 3], 2, torch.float32, dev, seed=2300)
    got = _gpu(p, cu, d_o, dsf, s0, dev)
    assert torch.equal(got[6][0], dsf[0])


def test_backward_is_deterministic(dev):
    p, cu, d_o, dsf, s0 = _case([300, 70], 2, torch.bfloat16, dev, seed=2400)
    a = _gpu(p, cu, d_o, dsf, s0, dev)
    b = _gpu(p, cu, d_o, dsf, s0, dev)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_full_size_2p9b_sampled(dev):
    """The 2.9B prefill workload (8 x 4096 tokens, H = 40, bf16 inputs), as the
    benchmark runs it; the oracle checks every gradient of four (sequence, head)
    pairs (heads 0 and 39 of sequences 0 and 7) and d_initial_state of those."""
    cfg = inputs.PREFILL_2P9B
    lens = [cfg["T"]] * cfg["num_seqs"]
    p, cu, d_o, dsf, s0 = _case(lens, cfg["H"], torch.bfloat16, dev, seed=inputs.CONFIG_SEEDS[2], with_s0=False)
    got = _gpu(p, cu, d_o, dsf, s0, dev)
    heads = [0, cfg["H"] - 1]
    for b in (0, cfg["num_seqs"] - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        sub = {n: p[n][t0:t1] for n in NAMES}
        cu1 = torch.tensor([0, t1 - t0], dtype=torch.int32)
        ref = _oracle(sub, cu1, d_o[t0:t1], dsf[b:b + 1], None, heads=heads)
        part = tuple(g[t0:t1] for g in got[:6]) + (got[6][b:b + 1],)
        _compare(part, ref, heads=heads)


def test_backward_full_size_7p2b_single_32768_sampled(dev):
    """The longest chain: one sequence of 32768 tokens (512 chunks), 64 heads,
    bf16 inputs, random initial states; the oracle checks heads 0 and 63."""
    cfg = inputs.VARLEN_7P2B
    p, cu, d_o, dsf, s0 = _case([cfg["single_T"]], cfg["H"], torch.bfloat16, dev, seed=inputs.CONFIG_SEEDS[4])
    got = _gpu(p, cu, d_o, dsf, s0, dev)
    heads = [0, cfg["H"] - 1]
    _compare(got, _oracle(p, cu, d_o, dsf, s0, heads=heads), heads=heads)


def test_backward_full_size_7p2b_varlen_sampled(dev):
    """16 sequences of U[1, 32768] tokens (seeded), 64 heads, bf16, random
    initial states; the oracle checks every sequence of head 17."""
    cfg = inputs.VARLEN_7P2B
    lens = inputs.seqlens_uniform(cfg["num_seqs"], cfg["lo"], cfg["hi"], seed=1004)
    p, cu, d_o, dsf, s0 = _case(lens, cfg["H"], torch.bfloat16, dev, seed=1004)
    got = _gpu(p, cu, d_o, dsf, s0, dev)
    heads = [17]
    _compare(got, _oracle(p, cu, d_o, dsf, s0, heads=heads), heads=heads)


def test_rejects_bad_arguments(dev):
    p, cu, d_o, dsf, s0 = _case([10], 1, torch.float32, dev, seed=2500)
    with pytest.raises(wkv7.WKV7Error):
        wkv7.prefill_backward(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), d_o,
                              workspace=torch.empty(16, device=dev, dtype=torch.uint8))
    grads = tuple(torch.empty_like(d_o) for _ in range(6))
    with pytest.raises(wkv7.WKV7Error):  # a gradient aliasing an input
        wkv7.prefill_backward(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), d_o,
                              grads=(p["r"],) + grads[1:])


def test_backward_concurrent_on_two_streams(dev):
    """Two backward calls with distinct workspaces and gradient buffers, issued on two
    streams so that their kernels overlap (every chunk-head's states and T travel
    through its call's workspace by bulk copies): each result is bit-identical to the
    same call run alone, and within the bound of the oracle."""
    cases = [([300, 77, 0, 129], 3, torch.bfloat16, 2700), ([2048], 2, torch.float32, 2701)]
    runs = []
    for lens, H, dtype, seed in cases:
        p, cu, d_o, dsf, s0 = _case(lens, H, dtype, dev, seed=seed)
        T_total = int(cu[-1])
        ws = torch.empty(wkv7.prefill_backward_workspace_size(len(lens), T_total, H), dtype=torch.uint8, device=dev)
        ref = wkv7.prefill_backward(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), d_o,
                                    initial_state=s0, d_final_state=dsf, workspace=ws, cu_seqlens_host=cu)
        runs.append((p, cu, d_o, dsf, s0, ws, tuple(None if g is None else g.clone() for g in ref)))
    torch.cuda.synchronize()
    wkv7.check_device_status()
    streams = [torch.cuda.Stream(device=dev) for _ in runs]
    for _ in range(3):
        outs = []
        for (p, cu, d_o, dsf, s0, ws, ref), st in zip(runs, streams):
            grads = tuple(torch.full_like(g, float("nan")) for g in ref[:6])
            st.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(st):
                got = wkv7.prefill_backward(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu.to(dev), d_o,
                                            initial_state=s0, d_final_state=dsf, grads=grads, workspace=ws,
                                            cu_seqlens_host=cu, stream=st)
            outs.append(got)
        torch.cuda.synchronize()
        wkv7.check_device_status()
        for got, run in zip(outs, runs):
            for x, y in zip(got, run[6]):
                if y is not None:
                    assert torch.equal(x, y)
    for p, cu, d_o, dsf, s0, _, ref in runs:
        _compare(ref, _oracle(p, cu, d_o, dsf, s0))
