"""Seeded synthetic inputs for the WKV-7 recurrence.

This module only draws random tensors; it holds none of the recurrence's
arithmetic, so both the CUDA path's tests and the oracle can take their inputs
from it.

Distributions (one per input, drawn in the order r, z, k, v, kk, a):

* r, k, v ~ N(0, 1), with k scaled by 1/sqrt(N);
* log-decay w = -0.606531 * sigmoid(z), z ~ N(0, 1), so exp(w) lies in
  (exp(-0.606531), 1) -- the range an RWKV-7 model's decay takes;
* kk ~ N(0, 1), L2-normalised over the N channels of each (token, head);
* a = sigmoid(N(0, 1)).

Head geometries follow the RWKV-7 models the pages name: 0.1B = 12 heads,
2.9B = 40 heads, 7.2B = 64 heads, all with head size N = 64.

Tensors are drawn with a ``torch.Generator`` on the requested device, so
large workloads are generated where they are used; a given (seed, device)
always yields the same values.
"""
from __future__ import annotations

import math

import torch

W_SCALE = 0.606531  # exp(-0.5): the bound of an RWKV-7 log-decay

# Named workloads (shapes only).
CONFIG_SEEDS = {0: 1000, 1: 1001, 2: 1002, 3: 1003, 4: 1004}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def draw_rwkkva(shape, seed: int, device="cpu", x_dtype=torch.float32, g=None):
    """Draw r, w, k, v, kk, a of ``shape`` (..., N); w always fp32.

    Returns a dict of tensors.  ``x_dtype`` (fp32 or bf16) applies to
    r, k, v, kk, a; the values are drawn in fp32 and then stored in x_dtype.
    """
    device = torch.device(device)
    g = g or _gen(seed, device)
    N = shape[-1]
    r = _normal(shape, g, device)
    z = _normal(shape, g, device)
    k = _normal(shape, g, device) * (1.0 / math.sqrt(N))
    v = _normal(shape, g, device)
    kk = _normal(shape, g, device)
    kk = kk / kk.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    a = torch.sigmoid(_normal(shape, g, device))
    w = -W_SCALE * torch.sigmoid(z)
    out = {"r": r, "w": w, "k": k, "v": v, "kk": kk, "a": a}
    if x_dtype != torch.float32:
        for name in ("r", "k", "v", "kk", "a"):
            out[name] = out[name].to(x_dtype)
    return out


def initial_state(num: int, H: int, N: int, seed: int, std: float = 0.1, device="cpu"):
    """Seeded N(0, std) fp32 state [num, H, N, N]."""
    device = torch.device(device)
    g = _gen(seed + 7919, device)
    return _normal((num, H, N, N), g, device) * std


def decode_inputs(B: int, H: int, N: int = 64, steps: int = 1, seed: int = 1001, device="cpu"):
    """Per-step decode inputs: dict of fp32 tensors [steps, B, H, N]."""
    return draw_rwkkva((steps, B, H, N), seed, device)


def seqlens_uniform(num: int, lo: int, hi: int, seed: int):
    """``num`` sequence lengths drawn uniformly from [lo, hi] (CPU generator)."""
    g = _gen(seed + 104729, "cpu")
    return torch.randint(lo, hi + 1, (num,), generator=g).tolist()


def cu_seqlens_of(seqlens) -> torch.Tensor:
    cu = [0]
    for n in seqlens:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def prefill_inputs(seqlens, H: int, N: int = 64, seed: int = 1002, device="cpu",
                   x_dtype=torch.bfloat16):
    """Packed varlen prefill inputs.

    Returns a dict with r, w, k, v, kk, a of shape [T_total, H, N] (x_dtype for
    r, k, v, kk, a; fp32 for w) and ``cu_seqlens`` (int32 [num_seqs + 1], CPU).
    """
    cu = cu_seqlens_of(seqlens)
    T_total = int(cu[-1])
    out = draw_rwkkva((T_total, H, N), seed, device, x_dtype=x_dtype)
    out["cu_seqlens"] = cu
    return out


def upstream_gradients(T_total: int, num_seqs: int, H: int, N: int = 64, seed: int = 1005, device="cpu",
                       state_std: float = 0.1):
    """Seeded upstream gradients for a prefill backward: d_o ~ N(0, 1) fp32
    [T_total, H, N] and d_final_state ~ N(0, state_std) fp32 [num_seqs, H, N, N]."""
    device = torch.device(device)
    g = _gen(seed + 15485863, device)
    d_o = _normal((T_total, H, N), g, device)
    d_sf = _normal((num_seqs, H, N, N), g, device) * state_std
    return d_o, d_sf


# Workload shapes of the five named configurations.
DECODE_2P9B = dict(layers=32, H=40, N=64, batches=(1, 8, 32), warm_tokens=256, pool=16, steps=1024)
PREFILL_2P9B = dict(num_seqs=8, T=4096, H=40, N=64)
DECODE_7P2B = dict(layers=32, H=64, N=64, B=256, pool=16, steps=1024, state_std=0.1)
VARLEN_7P2B = dict(num_seqs=16, lo=1, hi=32768, H=64, N=64, single_T=32768, state_std=0.1)
SMALL_0P1B = dict(B=1, T=64, H=12, N=64)
