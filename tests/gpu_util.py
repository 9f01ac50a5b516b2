"""Helpers for the GPU parity tests (CUDA path vs the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

NAMES = ("r", "w", "k", "v", "kk", "a")


def rel_err(x, ref) -> float:
    """max |x - ref| / max |ref| over one tensor (the parity metric)."""
    if isinstance(x, torch.Tensor):
        x = x.detach().double().cpu().numpy()
    if isinstance(ref, torch.Tensor):
        ref = ref.detach().double().cpu().numpy()
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = float(np.max(np.abs(ref)))
    return float(np.max(np.abs(x - ref))) / max(scale, 1e-30)


def host_f32(t: torch.Tensor) -> np.ndarray:
    """Exact fp32 host copy of a CUDA tensor (bf16 widens exactly)."""
    return t.detach().float().cpu().numpy()


def oracle_prefill(p: dict, cu, s0=None, heads=None):
    """Run the oracle on prefill inputs ``p`` (dict of [T, H, N] tensors).

    ``heads`` restricts the run to a list of head indices (the outputs then
    have H = len(heads)).  s0 is [num_seqs, H, N, N] (any float type).
    """
    sel = slice(None) if heads is None else list(heads)
    arrs = [host_f32(p[n][:, sel]) for n in NAMES]
    s0d = None
    if s0 is not None:
        s0d = s0[:, sel].detach().double().cpu().numpy() if isinstance(s0, torch.Tensor) else s0[:, sel]
    cu_np = cu.cpu().numpy().astype(np.int64) if isinstance(cu, torch.Tensor) else np.asarray(cu, np.int64)
    return oracle.run(*arrs, cu_seqlens=cu_np, s0=s0d)
