"""The linear decomposition that the prefill's tail split and the backward's chunk
chains are built on, checked on the fp64 oracle (CPU only).

The recurrence is affine in the state: over a segment of tokens, started from
S_in,
    S_end = P S_in + S_part,      o_t = o_part_t + S_in^T (P_t^T r_t),
where (o_part, S_part) is the run of the same tokens from S = 0, and P_t (the
product of the per-token transitions diag(e^w) - (kk a) kk^T up to token t) is
the state of the run from S = I with v = 0, whose outputs are P_t^T r_t.  The
split prefill runs later segments from 0 and from I and corrects them with the
true S_in; the backward's chains compose per-chunk transitions the same way
(S_C = A S0 + F).  Chaining the decomposition over several segments gives the
whole run back.
"""
import numpy as np
import pytest

import oracle
from tests.oracle_pins import _close, _draw


def _run(lib, x, s0):
    return oracle.run(*x, s0=s0, nthreads=2, lib=lib)


@pytest.mark.parametrize("T,H,N,seed", [(37, 2, 8, 31), (64, 3, 16, 32), (5, 1, 4, 33)])
def test_segment_decomposition(oracle_lib, T, H, N, seed):
    x = _draw(T, H, N, seed=seed)
    r, w, k, v, kk, a = x
    s_in = np.random.default_rng(seed + 100).standard_normal((1, H, N, N))
    o, s = _run(oracle_lib, x, s_in)
    o_part, s_part = _run(oracle_lib, x, np.zeros((1, H, N, N)))
    eye = np.broadcast_to(np.eye(N), (1, H, N, N)).copy()
    o_tr, p = _run(oracle_lib, (r, w, k, np.zeros_like(v), kk, a), eye)
    # S_end = P S_in + S_part (per head: P acts on the key dimension)
    _close(s[0], np.einsum("hij,hjv->hiv", p[0], s_in[0]) + s_part[0], 1e-12, "S_end")
    # o_t = o_part_t + S_in^T (P_t^T r_t)
    _close(o, o_part + np.einsum("hjv,thj->thv", s_in[0], o_tr), 1e-12, "o")


def test_chained_segments_give_the_whole_run(oracle_lib):
    """Cut a sequence into segments; run every segment from 0 and from I (v = 0);
    chain S_in(j+1) = P(j) S_in(j) + S_part(j) and correct each segment's outputs:
    the result equals one run over the whole sequence."""
    T, H, N = 50, 2, 8
    x = _draw(T, H, N, seed=34)
    r, w, k, v, kk, a = x
    s0 = np.random.default_rng(35).standard_normal((1, H, N, N))
    o_whole, s_whole = _run(oracle_lib, x, s0)
    cuts = [0, 13, 14, 31, 50]
    eye = np.broadcast_to(np.eye(N), (1, H, N, N)).copy()
    s_in = s0[0]
    outs = []
    for j in range(len(cuts) - 1):
        sl = slice(cuts[j], cuts[j + 1])
        seg = tuple(y[sl] for y in x)
        o_part, s_part = _run(oracle_lib, seg, np.zeros((1, H, N, N)))
        o_tr, p = _run(oracle_lib, (seg[0], seg[1], seg[2], np.zeros_like(seg[3]), seg[4], seg[5]), eye)
        outs.append(o_part + np.einsum("hjv,thj->thv", s_in, o_tr))
        s_in = np.einsum("hij,hjv->hiv", p[0], s_in) + s_part[0]
    _close(np.concatenate(outs), o_whole, 1e-12, "chained o")
    _close(s_in, s_whole[0], 1e-12, "chained S_end")
