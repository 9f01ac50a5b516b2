"""The chunk algebra the tensor-core kernels implement, written out in fp64 numpy
from its formulas and checked against the fp64 oracle over one chunk (CPU only).

Per chunk of C tokens and head, with the inclusive cumulative log-decay g, any
reference rho, R = r e^{g - rho}, Q = kk e^{g_{t-1} - rho}, K = k e^{rho - g},
Cm = c e^{rho - g} (c = kk a), the masked Grams Lc = tril_{-1}(Q Cm^T),
Lk = tril_{-1}(Q K^T), Mc = tril_0(R Cm^T), Mk = tril_0(R K^T),
T = (I + Lc)^{-1} and S0' = diag(e^{rho}) S0:

* forward (the prefill kernel's W form): W = Q S0' + Lk V, Z = T W,
  O = R S0' + Mk V - Mc Z,
  S_C = diag(e^{g_C}) S0 + diag(e^{g_C - rho}) (K^T V - Cm^T Z);
* backward (the summary pass): S_C = A S0 + F with
  A = diag(e^{g_C - rho}) (I - Cm^T T Q) diag(e^{rho}),
  F = diag(e^{g_C - rho}) (K^T - Cm^T T Lk) V, and the adjoint step
  dS0 = A^T G + E, E = diag(e^{rho}) (R^T - Q^T T^T Mc^T) dO, for a loss
  <dO, O> + <G, S_C>.

Here rho is taken at the middle of the chunk (the kernels take g_31); the
identities hold for any rho, which cancels.
"""
import numpy as np
import pytest

import oracle
from tests.oracle_pins import _close, _draw


def _chunk_terms(r, w, k, v, kk, a, rho_at):
    """The chunk's operands for one head, fp64 ([C, N] each)."""
    f = lambda x: x.astype(np.float64)  # noqa: E731
    r, w, k, v, kk, a = map(f, (r, w, k, v, kk, a))
    C, N = r.shape
    g = np.cumsum(w, axis=0)
    gprev = np.vstack([np.zeros((1, N)), g[:-1]])
    rho = g[rho_at]
    c = kk * a
    R, Q = r * np.exp(g - rho), kk * np.exp(gprev - rho)
    K, Cm = k * np.exp(rho - g), c * np.exp(rho - g)
    Lc, Lk = np.tril(Q @ Cm.T, -1), np.tril(Q @ K.T, -1)
    Mc, Mk = np.tril(R @ Cm.T), np.tril(R @ K.T)
    T = np.linalg.inv(np.eye(C) + Lc)
    return dict(g=g, rho=rho, R=R, Q=Q, K=K, Cm=Cm, Lc=Lc, Lk=Lk, Mc=Mc, Mk=Mk, T=T, v=v)


@pytest.mark.parametrize("C,N,seed", [(64, 16, 41), (37, 8, 42), (16, 64, 43)])
def test_forward_chunk_formulas(oracle_lib, C, N, seed):
    H = 1
    x = _draw(C, H, N, seed=seed)
    s0 = np.random.default_rng(seed + 7).standard_normal((1, H, N, N))
    o_ref, s_ref = oracle.run(*x, s0=s0, nthreads=1, lib=oracle_lib)
    m = _chunk_terms(*(y[:, 0] for y in x), rho_at=C // 2)
    S0 = s0[0, 0]
    S0p = np.exp(m["rho"])[:, None] * S0
    W = m["Q"] @ S0p + m["Lk"] @ m["v"]
    Z = m["T"] @ W
    O = m["R"] @ S0p + m["Mk"] @ m["v"] - m["Mc"] @ Z
    gC = m["g"][-1]
    SC = np.exp(gC)[:, None] * S0 + np.exp(gC - m["rho"])[:, None] * (m["K"].T @ m["v"] - m["Cm"].T @ Z)
    _close(O, o_ref[:, 0], 1e-10, "O")
    _close(SC, s_ref[0, 0], 1e-10, "S_C")


@pytest.mark.parametrize("C,N,seed", [(64, 16, 44), (29, 8, 45)])
def test_backward_chunk_summaries(oracle_lib, C, N, seed):
    H = 1
    x = _draw(C, H, N, seed=seed)
    g_ = np.random.default_rng(seed + 9)
    s0 = g_.standard_normal((1, H, N, N))
    d_o = g_.standard_normal((C, H, N))
    G = g_.standard_normal((1, H, N, N))
    m = _chunk_terms(*(y[:, 0] for y in x), rho_at=C // 2)
    eg = np.exp(m["g"][-1] - m["rho"])[:, None]
    A = eg * (np.eye(N) - m["Cm"].T @ m["T"] @ m["Q"]) * np.exp(m["rho"])[None, :]
    F = eg * ((m["K"].T - m["Cm"].T @ m["T"] @ m["Lk"]) @ m["v"])
    E = np.exp(m["rho"])[:, None] * ((m["R"].T - m["Q"].T @ m["T"].T @ m["Mc"].T) @ d_o[:, 0])
    _, s_ref = oracle.run(*x, s0=s0, nthreads=1, lib=oracle_lib)
    _close(A @ s0[0, 0] + F, s_ref[0, 0], 1e-10, "S_C = A S0 + F")
    # the adjoint step: dS0 of <dO, O> + <G, S_C> is A^T G + E
    grads = oracle.backward(*x, d_o, s0=s0, d_sfinal=G, nthreads=1, lib=oracle_lib)
    _close(grads[6][0, 0], A.T @ G[0, 0] + E, 1e-10, "dS0 = A^T G + E")
    grads0 = oracle.backward(*x, d_o, s0=s0, nthreads=1, lib=oracle_lib)
    _close(grads0[6][0, 0], E, 1e-10, "dS0 = E without a final-state gradient")
