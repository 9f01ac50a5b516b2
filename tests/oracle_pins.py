"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle.

Each pin takes a loaded oracle library (ctypes) and raises AssertionError when
the oracle disagrees with an independent statement of what the recurrence
must give.  The pins are written so that each plausible slip in the oracle --
a dropped term, a sign, an index, a transposed operand, the decay or the delta
taken on the wrong state, a missed reset -- fails at least one of them; the
mutation test compiles such slips into copies of the oracle and checks that.

The recurrence (per head, S = [K, V]; Core AI model zoo note "Recurrent /
linear-attention LLMs on Core AI", section 1):
    z = kk^T S_old ;  S = diag(exp w) S_old - (kk*a) z^T + k v^T ;  o = S^T r
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def _draw(T, H, N, seed, a_zero=False, w_zero=False):
    """Random inputs [T, H, N] as exact fp32 values (float64 views for math)."""
    g = _rng(seed)
    r = _f32(g.standard_normal((T, H, N)))
    w = _f32(-0.606531 / (1.0 + np.exp(-g.standard_normal((T, H, N)))))
    k = _f32(g.standard_normal((T, H, N)) / math.sqrt(N))
    v = _f32(g.standard_normal((T, H, N)))
    kk = g.standard_normal((T, H, N))
    kk = _f32(kk / np.linalg.norm(kk, axis=-1, keepdims=True))
    a = _f32(1.0 / (1.0 + np.exp(-g.standard_normal((T, H, N)))))
    if a_zero:
        a = np.zeros_like(a)
    if w_zero:
        w = np.zeros_like(w)
    return r, w, k, v, kk, a


def _run(lib, r, w, k, v, kk, a, cu=None, s0=None):
    return oracle.run(r, w, k, v, kk, a, cu_seqlens=cu, s0=s0, nthreads=2, lib=lib)


def _close(x, y, tol, what):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(y))) if y.size else 1.0)
    err = float(np.max(np.abs(x - y))) if x.size else 0.0
    assert err <= tol * scale, f"{what}: max|diff| {err:.3e} > {tol:.1e} * {scale:.3e}"


# --------------------------------------------------------------------------
# (a) small cases by hand


def pin_golden_hand_n2(lib):
    """N = 2, T = 3 worked by hand (tests/golden/wkv7_n2_t3_hand.txt)."""
    rows = {}
    tol = None
    with open(os.path.join(GOLDEN, "wkv7_n2_t3_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "tol":
                tol = float(parts[1])
                continue
            rows[(parts[0], int(parts[1]))] = [float(x) for x in parts[2:]]
    T, N = 3, 2

    def seq(name):
        return _f32([rows[(name, t)] for t in range(1, T + 1)]).reshape(T, 1, N)

    w = _f32(np.log(np.asarray([rows[("decay", t)] for t in range(1, T + 1)]))).reshape(T, 1, N)
    o, s = _run(lib, seq("r"), w, seq("k"), seq("v"), seq("kk"), seq("a"))
    exp_o = np.asarray([rows[("o", t)] for t in range(1, T + 1)]).reshape(T, 1, N)
    exp_s = np.asarray(rows[("S", 3)]).reshape(1, 1, N, N)
    _close(o, exp_o, tol, "golden o")
    _close(s, exp_s, tol, "golden S")


def pin_t1_zero_state(lib):
    """T = 1 from S0 = 0: S1 = k v^T (decay and delta act on zero), o1 = (r.k) v."""
    r, w, k, v, kk, a = _draw(1, 3, 8, seed=11)
    o, s = _run(lib, r, w, k, v, kk, a)
    for h in range(3):
        rd, kd, vd = (x[0, h].astype(np.float64) for x in (r, k, v))
        _close(o[0, h], np.dot(rd, kd) * vd, 1e-13, "o1")
        _close(s[0, h], np.outer(kd, vd), 1e-13, "S1")


def pin_t2_zero_state(lib):
    """T = 2 from S0 = 0, expanded by hand:

    S2 = [e^{w2} * k1 - (kk2 . k1) c2] v1^T + k2 v2^T,   c2 = kk2 * a2
    o2 = (r2 . (e^{w2} * k1) - (kk2 . k1)(r2 . c2)) v1 + (r2 . k2) v2
    """
    r, w, k, v, kk, a = _draw(2, 2, 8, seed=12)
    o, s = _run(lib, r, w, k, v, kk, a)
    for h in range(2):
        k1, k2 = k[0, h].astype(np.float64), k[1, h].astype(np.float64)
        v1, v2 = v[0, h].astype(np.float64), v[1, h].astype(np.float64)
        r2 = r[1, h].astype(np.float64)
        kk2 = kk[1, h].astype(np.float64)
        c2 = kk2 * a[1, h].astype(np.float64)
        d2 = np.exp(w[1, h].astype(np.float64))
        s2 = np.outer(d2 * k1 - np.dot(kk2, k1) * c2, v1) + np.outer(k2, v2)
        o2 = (np.dot(r2, d2 * k1) - np.dot(kk2, k1) * np.dot(r2, c2)) * v1 + np.dot(r2, k2) * v2
        _close(s[0, h], s2, 1e-13, "S2")
        _close(o[1, h], o2, 1e-13, "o2")


# --------------------------------------------------------------------------
# (b) a = 0: decayed causal linear attention


def pin_a0_decayed_linear_attention(lib):
    """a = 0:  o_t = sum_{s<=t} r_t^T diag(prod_{s<u<=t} e^{w_u}) k_s v_s^T,
    S_T = sum_s diag(prod_{s<u<=T} e^{w_u}) k_s v_s^T (+ decayed S0)."""
    T, H, N = 9, 2, 6
    r, w, k, v, kk, a = _draw(T, H, N, seed=13, a_zero=True)
    g = _rng(14)
    s0 = g.standard_normal((1, H, N, N))
    o, s = _run(lib, r, w, k, v, kk, a, s0=s0)
    rd, wd, kd, vd = (x.astype(np.float64) for x in (r, w, k, v))
    for h in range(H):
        cum = np.concatenate([np.zeros((1, N)), np.cumsum(wd[:, h], axis=0)])  # cum[t] = sum_{u<=t} w_u (1-based)
        for t in range(T):
            acc = (rd[t, h] * np.exp(cum[t + 1])) @ s0[0, h]
            for s_ in range(t + 1):
                decay = np.exp(cum[t + 1] - cum[s_ + 1])
                acc = acc + np.dot(rd[t, h] * decay, kd[s_, h]) * vd[s_, h]
            _close(o[t, h], acc, 1e-12, f"o[{t}]")
        sT = np.exp(cum[T])[:, None] * s0[0, h]
        for s_ in range(T):
            sT = sT + np.outer(np.exp(cum[T] - cum[s_ + 1]) * kd[s_, h], vd[s_, h])
        _close(s[0, h], sT, 1e-12, "S_T")


def pin_a0_w0_causal_linear_attention(lib):
    """a = 0 and w = 0: textbook causal linear attention, O = tril(R K^T) V."""
    T, H, N = 17, 3, 5
    r, w, k, v, kk, a = _draw(T, H, N, seed=15, a_zero=True, w_zero=True)
    o, s = _run(lib, r, w, k, v, kk, a)
    for h in range(H):
        R, K, V = (x[:, h].astype(np.float64) for x in (r, k, v))
        _close(o[:, h], np.tril(R @ K.T) @ V, 1e-12, "tril(RK^T)V")
        _close(s[0, h], K.T @ V, 1e-12, "K^T V")


# --------------------------------------------------------------------------
# (c) the projector case


def pin_projector(lib):
    """w = 0, a = 1, unit kk:  S' = (I - kk kk^T) S + k v^T.

    kk is chosen with an exactly unit fp32 norm.  Checked as
    (1) kk^T (S' - k v^T) = 0, (2) the matrix form, and (3) idempotence: a
    second step with the same kk and k = v = 0 removes only the kk-component
    of k v^T, i.e. S'' = S' - kk (kk^T k) v^T.
    """
    N, H = 7, 2
    g = _rng(16)
    s0 = g.standard_normal((1, H, N, N))
    units = [np.array([0.5, 0.5, 0.5, 0.5, 0, 0, 0]), np.array([0.75, 0.5, 0.25, 0.25, 0.25, 0, 0])]
    kk = np.zeros((2, H, N), np.float32)
    for h in range(H):
        q = units[h][g.permutation(N)] * np.where(g.random(N) < 0.5, -1.0, 1.0)
        assert float(np.dot(q, q)) == 1.0
        kk[0, h] = kk[1, h] = q
    k = _f32(g.standard_normal((2, H, N)))
    v = _f32(g.standard_normal((2, H, N)))
    k[1] = 0.0
    v[1] = 0.0
    r = _f32(g.standard_normal((2, H, N)))
    w = np.zeros((2, H, N), np.float32)
    a = np.ones((2, H, N), np.float32)
    o1, s1 = _run(lib, r[:1], w[:1], k[:1], v[:1], kk[:1], a[:1], s0=s0)
    o2, s2 = _run(lib, r, w, k, v, kk, a, s0=s0)
    for h in range(H):
        q = kk[0, h].astype(np.float64)
        kv = np.outer(k[0, h].astype(np.float64), v[0, h].astype(np.float64))
        _close(q @ (s1[0, h] - kv), np.zeros(N), 1e-12, "kk^T (S' - k v^T)")
        _close(s1[0, h], (np.eye(N) - np.outer(q, q)) @ s0[0, h] + kv, 1e-12, "projector form")
        _close(s2[0, h], s1[0, h] - np.outer(q, q @ kv), 1e-12, "idempotence")
        _close(o2[1, h], s2[0, h].T @ r[1, h].astype(np.float64), 1e-12, "read-out of S''")


# --------------------------------------------------------------------------
# (d) split invariance, (e) N = 1, (f) linearity, (g) equivariance,
# (h) packing, (i) zero length


def pin_split_invariance(lib):
    """Running [0, T1) then [T1, T) with the carried state equals one run."""
    T, H, N = 23, 2, 8
    r, w, k, v, kk, a = _draw(T, H, N, seed=17)
    s0 = _rng(18).standard_normal((1, H, N, N))
    o, s = _run(lib, r, w, k, v, kk, a, s0=s0)
    for T1 in (1, 9, 22):
        oa, sa = _run(lib, *(x[:T1] for x in (r, w, k, v, kk, a)), s0=s0)
        ob, sb = _run(lib, *(x[T1:] for x in (r, w, k, v, kk, a)), s0=sa)
        _close(np.concatenate([oa, ob]), o, 1e-13, f"o split at {T1}")
        _close(sb, s, 1e-13, f"S split at {T1}")


def pin_scalar_n1(lib):
    """N = 1: a scalar first-order recurrence s' = (e^w - a kk^2) s + k v, o = r s'."""
    T = 12
    g = _rng(19)
    r, k, v = (_f32(g.standard_normal((T, 1, 1))) for _ in range(3))
    w = _f32(-0.6 * g.random((T, 1, 1)))
    kk = _f32(np.where(g.random((T, 1, 1)) < 0.5, -1.0, 1.0) * g.random((T, 1, 1)))
    a = _f32(g.random((T, 1, 1)))
    s0 = np.array([[[[0.75]]]])
    o, s = _run(lib, r, w, k, v, kk, a, s0=s0)
    # closed form: s_t = P(t,0) s0 + sum_{u<=t} P(t,u) k_u v_u with P(t,u) = prod_{u<m<=t} g_m
    gm = np.exp(w[:, 0, 0].astype(np.float64)) - a[:, 0, 0] * kk[:, 0, 0].astype(np.float64) ** 2
    for t in range(T):
        st = np.prod(gm[: t + 1]) * 0.75
        for u in range(t + 1):
            st += np.prod(gm[u + 1: t + 1]) * float(k[u, 0, 0]) * float(v[u, 0, 0])
        _close(o[t, 0, 0], float(r[t, 0, 0]) * st, 1e-13, f"o[{t}]")
        if t == T - 1:
            _close(s[0, 0, 0, 0], st, 1e-13, "s_T")


def pin_linearity(lib):
    """(o, S_T) is linear in (S0, V) jointly."""
    T, H, N = 10, 2, 6
    r, w, k, v, kk, a = _draw(T, H, N, seed=20)
    g = _rng(21)
    s0a, s0b = g.standard_normal((2, 1, H, N, N))
    # v values on a 1/64 grid, so that al*v + be*vb is exact in fp32
    v = _f32(np.round(g.standard_normal((T, H, N)) * 64) / 64)
    vb = _f32(np.round(g.standard_normal((T, H, N)) * 64) / 64)
    al, be = 0.5, -1.25
    vc = _f32(al * v.astype(np.float64) + be * vb.astype(np.float64))
    assert np.array_equal(vc.astype(np.float64), al * v.astype(np.float64) + be * vb.astype(np.float64))
    oa, sa = _run(lib, r, w, k, v, kk, a, s0=s0a)
    ob, sb = _run(lib, r, w, k, vb, kk, a, s0=s0b)
    oc, sc = _run(lib, r, w, k, vc, kk, a, s0=al * s0a + be * s0b)
    _close(oc, al * oa + be * ob, 1e-12, "o linear")
    _close(sc, al * sa + be * sb, 1e-12, "S linear")


def pin_equivariance(lib):
    """Permuting value columns permutes o and the columns of S; permuting
    heads or sequences permutes the outputs the same way."""
    T, H, N = 8, 3, 6
    r, w, k, v, kk, a = _draw(T, H, N, seed=22)
    g = _rng(23)
    s0 = g.standard_normal((1, H, N, N))
    o, s = _run(lib, r, w, k, v, kk, a, s0=s0)
    pv = g.permutation(N)
    o2, s2 = _run(lib, r, w, k, v[:, :, pv], kk, a, s0=s0[..., pv])
    _close(o2, o[:, :, pv], 0.0, "value permutation o")
    _close(s2, s[..., pv], 0.0, "value permutation S")
    ph = g.permutation(H)
    o3, s3 = _run(lib, *(x[:, ph] for x in (r, w, k, v, kk, a)), s0=s0[:, ph])
    _close(o3, o[:, ph], 0.0, "head permutation o")
    _close(s3, s[:, ph], 0.0, "head permutation S")
    # sequences: two packed sequences (3 and 5 tokens) swapped
    cu = np.array([0, 3, 8])
    s0b = g.standard_normal((2, H, N, N))
    o4, s4 = _run(lib, r, w, k, v, kk, a, cu=cu, s0=s0b)
    sw = lambda x: np.concatenate([x[3:], x[:3]])  # noqa: E731
    o5, s5 = _run(lib, *(sw(x) for x in (r, w, k, v, kk, a)), cu=np.array([0, 5, 8]), s0=s0b[::-1].copy())
    _close(o5, sw(o4), 0.0, "sequence permutation o")
    _close(s5, s4[::-1], 0.0, "sequence permutation S")


def pin_packing(lib):
    """A varlen packed run equals separate runs of each sequence."""
    H, N = 2, 8
    lens = [4, 1, 0, 11, 7]
    T = sum(lens)
    r, w, k, v, kk, a = _draw(T, H, N, seed=24)
    cu = np.concatenate([[0], np.cumsum(lens)])
    s0 = _rng(25).standard_normal((len(lens), H, N, N))
    o, s = _run(lib, r, w, k, v, kk, a, cu=cu, s0=s0)
    for b, n in enumerate(lens):
        sl = slice(cu[b], cu[b + 1])
        ob, sb = _run(lib, *(x[sl] for x in (r, w, k, v, kk, a)), s0=s0[b:b + 1])
        _close(o[sl], ob, 0.0, f"packed o seq {b}")
        _close(s[b], sb[0], 0.0, f"packed S seq {b}")


def pin_zero_length(lib):
    """A 0-token sequence returns its initial state; zeros when none given."""
    H, N = 2, 4
    r, w, k, v, kk, a = _draw(0, H, N, seed=26)
    s0 = _rng(27).standard_normal((1, H, N, N))
    o, s = _run(lib, r, w, k, v, kk, a, s0=s0)
    assert o.shape == (0, H, N)
    _close(s, s0, 0.0, "zero-length keeps S0")
    o, s = _run(lib, r, w, k, v, kk, a)
    _close(s, np.zeros_like(s0), 0.0, "zero-length zero state")


# --------------------------------------------------------------------------
# (e) the time-mix tail after WKV: y = (GroupNorm_head(o) * ln_w + ln_b
#     + (sum_i r_i k_i rk_i) v) * g   (SwiftRWKV page: "group norm, bonus, gate")


def _tail_draw(rows, H, N, seed):
    g = _rng(seed)
    o = g.standard_normal((rows, H, N))
    r, k, v, gate = (_f32(g.standard_normal((rows, H, N))) for _ in range(4))
    rk, ln_w, ln_b = (_f32(g.standard_normal((H, N))) for _ in range(3))
    return o, r, k, v, rk, ln_w, ln_b, gate


def _tail(lib, o, r, k, v, rk, ln_w, ln_b, gate, eps):
    return oracle.tail(o, r, k, v, rk, ln_w, ln_b, gate, eps, lib=lib)


def pin_tail_golden_hand_n2(lib):
    """One row, one head, N = 2, worked by hand (tests/golden/tail_n2_hand.txt)."""
    vals = {}
    for line in open(os.path.join(GOLDEN, "tail_n2_hand.txt")):
        line = line.split("#", 1)[0].split()
        if line:
            vals[line[0]] = [float(x) for x in line[1:]]
    row = lambda n: _f32(vals[n]).reshape(1, 1, 2)
    par = lambda n: _f32(vals[n]).reshape(1, 2)
    o = np.array(vals["o"], dtype=np.float64).reshape(1, 1, 2)
    for eps, want in ((0.0, "eps0"), (3.0, "eps3")):
        y = _tail(lib, o, row("r"), row("k"), row("v"), par("rk"), par("ln_w"), par("ln_b"), row("g"), eps)
        _close(y.reshape(2), vals[want], 1e-15, f"hand-worked tail, eps={eps}")


def pin_tail_standardises(lib):
    """ln_w = 1, ln_b = 0, rk = 0, g = 1, eps = 0: every (row, head) of y has mean 0 and
    mean square 1 (the group norm with the population variance)."""
    rows, H, N = 5, 3, 16
    o, r, k, v, _, _, _, _ = _tail_draw(rows, H, N, seed=40)
    ones, zeros = np.ones((H, N), np.float32), np.zeros((H, N), np.float32)
    y = _tail(lib, o, r, k, v, zeros, ones, zeros, np.ones((rows, H, N), np.float32), 0.0)
    _close(y.mean(axis=-1), np.zeros((rows, H)), 1e-13, "mean of the normalised head")
    _close((y * y).mean(axis=-1), np.ones((rows, H)), 1e-12, "mean square of the normalised head")


def pin_tail_shift_and_scale_invariance(lib):
    """With eps = 0 the tail ignores a shift and a positive scale of each head's o."""
    rows, H, N = 4, 2, 8
    o, r, k, v, rk, ln_w, ln_b, gate = _tail_draw(rows, H, N, seed=41)
    y0 = _tail(lib, o, r, k, v, rk, ln_w, ln_b, gate, 0.0)
    shift = _rng(42).standard_normal((rows, H, 1))
    y1 = _tail(lib, 2.5 * o + shift, r, k, v, rk, ln_w, ln_b, gate, 0.0)
    _close(y1, y0, 1e-12, "shift and scale of o")


def pin_tail_gate_scales_the_sum(lib):
    """y is linear in the gate: doubling g doubles every y (the gate multiplies the
    normalised part and the bonus together)."""
    rows, H, N = 3, 2, 8
    o, r, k, v, rk, ln_w, ln_b, gate = _tail_draw(rows, H, N, seed=43)
    y1 = _tail(lib, o, r, k, v, rk, ln_w, ln_b, gate, 1e-3)
    y2 = _tail(lib, o, r, k, v, rk, ln_w, ln_b, 2 * gate, 1e-3)
    _close(y2, 2 * y1, 1e-14, "gate linearity")


def pin_tail_bonus_unit_vectors(lib):
    """ln_w = ln_b = 0, g = 1: y = (sum_i r_i k_i rk_i) v.  With r = k = e_p the bonus is
    rk_p; with r = e_p, k = e_q (p != q) it is 0."""
    rows, H, N = 1, 2, 6
    o, _, _, v, rk, _, _, _ = _tail_draw(rows, H, N, seed=44)
    zeros = np.zeros((H, N), np.float32)
    ones = np.ones((rows, H, N), np.float32)
    for p, q in ((1, 1), (4, 4), (1, 4)):
        r = np.zeros((rows, H, N), np.float32)
        k = np.zeros((rows, H, N), np.float32)
        r[..., p] = 1.0
        k[..., q] = 1.0
        y = _tail(lib, o, r, k, v, rk, zeros, zeros, ones, 1e-3)
        want = (rk[:, p] if p == q else np.zeros(H)).reshape(1, H, 1) * v.astype(np.float64)
        _close(y, want, 0.0, f"bonus with r = e_{p}, k = e_{q}")


def pin_tail_constant_head(lib):
    """A head whose o is constant has zero variance: with eps > 0 its normalised part is
    0 and y = (ln_b + bonus v) g."""
    rows, H, N = 2, 2, 4
    _, r, k, v, rk, ln_w, ln_b, gate = _tail_draw(rows, H, N, seed=45)
    o = np.full((rows, H, N), 0.75)
    y = _tail(lib, o, r, k, v, rk, ln_w, ln_b, gate, 1e-2)
    zeros = np.zeros((H, N), np.float32)
    y_b = _tail(lib, np.zeros((rows, H, N)), r, k, v, rk, zeros, ln_b, gate, 1e-2)
    _close(y, y_b, 0.0, "constant head equals zero head with ln_w = 0")


def pin_tail_heads_use_their_parameters(lib):
    """Permuting heads together with their per-head parameters permutes y."""
    rows, H, N = 3, 4, 8
    o, r, k, v, rk, ln_w, ln_b, gate = _tail_draw(rows, H, N, seed=46)
    y = _tail(lib, o, r, k, v, rk, ln_w, ln_b, gate, 1e-3)
    perm = [2, 0, 3, 1]
    yp = _tail(lib, o[:, perm], r[:, perm], k[:, perm], v[:, perm], rk[perm], ln_w[perm], ln_b[perm],
               gate[:, perm], 1e-3)
    _close(yp, y[:, perm], 0.0, "head permutation")


# --------------------------------------------------------------------------
# (f) the backward: reverse-mode derivative of the recurrence for
#     L = <dO, o> + <dS_T, S_T>, pinned to the forward oracle (itself pinned
#     above) by finite differences, to a scalar closed form, to Euler's
#     identity for inputs the loss is homogeneous in, and to chaining.


def _bwd(lib, r, w, k, v, kk, a, d_o, cu=None, s0=None, dsf=None):
    return oracle.backward(r, w, k, v, kk, a, d_o, cu_seqlens=cu, s0=s0, d_sfinal=dsf, nthreads=2, lib=lib)


def _loss(lib, xs, d_o, cu, s0, dsf):
    o, s = _run(lib, *xs, cu=cu, s0=s0)
    return float(np.sum(o * d_o) + np.sum(s * dsf))


def pin_bwd_finite_differences(lib):
    """Every gradient equals the central difference of the forward loss.

    Two packed sequences (3 and 4 tokens), N = 4, random S0, dO and dS_T.  The
    step is 2^-10 on the fp32 inputs (the difference of the two rounded fp32
    points is used as the step) and 2^-10 on S0; the truncation error is
    O(step^2), far below the tolerance, and a dropped term, a sign or a
    transposed operand gives O(1) errors.
    """
    H, N = 2, 4
    cu = np.array([0, 3, 7])
    T = 7
    xs = list(_draw(T, H, N, seed=40))
    g = _rng(41)
    s0 = g.standard_normal((2, H, N, N))
    d_o = g.standard_normal((T, H, N))
    dsf = g.standard_normal((2, H, N, N))
    grads = _bwd(lib, *xs, d_o, cu=cu, s0=s0, dsf=dsf)
    h = 2.0 ** -10
    names = ["r", "w", "k", "v", "kk", "a"]
    for q, name in enumerate(names):
        fd = np.zeros((T, H, N))
        for idx in np.ndindex(T, H, N):
            x0 = xs[q][idx]
            xp = np.float32(float(x0) + h)
            xm = np.float32(float(x0) - h)
            xs[q][idx] = xp
            lp = _loss(lib, xs, d_o, cu, s0, dsf)
            xs[q][idx] = xm
            lm = _loss(lib, xs, d_o, cu, s0, dsf)
            xs[q][idx] = x0
            fd[idx] = (lp - lm) / (float(xp) - float(xm))
        _close(grads[q], fd, 1e-5, f"d{name} against finite differences")
    fd = np.zeros_like(s0)
    for idx in np.ndindex(*s0.shape):
        x0 = s0[idx]
        s0[idx] = x0 + h
        lp = _loss(lib, xs, d_o, cu, s0, dsf)
        s0[idx] = x0 - h
        lm = _loss(lib, xs, d_o, cu, s0, dsf)
        s0[idx] = x0
        fd[idx] = (lp - lm) / (2 * h)
    _close(grads[6], fd, 1e-5, "dS0 against finite differences")


def pin_bwd_scalar_n1(lib):
    """N = 1: s_t = g_t s_{t-1} + k_t v_t with g_t = e^{w_t} - a_t kk_t^2, o_t = r_t s_t.

    With the adjoint lam_t = r_t do_t + g_{t+1} lam_{t+1} (lam_T = r_T do_T + dS_T):
    dr = s_t do_t, dk = lam_t v_t, dv = lam_t k_t, dw = lam_t e^{w_t} s_{t-1},
    dkk = -2 lam_t a_t kk_t s_{t-1}, da = -lam_t kk_t^2 s_{t-1}, dS0 = g_1 lam_1.
    """
    T = 9
    g = _rng(42)
    r, k, v, d_o = (g.standard_normal((T, 1, 1)) for _ in range(4))
    r, k, v = _f32(r), _f32(k), _f32(v)
    w = _f32(-0.6 * g.random((T, 1, 1)))
    kk = _f32(np.where(g.random((T, 1, 1)) < 0.5, -1.0, 1.0) * g.random((T, 1, 1)))
    a = _f32(g.random((T, 1, 1)))
    s0, dsf = 0.625, -1.5
    dr, dw, dk, dv, dkk, da, ds0 = _bwd(lib, r, w, k, v, kk, a, d_o, s0=np.full((1, 1, 1, 1), s0),
                                        dsf=np.full((1, 1, 1, 1), dsf))
    f = lambda x: x[:, 0, 0].astype(np.float64)  # noqa: E731
    r, w, k, v, kk, a, d_o = map(f, (r, w, k, v, kk, a, d_o))
    gm = np.exp(w) - a * kk * kk
    s = np.zeros(T + 1)
    s[0] = s0
    for t in range(T):
        s[t + 1] = gm[t] * s[t] + k[t] * v[t]
    lam = np.zeros(T)
    nxt = dsf
    for t in range(T - 1, -1, -1):
        lam[t] = r[t] * d_o[t] + nxt
        nxt = gm[t] * lam[t]
    _close(dr[:, 0, 0], s[1:] * d_o, 1e-12, "dr")
    _close(dk[:, 0, 0], lam * v, 1e-12, "dk")
    _close(dv[:, 0, 0], lam * k, 1e-12, "dv")
    _close(dw[:, 0, 0], lam * np.exp(w) * s[:-1], 1e-12, "dw")
    _close(dkk[:, 0, 0], -2.0 * lam * a * kk * s[:-1], 1e-12, "dkk")
    _close(da[:, 0, 0], -lam * kk * kk * s[:-1], 1e-12, "da")
    _close(ds0[0, 0, 0, 0], gm[0] * lam[0], 1e-12, "dS0")


def pin_bwd_euler_identities(lib):
    """The loss is linear in r, and homogeneous of degree one in (S0, v) and
    in (S0, k) jointly, so <r, dr> = <dO, o> and
    <S0, dS0> + <v, dv> = <S0, dS0> + <k, dk> = L."""
    H, N = 3, 8
    cu = np.array([0, 5, 5, 19])
    T = 19
    r, w, k, v, kk, a = _draw(T, H, N, seed=43)
    g = _rng(44)
    s0 = g.standard_normal((3, H, N, N))
    d_o = g.standard_normal((T, H, N))
    dsf = g.standard_normal((3, H, N, N))
    o, s = _run(lib, r, w, k, v, kk, a, cu=cu, s0=s0)
    lo = float(np.sum(o * d_o))
    L = lo + float(np.sum(s * dsf))
    dr, dw, dk, dv, dkk, da, ds0 = _bwd(lib, r, w, k, v, kk, a, d_o, cu=cu, s0=s0, dsf=dsf)
    f = lambda x: x.astype(np.float64)  # noqa: E731
    _close(np.sum(f(r) * dr), lo, 1e-12, "<r, dr> = <dO, o>")
    _close(np.sum(s0 * ds0) + np.sum(f(v) * dv), L, 1e-12, "<S0, dS0> + <v, dv> = L")
    _close(np.sum(s0 * ds0) + np.sum(f(k) * dk), L, 1e-12, "<S0, dS0> + <k, dk> = L")


def pin_bwd_split_invariance(lib):
    """The backward of [0, T) equals the backward of [T1, T) (from the carried
    state) followed by that of [0, T1) with dS_T1 = the second part's dS0."""
    T, H, N = 21, 2, 8
    r, w, k, v, kk, a = _draw(T, H, N, seed=45)
    g = _rng(46)
    s0 = g.standard_normal((1, H, N, N))
    d_o = g.standard_normal((T, H, N))
    dsf = g.standard_normal((1, H, N, N))
    whole = _bwd(lib, r, w, k, v, kk, a, d_o, s0=s0, dsf=dsf)
    xs = (r, w, k, v, kk, a)
    for T1 in (1, 8, 20):
        _, s_mid = _run(lib, *(x[:T1] for x in xs), s0=s0)
        second = _bwd(lib, *(x[T1:] for x in xs), d_o[T1:], s0=s_mid, dsf=dsf)
        first = _bwd(lib, *(x[:T1] for x in xs), d_o[:T1], s0=s0, dsf=second[6])
        for q in range(6):
            _close(np.concatenate([first[q], second[q]]), whole[q], 1e-12, f"grad {q} split at {T1}")
        _close(first[6], whole[6], 1e-12, f"dS0 split at {T1}")


def pin_bwd_packing_and_zero_length(lib):
    """A packed backward equals per-sequence backwards; a 0-token sequence
    passes dS_T through as dS0 (zeros when none given)."""
    H, N = 2, 4
    lens = [3, 0, 6]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = sum(lens)
    r, w, k, v, kk, a = _draw(T, H, N, seed=47)
    g = _rng(48)
    s0 = g.standard_normal((3, H, N, N))
    d_o = g.standard_normal((T, H, N))
    dsf = g.standard_normal((3, H, N, N))
    packed = _bwd(lib, r, w, k, v, kk, a, d_o, cu=cu, s0=s0, dsf=dsf)
    for b, n in enumerate(lens):
        sl = slice(cu[b], cu[b + 1])
        one = _bwd(lib, *(x[sl] for x in (r, w, k, v, kk, a)), d_o[sl], s0=s0[b:b + 1], dsf=dsf[b:b + 1])
        for q in range(6):
            _close(packed[q][sl], one[q], 0.0, f"packed grad {q} seq {b}")
        _close(packed[6][b], one[6][0], 0.0, f"packed dS0 seq {b}")
    _close(packed[6][1], dsf[1], 0.0, "zero-length passes dS_T")
    none = _bwd(lib, r, w, k, v, kk, a, d_o, cu=cu, s0=s0)
    _close(none[6][1], np.zeros((H, N, N)), 0.0, "zero-length without dS_T")


ALL_PINS = [
    pin_golden_hand_n2,
    pin_t1_zero_state,
    pin_t2_zero_state,
    pin_a0_decayed_linear_attention,
    pin_a0_w0_causal_linear_attention,
    pin_projector,
    pin_split_invariance,
    pin_scalar_n1,
    pin_linearity,
    pin_equivariance,
    pin_packing,
    pin_zero_length,
    pin_tail_golden_hand_n2,
    pin_tail_standardises,
    pin_tail_shift_and_scale_invariance,
    pin_tail_gate_scales_the_sum,
    pin_tail_bonus_unit_vectors,
    pin_tail_constant_head,
    pin_tail_heads_use_their_parameters,
    pin_bwd_finite_differences,
    pin_bwd_scalar_n1,
    pin_bwd_euler_identities,
    pin_bwd_split_invariance,
    pin_bwd_packing_and_zero_length,
]
