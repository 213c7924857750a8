"""Independent checks that pin the oracle.

Each check returns ``(err, tol)``: the max error relative to the reference's max
magnitude, and the bound it must meet.

Every check takes an oracle callable ``fn(q, k, v, g, scale, h0) -> (o, hT)`` working
on [B, T, H, D] arrays, so the same checks run on every oracle implementation and on
deliberately broken copies of it (``tests/test_oracle_pins.py``). None of these
re-types the recurrence: each compares against a different formula or an exact fact.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(float(np.max(np.abs(b))), 1e-300)
    return float(np.max(np.abs(a - b))) / den


def rand_case(rng, B=1, T=12, H=2, Dk=6, Dv=5, gate_scale=0.3, with_h0=True):
    q = rng.standard_normal((B, T, H, Dk)).astype(np.float32)
    k = rng.standard_normal((B, T, H, Dk)).astype(np.float32)
    v = rng.standard_normal((B, T, H, Dv)).astype(np.float32)
    # log-gates of both signs-of-magnitude: mostly decays, exact float32 values
    g = (-gate_scale * rng.random((B, T, H, Dk)) ** 2).astype(np.float32)
    h0 = rng.standard_normal((B, H, Dk, Dv)).astype(np.float32) if with_h0 else None
    return q, k, v, g, h0


def brute_force(q, k, v, g, scale, h0):
    """O(T^2) parallel (attention) form with the decay matrix written out term by term.

    o_i = scale * [ sum_{j<=i} sum_d q_id k_jd (prod_{s=j+1..i} exp(g_sd)) v_j
                    + sum_d q_id (prod_{s=0..i} exp(g_sd)) h0_d ]
    hT  = sum_j diag(prod_{s=j+1..T-1} exp(g_s)) k_j^T v_j + diag(prod_s exp(g_s)) h0
    The decay products are multiplied out one factor at a time (no cumulative sums).
    """
    q, k, v, g = (np.asarray(x, np.float64) for x in (q, k, v, g))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    a = np.exp(g)
    o = np.zeros((B, T, H, Dv))
    hT = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            for i in range(T):
                acc = np.zeros(Dv)
                for j in range(i + 1):
                    dec = np.ones(Dk)
                    for s in range(j + 1, i + 1):
                        dec = dec * a[b, s, h]
                    acc += np.sum(q[b, i, h] * k[b, j, h] * dec) * v[b, j, h]
                if h0 is not None:
                    dec = np.ones(Dk)
                    for s in range(0, i + 1):
                        dec = dec * a[b, s, h]
                    acc += (q[b, i, h] * dec) @ np.asarray(h0[b, h], np.float64)
                o[b, i, h] = scale * acc
            st = np.zeros((Dk, Dv))
            for j in range(T):
                dec = np.ones(Dk)
                for s in range(j + 1, T):
                    dec = dec * a[b, s, h]
                st += (dec * k[b, j, h])[:, None] * v[b, j, h][None, :]
            if h0 is not None:
                dec = np.ones(Dk)
                for s in range(T):
                    dec = dec * a[b, s, h]
                st += dec[:, None] * np.asarray(h0[b, h], np.float64)
            hT[b, h] = st
    return o, hT


def check_brute_force(fn, rng, **kw):
    q, k, v, g, h0 = rand_case(rng, **kw)
    o, hT = fn(q, k, v, g, 0.37, h0)
    ob, hb = brute_force(q, k, v, g, 0.37, h0)
    return max(rel(o, ob), rel(hT, hb)), 1e-12


def check_ungated_textbook(fn, rng, T=20, Dk=7, Dv=9):
    """g = 0, h0 = 0 reduces to causal linear attention scale * tril(Q K^T) V."""
    q, k, v, _, _ = rand_case(rng, B=2, T=T, H=2, Dk=Dk, Dv=Dv, with_h0=False)
    g = np.zeros_like(q)
    o, hT = fn(q, k, v, g, 0.5, None)
    err = 0.0
    for b in range(2):
        for h in range(2):
            Q = q[b, :, h].astype(np.float64)
            K = k[b, :, h].astype(np.float64)
            V = v[b, :, h].astype(np.float64)
            err = max(err, rel(o[b, :, h], 0.5 * np.tril(Q @ K.T) @ V))
            err = max(err, rel(hT[b, h], K.T @ V))
    return err, 1e-12


def check_full_forgetting(fn, rng):
    """g = -1e4 makes exp(g) underflow to 0: each token sees only itself.

    o_t = scale (q_t . k_t) v_t, and hT = k_{T-1}^T v_{T-1} whatever h0 was.
    """
    q, k, v, _, h0 = rand_case(rng, B=1, T=9, H=3, Dk=5, Dv=4)
    g = np.full_like(q, -1e4)
    o, hT = fn(q, k, v, g, 0.8, h0)
    q64, k64, v64 = (x.astype(np.float64) for x in (q, k, v))
    o_ref = 0.8 * np.sum(q64 * k64, axis=-1, keepdims=True) * v64
    hT_ref = k64[:, -1, :, :, None] * v64[:, -1, :, None, :]
    return max(rel(o, o_ref), rel(hT, hT_ref)), 1e-14


def check_geometric(fn, gamma=0.9, T=40, h0val=0.25, scale=0.7):
    """Dk = Dv = 1 with q = k = v = 1 and a constant decay gamma: a geometric series.

    o_t = scale * ((1 - gamma^(t+1)) / (1 - gamma) + gamma^(t+1) h0).
    """
    ones = np.ones((1, T, 1, 1), np.float32)
    g = np.full((1, T, 1, 1), np.log(gamma), np.float32)
    gam = float(np.exp(np.float64(g.flat[0])))     # the float32 gate's exact decay
    h0 = np.full((1, 1, 1, 1), h0val, np.float32)
    o, hT = fn(ones, ones, ones, g, scale, h0)
    t = np.arange(T, dtype=np.float64)
    ref = scale * ((1 - gam ** (t + 1)) / (1 - gam) + gam ** (t + 1) * h0val)
    href = (1 - gam ** T) / (1 - gam) + gam ** T * h0val
    return max(rel(o[0, :, 0, 0], ref), rel(hT[0, 0, 0, 0], href)), 1e-12


def check_single_token(fn, rng):
    """T = 1: o = scale * q (diag(exp(g)) h0 + k^T v), hT = diag(exp(g)) h0 + k^T v."""
    q, k, v, g, h0 = rand_case(rng, B=2, T=1, H=2, Dk=6, Dv=3)
    o, hT = fn(q, k, v, g, 1.3, h0)
    q64, k64, v64, g64, h64 = (x.astype(np.float64) for x in (q, k, v, g, h0))
    S = np.exp(g64[:, 0])[..., None] * h64 + k64[:, 0, :, :, None] * v64[:, 0, :, None, :]
    o_ref = 1.3 * np.einsum("bhd,bhde->bhe", q64[:, 0], S)
    return max(rel(o[:, 0], o_ref), rel(hT, S)), 1e-14


def check_state_carry(fn, rng, T=24, split=11):
    """Running [0, T) equals running [0, split) and then [split, T) from the returned state."""
    q, k, v, g, h0 = rand_case(rng, B=1, T=T, H=2, Dk=6, Dv=5)
    o, hT = fn(q, k, v, g, 0.6, h0)
    o1, h1 = fn(q[:, :split], k[:, :split], v[:, :split], g[:, :split], 0.6, h0)
    o2, h2 = fn(q[:, split:], k[:, split:], v[:, split:], g[:, split:], 0.6,
                h1.astype(np.float32))
    # The first half must match to fp64 rounding. The second half restarts from h1
    # rounded to float32 (the oracle takes float32 inputs), so it matches to float32
    # resolution of the carried state (~6e-8 relative), not better.
    e1 = rel(o[:, :split], o1) / 1e-13
    e2 = max(rel(o[:, split:], o2), rel(hT, h2)) / 1e-6
    return max(e1, e2), 1.0


def check_state_carry_exact(fn, rng, T=24, split=11):
    """State carry with a state that is exactly representable in float32 (g = 0, k,v small
    integers): the split run must match the whole run to fp64 rounding."""
    q = rng.integers(-3, 4, (1, T, 2, 4)).astype(np.float32)
    k = rng.integers(-3, 4, (1, T, 2, 4)).astype(np.float32)
    v = rng.integers(-3, 4, (1, T, 2, 3)).astype(np.float32)
    g = np.zeros_like(q)
    o, hT = fn(q, k, v, g, 0.5, None)
    o1, h1 = fn(q[:, :split], k[:, :split], v[:, :split], g[:, :split], 0.5, None)
    o2, h2 = fn(q[:, split:], k[:, split:], v[:, split:], g[:, split:], 0.5,
                h1.astype(np.float32))
    return max(rel(o[:, :split], o1), rel(o[:, split:], o2), rel(hT, h2)), 1e-13


def check_linearity(fn, rng):
    """o is linear in v (h0 = 0), and o(h0) - o(0) = scale (q * exp(G_t)) h0 with
    G_t = sum_{s<=t} g_s (the h0 term of the unrolled recurrence)."""
    q, k, v, g, h0 = rand_case(rng, B=1, T=15, H=2, Dk=6, Dv=4)
    v2 = rng.standard_normal(v.shape).astype(np.float32)
    oa, _ = fn(q, k, v, g, 0.9, None)
    ob, _ = fn(q, k, v2, g, 0.9, None)
    vs = (v.astype(np.float64) + 2.0 * v2.astype(np.float64)).astype(np.float32)
    oc, _ = fn(q, k, vs, g, 0.9, None)
    # vs was rounded to float32, so linearity holds to float32 input rounding
    e1 = rel(oc, oa + 2.0 * ob) / 1e-6
    oh, _ = fn(q, k, v, g, 0.9, h0)
    G = np.cumsum(g.astype(np.float64), axis=1)
    ref = 0.9 * np.einsum("bthd,bhde->bthe", q.astype(np.float64) * np.exp(G),
                          h0.astype(np.float64))
    e2 = rel(oh - oa, ref) / 1e-12
    return max(e1, e2), 1.0


def check_exact_rational(fn):
    """Exact arithmetic: decays 1/2 and 1/4, small-integer q, k, v, h0.

    The expected values are computed with python Fractions from the unrolled sum
    o_t = scale * q_t (sum_{j<=t} D(j,t) k_j^T v_j + D(-1,t) h0), D = product of decays.
    exp(log(1/2)) and exp(log(1/4)) are within one ulp of 1/2 and 1/4, so the oracle
    must agree to ~1e-15.
    """
    T, Dk, Dv = 5, 2, 2
    qi = [[1, -2], [0, 3], [2, 1], [-1, -1], [3, 0]]
    ki = [[2, 1], [-1, 1], [1, 0], [0, 2], [1, -3]]
    vi = [[1, 0], [2, -1], [-3, 1], [1, 1], [0, 2]]
    h0i = [[1, -1], [2, 0]]
    scale = Fraction(1, 2)
    f = lambda rows: np.array(rows, np.float32)[None, :, None, :]  # noqa: E731
    g = np.array([[np.log(0.5), np.log(0.25)]] * T, np.float32)[None, :, None, :]
    # the float32 gates are not exactly log(1/2), log(1/4): rescale the reference by the
    # exact decays the oracle sees, recomputing with those decays in Fractions
    a_exact = [Fraction(float(np.exp(np.float64(g[0, 0, 0, d])))) for d in range(Dk)]
    S = [[Fraction(x) for x in row] for row in h0i]
    o_ref = []
    for t in range(T):
        S = [[a_exact[d] * S[d][e] + ki[t][d] * vi[t][e] for e in range(Dv)] for d in range(Dk)]
        o_ref.append([scale * sum(qi[t][d] * S[d][e] for d in range(Dk)) for e in range(Dv)])
    h0 = np.array(h0i, np.float32)[None, None]
    o, hT = fn(f(qi), f(ki), f(vi), g, 0.5, h0)
    o_ref = np.array([[float(x) for x in row] for row in o_ref])
    hT_ref = np.array([[float(x) for x in row] for row in S])
    return max(rel(o[0, :, 0, :], o_ref), rel(hT[0, 0], hT_ref)), 1e-15


ALL_CHECKS = {
    "brute_force": lambda fn, rng: check_brute_force(fn, rng),
    "brute_force_wide": lambda fn, rng: check_brute_force(fn, rng, T=6, H=1, Dk=128, Dv=128),
    "ungated_textbook": check_ungated_textbook,
    "full_forgetting": lambda fn, rng: check_full_forgetting(fn, rng),
    "geometric": lambda fn, rng: check_geometric(fn),
    "single_token": check_single_token,
    "state_carry": check_state_carry,
    "state_carry_exact": check_state_carry_exact,
    "linearity": check_linearity,
    "exact_rational": lambda fn, rng: check_exact_rational(fn),
}
