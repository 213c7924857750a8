"""Independent checks that pin the gated-delta-rule oracle.

Every check takes a callable ``fn(q, k, v, g, beta, scale, h0) -> (o, hT)`` on
[B, T, H, D] arrays (g, beta [B, T, H]) and returns ``(err, tol)``. None of them
re-types the token loop: each compares against a closed form, an exact property of the
delta write, a different formula (products of the transition matrices), or an
invariant (linearity, state carry).
"""
from __future__ import annotations

import numpy as np

from pins import rel


def unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_case(rng, B=1, T=12, H=2, Dk=6, Dv=5, with_h0=True, unit_keys=True):
    """Small random inputs: unit-norm keys (the delta rule's usual regime), gates in
    (-0.5, 0], write strengths in (0, 1)."""
    q = rng.standard_normal((B, T, H, Dk))
    k = rng.standard_normal((B, T, H, Dk))
    if unit_keys:
        k = unit_rows(k)
    v = rng.standard_normal((B, T, H, Dv))
    g = -0.5 * rng.random((B, T, H))
    beta = rng.random((B, T, H))
    h0 = rng.standard_normal((B, H, Dk, Dv)) if with_h0 else None
    f = lambda x: None if x is None else np.asarray(x, np.float32)   # noqa: E731
    return f(q), f(k), f(v), f(g), f(beta), f(h0)


def check_no_write(fn, rng, T=15, Dk=5, Dv=4):
    """beta = 0: nothing is written, the state only decays.
    S_t = exp(g_0 + ... + g_t) h0 and o_t = scale exp(g_0 + ... + g_t) q_t h0."""
    q, k, v, g, beta, h0 = rand_case(rng, B=2, T=T, H=2, Dk=Dk, Dv=Dv)
    beta = np.zeros_like(beta)
    scale = 0.8
    o, hT = fn(q, k, v, g, beta, scale, h0)
    G = np.cumsum(g.astype(np.float64), axis=1)                       # [B, T, H]
    o_ref = scale * np.exp(G)[..., None] * np.einsum("bthd,bhde->bthe", q.astype(np.float64), h0)
    h_ref = np.exp(G[:, -1])[..., None, None] * h0
    return max(rel(o, o_ref), rel(hT, h_ref)), 1e-12


def check_readback(fn, rng, T=20, Dk=8, Dv=6):
    """Unit keys and beta = 1: right after token t writes, reading the state with key
    k_t returns v_t exactly, whatever the decay and the earlier contents
    (k^T [alpha (I - k k^T) S + k v^T] = alpha (k^T - k^T) S + v^T = v^T)."""
    q, k, v, g, beta, h0 = rand_case(rng, B=1, T=T, H=3, Dk=Dk, Dv=Dv)
    k = unit_rows(k.astype(np.float64))
    beta = np.ones_like(beta)
    o, hT = fn(k, k, v, g, beta, 1.0, h0)          # queries = keys, scale 1
    err = rel(o, v)
    # and the final state returns the last value under the last key
    err = max(err, rel(np.einsum("bhd,bhde->bhe", k[:, -1], hT), v[:, -1]))
    return err, 1e-6    # keys are unit-norm only to float32 rounding


def check_lookup_table(fn, rng, T=30, Dk=6, Dv=4):
    """Keys drawn from the standard basis and beta = 1: each write overwrites one row of
    the state (row i <- v_t), and every row decays by alpha per step afterwards. The
    expected state is built by plain assignment, token by token."""
    B, H = 1, 2
    idx = rng.integers(0, Dk, size=(B, T, H))                           # repeats on purpose
    k = np.zeros((B, T, H, Dk), np.float32)
    for b in range(B):
        for t in range(T):
            for h in range(H):
                k[b, t, h, idx[b, t, h]] = 1.0
    q = rng.standard_normal((B, T, H, Dk)).astype(np.float32)
    v = rng.standard_normal((B, T, H, Dv)).astype(np.float32)
    g = (-0.3 * rng.random((B, T, H))).astype(np.float32)
    beta = np.ones((B, T, H), np.float32)
    h0 = rng.standard_normal((B, H, Dk, Dv)).astype(np.float32)
    scale = 0.6
    o, hT = fn(q, k, v, g, beta, scale, h0)
    o_ref = np.zeros((B, T, H, Dv))
    table = h0.astype(np.float64).copy()
    for t in range(T):
        for b in range(B):
            for h in range(H):
                table[b, h] *= np.exp(np.float64(g[b, t, h]))               # every row decays
                table[b, h, idx[b, t, h]] = v[b, t, h]                      # the keyed row is replaced
                o_ref[b, t, h] = scale * q[b, t, h].astype(np.float64) @ table[b, h]
    return max(rel(o, o_ref), rel(hT, table)), 1e-12


def check_product_form(fn, rng, T=7, Dk=4, Dv=3):
    """Closed form through the Dk x Dk transition matrices Phi_t = alpha_t (I - beta_t
    k_t k_t^T), multiplied out one factor at a time:
        S_t = Phi_t ... Phi_0 h0 + sum_{j<=t} Phi_t ... Phi_{j+1} beta_j k_j v_j^T."""
    q, k, v, g, beta, h0 = rand_case(rng, B=1, T=T, H=2, Dk=Dk, Dv=Dv, unit_keys=False)
    scale = 1.3
    o, hT = fn(q, k, v, g, beta, scale, h0)
    q, k, v, g, beta, h0 = (x.astype(np.float64) for x in (q, k, v, g, beta, h0))
    B, _, H, _ = q.shape
    o_ref = np.zeros((B, T, H, Dv))
    h_ref = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            phi = [np.exp(g[b, t, h]) * (np.eye(Dk) - beta[b, t, h] * np.outer(k[b, t, h], k[b, t, h]))
                   for t in range(T)]
            for t in range(T):
                prod = np.eye(Dk)
                for s in range(t, -1, -1):      # Phi_t ... Phi_0
                    prod = prod @ phi[s]
                St = prod @ h0[b, h]
                for j in range(t + 1):
                    prod = np.eye(Dk)
                    for s in range(t, j, -1):   # Phi_t ... Phi_{j+1}
                        prod = prod @ phi[s]
                    St = St + prod @ (beta[b, j, h] * np.outer(k[b, j, h], v[b, j, h]))
                o_ref[b, t, h] = scale * q[b, t, h] @ St
            h_ref[b, h] = St
    return max(rel(o, o_ref), rel(hT, h_ref)), 1e-12


def check_linearity(fn, rng, T=16, Dk=6, Dv=5):
    """For fixed q, k, g, beta the map (v, h0) -> (o, hT) is linear."""
    q, k, _, g, beta, _ = rand_case(rng, B=1, T=T, H=2, Dk=Dk, Dv=Dv)
    # values on a coarse dyadic grid, so that v1 + 2 v2 and h1 + 2 h2 are exact in float32
    grid = lambda shape: (rng.integers(-64, 65, size=shape) / 16.0).astype(np.float32)   # noqa: E731
    v1, v2 = grid((1, T, 2, Dv)), grid((1, T, 2, Dv))
    h1, h2 = grid((1, 2, Dk, Dv)), grid((1, 2, Dk, Dv))
    c = np.float32(2.0)
    o1, s1 = fn(q, k, v1, g, beta, 0.5, h1)
    o2, s2 = fn(q, k, v2, g, beta, 0.5, h2)
    o3, s3 = fn(q, k, v1 + c * v2, g, beta, 0.5, h1 + c * h2)
    return max(rel(o3, o1 + 2.0 * o2), rel(s3, s1 + 2.0 * s2)), 1e-12


def check_state_carry(fn, rng, T=26, split=11, Dk=6, Dv=5):
    """Running [0, T) equals running [0, split) and then [split, T) from its final state."""
    q, k, v, g, beta, h0 = rand_case(rng, B=2, T=T, H=2, Dk=Dk, Dv=Dv)
    o, hT = fn(q, k, v, g, beta, 0.7, h0)
    sl = lambda x, a, b: x[:, a:b]   # noqa: E731
    oa, ha = fn(*(sl(x, 0, split) for x in (q, k, v, g, beta)), 0.7, h0)
    ob, hb = fn(*(sl(x, split, T) for x in (q, k, v, g, beta)), 0.7, ha.astype(np.float32))
    # the carried state is rounded to float32 on the way in: compare at that precision
    return max(rel(np.concatenate([oa, ob], axis=1), o), rel(hb, hT)), 1e-6


ALL_CHECKS = {
    "no_write": check_no_write,
    "readback": check_readback,
    "lookup_table": check_lookup_table,
    "product_form": check_product_form,
    "linearity": check_linearity,
    "state_carry": check_state_carry,
}
