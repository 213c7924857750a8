"""fp64 oracle for the gated delta rule forward pass (test infrastructure only).

The pages name the gated-delta-network (GDN) family as the target of the operator
libraries they discuss ("面向长序列大模型的线性注意力算子性能评测方法与优化实践",
section 三.3 GDN类机制的引入: a gate and an incremental (delta) update on the recurrent
state; "线性注意力GPU算子库的定义与技术解析", section 三: gated linear attention of the
Gated Delta Network kind). They print no formula. The reading taken here is the published
gated delta rule, with one scalar gate and one writing strength per token and head:

    S_0 = h0 (or 0)
    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T     (Dk x Dv state)
    o_t = scale q_t S_t                                               (row vector, Dv)
    hT  = S_T

with alpha_t = exp(g_t). This is the GLA recurrence of the other oracle (same state
layout [Dk, Dv], same read after the update) with the additive write k_t^T v_t replaced
by the delta write: the state first forgets what it stored under key k_t (a rank-one
projection), then stores beta_t v_t there.

Layouts: q, k [B, T, H, Dk]; v, o [B, T, H, Dv]; g, beta [B, T, H]; h0, hT [B, H, Dk, Dv].
Inputs are widened exactly to float32 and every operation runs in float64.

Functions:

* ``recurrent`` — the token loop above, literally (fp64, numpy, vectorised over batch
  and heads).
* ``recurrent_c`` — the same token loop written independently in C (``gdn_oracle.c``,
  OpenMP over the (batch, head) pairs), for the CPU baselines and large checks.
* ``recurrent_head`` — the numpy loop for one (batch, head), for sampled checks at full
  size.
* ``chunkwise`` — the chunk algebra the GPU path uses, in fp64: per chunk a unit lower
  triangular solve turns the delta writes into "new values" U, and the chunk's outputs
  and end state follow from U by matrix products. It is pinned against ``recurrent``.

Pins: ``tests/test_gdn_oracle_pins.py`` checks the recurrence against closed forms
(no writes: pure decay; unit keys with beta = 1: the state returns v_t exactly under
k_t; orthonormal keys without decay: a lookup table whose slots are overwritten),
against the explicit product of the Dk x Dk transition matrices on tiny inputs, and
against linearity and state carry. The formula itself is the outside reading stated
above; within that reading no function here is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``oracle/_build/libgdn_oracle.so`` with gcc (OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.gdn_oracle_batch.argtypes = [p, p, p, p, p, ctypes.c_double, p, p, p,
                                             i64, i64, i64, i64, i64]
            lib.gdn_oracle_batch.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    """Widen a numpy array or torch CPU tensor to float64 (through float32: exact for bf16)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def recurrent(q, k, v, g, beta, scale: float, h0=None):
    """The gated delta rule, token by token, in fp64. Returns (o, hT) as float64."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    assert k.shape == q.shape and v.shape == (B, T, H, Dv)
    assert g.shape == (B, T, H) and beta.shape == (B, T, H)
    S = np.zeros((B, H, Dk, Dv)) if h0 is None else _f64(h0).copy()
    o = np.empty((B, T, H, Dv))
    for t in range(T):
        kt, vt = k[:, t], v[:, t]                       # [B, H, Dk], [B, H, Dv]
        a = np.exp(g[:, t])[..., None, None]            # alpha_t
        bt = beta[:, t][..., None, None]                # beta_t
        # (I - beta k k^T) S = S - beta k (k^T S)
        kS = np.einsum("bhd,bhde->bhe", kt, S)           # k_t^T S_{t-1}, [B, H, Dv]
        S = a * (S - bt * kt[..., :, None] * kS[..., None, :]) + bt * kt[..., :, None] * vt[..., None, :]
        o[:, t] = scale * np.einsum("bhd,bhde->bhe", q[:, t], S)
    return o, S


def _c32(x):
    """Contiguous float32 copy (exact for bf16 inputs), or None."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().contiguous().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def recurrent_c(q, k, v, g, beta, scale: float, h0=None):
    """The token loop in C (fp64, OpenMP over (batch, head)). Returns (o, hT) as float64."""
    q, k, v, g, beta, h0 = (_c32(x) for x in (q, k, v, g, beta, h0))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    assert k.shape == q.shape and v.shape == (B, T, H, Dv)
    assert g.shape == (B, T, H) and beta.shape == (B, T, H)
    if h0 is not None:
        assert h0.shape == (B, H, Dk, Dv)
    o = np.empty((B, T, H, Dv), dtype=np.float64)
    hT = np.empty((B, H, Dk, Dv), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)   # noqa: E731
    rc = _load().gdn_oracle_batch(ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), float(scale),
                                  ptr(h0), ptr(o), ptr(hT), B, T, H, Dk, Dv)
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return o, hT


def recurrent_head(q, k, v, g, beta, scale: float, h0, b: int, h: int, t_end: int | None = None):
    """The token loop for one (batch b, head h) over tokens [0, t_end).

    Returns (o [t_end, Dv], hT [Dk, Dv]) as float64.
    """
    T = q.shape[1]
    t_end = T if t_end is None else int(t_end)
    sl = lambda x: None if x is None else x[b:b + 1, :t_end, h:h + 1]   # noqa: E731
    h0h = None if h0 is None else h0[b:b + 1, h:h + 1]
    o, S = recurrent(sl(q), sl(k), sl(v), sl(g), sl(beta), scale, h0h)
    return o[0, :, 0], S[0, 0]


def chunkwise(q, k, v, g, beta, scale: float, h0=None, C: int = 64):
    """The chunk algebra of the gated delta rule in fp64 (the GPU path's method).

    For one chunk of L tokens starting from state S0, with b_i the inclusive in-chunk
    cumulative log-gate and gamma_i = exp(b_i):

      * the state just before the delta write of token j is
            gamma_j S0 + sum_{m<j} exp(b_j - b_m) k_m u_m^T,
        where u_m = beta_m (v_m - (that state)^T k_m) is the "new value" token m wrote;
      * so the rows u_j solve the unit lower triangular system
            u_j + sum_{m<j} beta_j exp(b_j - b_m) (k_j . k_m) u_m = beta_j (v_j - gamma_j S0^T k_j),
        i.e. U = Ut - W S0 with (I + A) Ut = diag(beta) V and (I + A) W = diag(beta gamma) K;
      * the outputs are o_i = scale (gamma_i q_i S0 + sum_{j<=i} exp(b_i - b_j) (q_i . k_j) u_j);
      * the end state is gamma_{L-1} S0 + sum_j exp(b_{L-1} - b_j) k_j u_j^T.

    The sequence split into chunks and the matrix form of the in-chunk work follow
    "线性注意力GPU算子库的定义与技术解析", section 三 (sequence parallelism with the state
    passed from block to block; rewriting the recurrence as block matrix products).
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    S = np.zeros((B, H, Dk, Dv)) if h0 is None else _f64(h0).copy()
    o = np.empty((B, T, H, Dv))
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        L = t1 - t0
        qc = q[:, t0:t1].transpose(0, 2, 1, 3)            # [B, H, L, Dk]
        kc = k[:, t0:t1].transpose(0, 2, 1, 3)
        vc = v[:, t0:t1].transpose(0, 2, 1, 3)            # [B, H, L, Dv]
        bc = beta[:, t0:t1].transpose(0, 2, 1)            # [B, H, L]
        lb = np.cumsum(g[:, t0:t1].transpose(0, 2, 1), axis=2)   # b_i, [B, H, L]
        diff = lb[..., :, None] - lb[..., None, :]        # b_i - b_j
        low = np.tril(np.ones((L, L)), -1)                # m < j
        A = bc[..., :, None] * np.exp(np.where(low > 0, diff, 0.0)) * low \
            * np.einsum("bhjd,bhmd->bhjm", kc, kc)
        I = np.eye(L)
        rhs_v = bc[..., None] * vc
        rhs_k = (bc * np.exp(lb))[..., None] * kc
        Ut = np.linalg.solve(I + A, rhs_v)                # [B, H, L, Dv]
        W = np.linalg.solve(I + A, rhs_k)                 # [B, H, L, Dk]
        U = Ut - np.einsum("bhjd,bhde->bhje", W, S)
        incl = np.tril(np.ones((L, L)))
        P = np.exp(np.where(incl > 0, diff, 0.0)) * incl * np.einsum("bhid,bhjd->bhij", qc, kc)
        O = scale * (np.exp(lb)[..., None] * np.einsum("bhid,bhde->bhie", qc, S)
                     + np.einsum("bhij,bhje->bhie", P, U))
        o[:, t0:t1] = O.transpose(0, 2, 1, 3)
        last = lb[..., -1]                                # b_{L-1}, [B, H]
        Kh = np.exp(last[..., None] - lb)[..., None] * kc
        S = np.exp(last)[..., None, None] * S + np.einsum("bhjd,bhje->bhde", Kh, U)
    return o, S
