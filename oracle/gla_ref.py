"""fp64 oracle for the GLA prefill forward pass (test infrastructure only).

Three functions compute the same thing:

* ``recurrent``      — the C token-by-token recurrence (``gla_oracle.c``), all heads.
* ``recurrent_head`` — the same C routine on one (batch, head) of a large batch,
                       reading the float32 inputs in place (for sampled checks at
                       full size).
* ``recurrent_np``   — an independent pure-numpy token loop of the same definition.
* ``chunkwise_np``   — the chunkwise form in fp64 (chunk steps of the GPU method),
                       used to check that the chunk algebra reaches the recurrence.

Definition (per batch b and head h; "Linear Attention 在 GPU 上到底慢在哪",
section 学长的反馈, and "线性注意力GPU算子库的定义与技术解析", section 四):

    S_0 = h0 (or 0);  S_t = diag(exp(g_t)) S_{t-1} + k_t^T v_t;  o_t = scale q_t S_t;
    hT = S_T.

Layouts: q, k, g are [B, T, H, Dk]; v, o are [B, T, H, Dv]; h0, hT are [B, H, Dk, Dv].
Inputs may be numpy arrays or torch CPU tensors of any float dtype; they are widened
exactly to float32 (bf16 -> fp32 is exact) and every operation runs in float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gla_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc (OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, f32p, f64p = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            lib.gla_oracle_head.argtypes = [f32p, f32p, f32p, f32p, i64, i64, i64,
                                            i64, i64, i64, i64, ctypes.c_double,
                                            f32p, f64p, i64, f64p]
            lib.gla_oracle_head.restype = ctypes.c_int
            lib.gla_oracle_batch.argtypes = [f32p, f32p, f32p, f32p, ctypes.c_double,
                                             f32p, f64p, f64p, i64, i64, i64, i64, i64]
            lib.gla_oracle_batch.restype = ctypes.c_int
            lib.gla_oracle_num_threads.argtypes = []
            lib.gla_oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the C oracle's OpenMP loop uses on this host."""
    return int(_load().gla_oracle_num_threads())


def _f32(x) -> np.ndarray:
    """Widen a numpy array or torch CPU tensor to contiguous float32 (exact for bf16/fp16)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").float().contiguous().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def recurrent(q, k, v, g, scale: float, h0=None):
    """Token-by-token fp64 recurrence over all heads (C). Returns (o, hT) as float64."""
    q, k, v, g, h0 = _f32(q), _f32(k), _f32(v), _f32(g), _f32(h0)
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    assert k.shape == q.shape and g.shape == q.shape and v.shape == (B, T, H, Dv)
    if h0 is not None:
        assert h0.shape == (B, H, Dk, Dv)
    o = np.empty((B, T, H, Dv), dtype=np.float64)
    hT = np.empty((B, H, Dk, Dv), dtype=np.float64)
    rc = _load().gla_oracle_batch(_ptr(q), _ptr(k), _ptr(v), _ptr(g), float(scale), _ptr(h0),
                                  _ptr(o), _ptr(hT), B, T, H, Dk, Dv)
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return o, hT


def recurrent_head(q, k, v, g, scale: float, h0, b: int, h: int, t_end: int | None = None):
    """The C recurrence for one (b, h) of a large batch, reading float32 inputs in place.

    ``q, k, v, g`` must already be contiguous float32 numpy arrays of the full
    [B, T, H, D] shape (use ``_f32`` once and reuse). ``h0`` is the full [B,H,Dk,Dv]
    array or None. Only tokens [0, t_end) are run. Returns (o [t_end, Dv], hT [Dk, Dv]).
    """
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    t_end = T if t_end is None else int(t_end)
    for a in (q, k, v, g):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    o = np.empty((t_end, Dv), dtype=np.float64)
    hT = np.empty((Dk, Dv), dtype=np.float64)
    offk = (b * T * H + h) * Dk
    offv = (b * T * H + h) * Dv
    f32 = ctypes.sizeof(ctypes.c_float)
    base = lambda a, off: ctypes.c_void_p(a.ctypes.data + off * f32)  # noqa: E731
    h0p = None
    if h0 is not None:
        assert h0.dtype == np.float32 and h0.flags["C_CONTIGUOUS"]
        h0p = base(h0, (b * H + h) * Dk * Dv)
    rc = _load().gla_oracle_head(base(q, offk), base(k, offk), base(v, offv), base(g, offk),
                                 t_end, Dk, Dv, H * Dk, H * Dk, H * Dv, H * Dk, float(scale),
                                 h0p, _ptr(o), Dv, _ptr(hT))
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return o, hT


def recurrent_np(q, k, v, g, scale: float, h0=None):
    """Independent pure-numpy fp64 token loop of the same definition (small cases)."""
    q, k, v, g = (_f32(x).astype(np.float64) for x in (q, k, v, g))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    S = np.zeros((B, H, Dk, Dv)) if h0 is None else _f32(h0).astype(np.float64).copy()
    o = np.empty((B, T, H, Dv))
    for t in range(T):
        alpha = np.exp(g[:, t])                                # [B, H, Dk]
        S = alpha[..., None] * S + k[:, t, :, :, None] * v[:, t, :, None, :]
        o[:, t] = scale * np.einsum("bhd,bhde->bhe", q[:, t], S)
    return o, S


def chunkwise_np(q, k, v, g, scale: float, h0=None, C: int = 64):
    """fp64 chunkwise form of the same recurrence ("线性注意力GPU算子库的定义与技术解析",
    section 四: split the sequence into blocks, recur inside each block, carry the
    state from block to block, and do the in-block work as matrix products).

    Per chunk of length L (the last one may be shorter), with b_i the inclusive
    in-chunk cumulative log-gate (a Dk vector per token) and Bc = b_{L-1}:

        Q~ = q * exp(b),  K~ = k * exp(-b),  K^ = k * exp(Bc - b)
        P  = (Q~ K~^T) masked to j <= i              (decay-masked intra attention)
        O  = scale * (Q~ S + P v)                    (inter + intra)
        S <- diag(exp(Bc)) S + K^^T v                (state scan)
    """
    q, k, v, g = (_f32(x).astype(np.float64) for x in (q, k, v, g))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    S = np.zeros((B, H, Dk, Dv)) if h0 is None else _f32(h0).astype(np.float64).copy()
    o = np.empty((B, T, H, Dv))
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        L = t1 - t0
        # [B, H, L, D] views of this chunk
        qc = q[:, t0:t1].transpose(0, 2, 1, 3)
        kc = k[:, t0:t1].transpose(0, 2, 1, 3)
        vc = v[:, t0:t1].transpose(0, 2, 1, 3)
        b = np.cumsum(g[:, t0:t1].transpose(0, 2, 1, 3), axis=2)
        Bc = b[:, :, -1, :]                                   # [B, H, Dk]
        Qt = qc * np.exp(b)
        Kt = kc * np.exp(-b)
        Kh = kc * np.exp(Bc[:, :, None, :] - b)
        P = np.einsum("bhid,bhjd->bhij", Qt, Kt) * np.tril(np.ones((L, L)))
        O = scale * (np.einsum("bhid,bhde->bhie", Qt, S) + np.einsum("bhij,bhje->bhie", P, vc))
        o[:, t0:t1] = O.transpose(0, 2, 1, 3)
        S = np.exp(Bc)[..., None] * S + np.einsum("bhjd,bhje->bhde", Kh, vc)
    return o, S
