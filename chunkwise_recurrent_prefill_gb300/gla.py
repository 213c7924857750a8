"""Python binding of libgla.so (argument marshalling only).

Every step of the forward pass runs inside the library's CUDA kernels; this module
checks tensor dtypes/shapes/devices, allocates outputs with torch (device memory is
plumbing here) and passes raw pointers and the current CUDA stream to the C ABI
declared in ``include/gla.h``. There is no CPU or PyTorch fallback: if the library is
missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgla.so")

GLA_OK = 0
STATUS = {
    0: "GLA_OK", 1: "GLA_ERR_NULL_ARG", 2: "GLA_ERR_BAD_SHAPE", 3: "GLA_ERR_UNSUPPORTED_DIM",
    4: "GLA_ERR_MISALIGNED", 5: "GLA_ERR_ALIAS", 6: "GLA_ERR_LAUNCH",
    7: "GLA_ERR_DEVICE_TIMEOUT", 8: "GLA_ERR_UNSUPPORTED_DEVICE", 9: "GLA_ERR_WORKSPACE",
    10: "GLA_ERR_BAD_OPTION", 11: "GLA_ERR_BAD_SEQLENS",
}
PATHS = {"auto": 0, "exact": 1, "tc": 2}
GATES = {"key": 0, "scalar": 1}
IO_BF16, IO_F32 = 0, 1


class GLAError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


class _Options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("seq_splits", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("gate", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgla.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libgla.so is not built ({path}); run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            vp, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
            sig = [vp, vp, vp, vp, f32, vp, vp, vp, i64, i64, i64, i64, i64]
            lib.gla_fwd.argtypes = sig + [vp]
            lib.gla_fwd_f32.argtypes = sig + [vp]
            lib.gla_fwd_ex.argtypes = sig + [ctypes.c_int, ctypes.POINTER(_Options), vp]
            for f in (lib.gla_fwd, lib.gla_fwd_f32, lib.gla_fwd_ex):
                f.restype = ctypes.c_int
            lib.gla_step.argtypes = [vp, vp, vp, vp, f32, vp, vp, i64, i64, i64, i64,
                                     ctypes.c_int, vp]
            lib.gla_fwd_varlen.argtypes = [vp, vp, vp, vp, f32, vp, vp, vp, vp, i64, i64, i64,
                                           i64, i64, ctypes.c_int, ctypes.POINTER(_Options), vp]
            lib.gla_fwd_varlen.restype = ctypes.c_int
            lib.gla_step.restype = ctypes.c_int
            lib.gla_fwd_noalloc.argtypes = sig + [ctypes.c_int, vp]
            lib.gla_fwd_noalloc.restype = ctypes.c_int
            lib.gla_fwd_workspace_size.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int,
                                                   ctypes.POINTER(_Options)]
            lib.gla_fwd_workspace_size.restype = ctypes.c_size_t
            lib.gla_last_device_status.argtypes = [vp]
            lib.gla_last_device_status.restype = ctypes.c_int
            lib.gla_status_string.argtypes = [ctypes.c_int]
            lib.gla_status_string.restype = ctypes.c_char_p
            lib.gla_path_for.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int,
                                         ctypes.POINTER(_Options)]
            lib.gla_path_for.restype = ctypes.c_int
            lib.gla_last_error_detail.argtypes = []
            lib.gla_last_error_detail.restype = ctypes.c_char_p
            lib.gla_launch_counter.argtypes = []
            lib.gla_launch_counter.restype = ctypes.c_uint64
            lib.gla_workspace_allocations.argtypes = []
            lib.gla_workspace_allocations.restype = ctypes.c_uint64
            lib.gla_version.argtypes = []
            lib.gla_version.restype = ctypes.c_int
            lib.gdn_fwd.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp, i64, i64, i64, i64, i64,
                                    ctypes.c_int, vp, ctypes.c_size_t, vp]
            lib.gdn_fwd.restype = ctypes.c_int
            lib.gdn_fwd_workspace_size.argtypes = [i64, i64, i64, i64, i64]
            lib.gdn_fwd_workspace_size.restype = ctypes.c_size_t
            _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def options(path: str = "auto", seq_splits: int = 0, workspace: torch.Tensor | None = None,
            gate: str = "key"):
    opt = _Options()
    opt.path = PATHS[path]
    opt.gate = GATES[gate]
    opt.seq_splits = int(seq_splits)
    opt.workspace = None if workspace is None else workspace.data_ptr()
    opt.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return opt


def workspace_size(B, T, H, Dk=128, Dv=128, io="bf16", path="auto", seq_splits=0) -> int:
    opt = options(path, seq_splits)
    return int(load_library().gla_fwd_workspace_size(B, T, H, Dk, Dv,
                                                      IO_BF16 if io == "bf16" else IO_F32,
                                                      ctypes.byref(opt)))


def path_for(B, T, H, Dk=128, Dv=128, io="bf16", path="auto") -> str | None:
    """Name of the path gla_fwd would run ("exact" / "tc"), or None if unsupported."""
    opt = options(path)
    r = int(load_library().gla_path_for(B, T, H, Dk, Dv, IO_BF16 if io == "bf16" else IO_F32,
                                        ctypes.byref(opt)))
    return {1: "exact", 2: "tc"}.get(r)


def gla_fwd(q, k, v, g, scale: float, h0=None, *, o=None, hT=None, return_state: bool = False,
            path: str = "auto", seq_splits: int = 0, workspace=None, gate: str = "key",
            stream=None):
    """GLA prefill forward through ``gla_fwd_ex``.

    q, k: [B,T,H,Dk]; v: [B,T,H,Dv] (all bf16, or all float32); g: float32 log-gates,
    [B,T,H,Dk] (``gate="key"``) or [B,T,H] (``gate="scalar"``: one gate per token and head);
    h0: [B,H,Dk,Dv] float32 or None. Outputs o (same dtype as q) and, when ``return_state``
    or ``hT`` is given, the float32 final state. Returns (o, hT|None). Asynchronous on
    ``stream`` (default: torch's current stream).
    """
    lib = load_library()
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q/k/v must be bfloat16 or float32")
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(q, "q", q.dtype, (B, T, H, Dk), dev)
    _check(k, "k", q.dtype, (B, T, H, Dk), dev)
    _check(v, "v", q.dtype, (B, T, H, Dv), dev)
    _check(g, "g", torch.float32, (B, T, H, Dk) if gate == "key" else (B, T, H), dev)
    if h0 is not None:
        _check(h0, "h0", torch.float32, (B, H, Dk, Dv), dev)
    if o is None:
        o = torch.empty((B, T, H, Dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", q.dtype, (B, T, H, Dv), dev)
    if hT is None and return_state:
        hT = torch.empty((B, H, Dk, Dv), dtype=torch.float32, device=dev)
    elif hT is not None:
        _check(hT, "hT", torch.float32, (B, H, Dk, Dv), dev)
    opt = options(path, seq_splits, workspace, gate)
    io = IO_BF16 if q.dtype == torch.bfloat16 else IO_F32
    with torch.cuda.device(dev):
        rc = lib.gla_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), ctypes.c_float(scale), _ptr(h0),
                            _ptr(o), _ptr(hT), B, T, H, Dk, Dv, io, ctypes.byref(opt),
                            _stream_handle(stream))
    if rc != GLA_OK:
        detail = lib.gla_last_error_detail().decode() if rc in (6, 9) else ""
        raise GLAError(rc, "gla_fwd_ex", detail)
    return o, hT


def gla_fwd_noalloc(q, k, v, g, scale: float, h0=None, *, o, hT=None, seq_splits: int = 0,
                    stream=None):
    """GLA prefill forward through ``gla_fwd_noalloc``: bf16 q, k, v, o; the library takes
    its scratch from a fixed array compiled into it and allocates no device memory. The
    caller passes the outputs (``o`` and, optionally, ``hT``) already allocated. Calls that
    overlap on the GPU share that array and race; keep them on one stream. Returns (o, hT).
    """
    lib = load_library()
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for t, name, shape in ((q, "q", (B, T, H, Dk)), (k, "k", (B, T, H, Dk)),
                           (v, "v", (B, T, H, Dv)), (o, "o", (B, T, H, Dv))):
        _check(t, name, torch.bfloat16, shape, dev)
    _check(g, "g", torch.float32, (B, T, H, Dk), dev)
    if h0 is not None:
        _check(h0, "h0", torch.float32, (B, H, Dk, Dv), dev)
    if hT is not None:
        _check(hT, "hT", torch.float32, (B, H, Dk, Dv), dev)
    with torch.cuda.device(dev):
        rc = lib.gla_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), ctypes.c_float(scale),
                                 _ptr(h0), _ptr(o), _ptr(hT), B, T, H, Dk, Dv, int(seq_splits),
                                 _stream_handle(stream))
    if rc != GLA_OK:
        detail = lib.gla_last_error_detail().decode() if rc in (6, 9) else ""
        raise GLAError(rc, "gla_fwd_noalloc", detail)
    return o, hT


def gla_fwd_varlen(q, k, v, g, scale: float, cu_seqlens, h0=None, *, o=None, hT=None,
                   return_state: bool = False, path: str = "auto", gate: str = "key",
                   stream=None):
    """GLA prefill over packed sequences through ``gla_fwd_varlen``.

    q, k: [T,H,Dk]; v: [T,H,Dv] (all bf16, or all float32); g: float32 [T,H,Dk] (or [T,H]
    with ``gate="scalar"``); cu_seqlens: int32 [N+1] on the device (sequence i is tokens
    cu_seqlens[i] .. cu_seqlens[i+1]-1); h0: [N,H,Dk,Dv] float32 or None. Returns (o, hT|None).
    """
    lib = load_library()
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q/k/v must be bfloat16 or float32")
    T, H, Dk = q.shape
    Dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(k, "k", q.dtype, (T, H, Dk), dev)
    _check(v, "v", q.dtype, (T, H, Dv), dev)
    _check(g, "g", torch.float32, (T, H, Dk) if gate == "key" else (T, H), dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    if h0 is not None:
        _check(h0, "h0", torch.float32, (N, H, Dk, Dv), dev)
    if o is None:
        o = torch.empty((T, H, Dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", q.dtype, (T, H, Dv), dev)
    if hT is None and return_state:
        hT = torch.empty((N, H, Dk, Dv), dtype=torch.float32, device=dev)
    elif hT is not None:
        _check(hT, "hT", torch.float32, (N, H, Dk, Dv), dev)
    opt = options(path, 0, None, gate)
    io = IO_BF16 if q.dtype == torch.bfloat16 else IO_F32
    with torch.cuda.device(dev):
        rc = lib.gla_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(g), ctypes.c_float(scale),
                                _ptr(h0), _ptr(o), _ptr(hT), _ptr(cu_seqlens), N, T, H, Dk, Dv,
                                io, ctypes.byref(opt), _stream_handle(stream))
    if rc != GLA_OK:
        detail = lib.gla_last_error_detail().decode() if rc == 6 else ""
        raise GLAError(rc, "gla_fwd_varlen", detail)
    return o, hT


def gla_step(q, k, v, g, scale: float, S, *, o=None, stream=None):
    """One decode step through ``gla_step``: q, k [B,H,Dk]; v [B,H,Dv] (all bf16, or all
    float32); g [B,H,Dk] float32 log-gates; S [B,H,Dk,Dv] float32, updated in place
    (S <- diag(exp(g)) S + k^T v). Returns o = scale q S [B,H,Dv] (same dtype as q)."""
    lib = load_library()
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q/k/v must be bfloat16 or float32")
    B, H, Dk = q.shape
    Dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(k, "k", q.dtype, (B, H, Dk), dev)
    _check(v, "v", q.dtype, (B, H, Dv), dev)
    _check(g, "g", torch.float32, (B, H, Dk), dev)
    _check(S, "S", torch.float32, (B, H, Dk, Dv), dev)
    if o is None:
        o = torch.empty((B, H, Dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", q.dtype, (B, H, Dv), dev)
    io = IO_BF16 if q.dtype == torch.bfloat16 else IO_F32
    with torch.cuda.device(dev):
        rc = lib.gla_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), ctypes.c_float(scale), _ptr(S),
                          _ptr(o), B, H, Dk, Dv, io, _stream_handle(stream))
    if rc != GLA_OK:
        detail = lib.gla_last_error_detail().decode() if rc == 6 else ""
        raise GLAError(rc, "gla_step", detail)
    return o


def gdn_workspace_size(B: int, T: int, H: int, Dk: int, Dv: int) -> int:
    """Bytes of device workspace ``gdn_fwd`` needs for this shape (0 if unsupported)."""
    return int(load_library().gdn_fwd_workspace_size(B, T, H, Dk, Dv))


def gdn_fwd(q, k, v, g, beta, scale: float, h0=None, *, o=None, hT=None,
            return_state: bool = False, workspace: torch.Tensor | None = None, stream=None):
    """Gated delta rule forward through ``gdn_fwd``.

    q, k: [B,T,H,Dk]; v: [B,T,H,Dv] (all bf16, or all float32); g (log-gates) and beta
    (write strengths): float32 [B,T,H]; h0: [B,H,Dk,Dv] float32 or None. ``workspace``: a
    CUDA tensor of at least ``gdn_workspace_size`` bytes, or None for the library's own.
    Returns (o, hT|None).
    """
    lib = load_library()
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q/k/v must be bfloat16 or float32")
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(k, "k", q.dtype, (B, T, H, Dk), dev)
    _check(v, "v", q.dtype, (B, T, H, Dv), dev)
    _check(g, "g", torch.float32, (B, T, H), dev)
    _check(beta, "beta", torch.float32, (B, T, H), dev)
    if h0 is not None:
        _check(h0, "h0", torch.float32, (B, H, Dk, Dv), dev)
    if o is None:
        o = torch.empty((B, T, H, Dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", q.dtype, (B, T, H, Dv), dev)
    if hT is None and return_state:
        hT = torch.empty((B, H, Dk, Dv), dtype=torch.float32, device=dev)
    elif hT is not None:
        _check(hT, "hT", torch.float32, (B, H, Dk, Dv), dev)
    ws, ws_bytes = None, 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the inputs' device")
        ws, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    io = IO_BF16 if q.dtype == torch.bfloat16 else IO_F32
    with torch.cuda.device(dev):
        rc = lib.gdn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), ctypes.c_float(scale),
                         _ptr(h0), _ptr(o), _ptr(hT), B, T, H, Dk, Dv, io, ws, ws_bytes,
                         _stream_handle(stream))
    if rc != GLA_OK:
        detail = lib.gla_last_error_detail().decode() if rc in (6, 9) else ""
        raise GLAError(rc, "gdn_fwd", detail)
    return o, hT


def launch_counter() -> int:
    """Kernel launches the library has issued in this process."""
    return int(load_library().gla_launch_counter())


def workspace_allocations() -> int:
    """Device allocations the library has made for its per-stream workspaces so far."""
    return int(load_library().gla_workspace_allocations())


def last_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load_library().gla_last_device_status(_stream_handle(stream)))
