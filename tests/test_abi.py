"""The C ABI library loads, exports every symbol include/gla.h declares, and rejects bad
arguments on the host (no GPU needed: validation returns before any CUDA call).

The pointers passed here are fake device addresses. Every call must therefore be rejected by
validation, or have nothing to launch: a call that passed validation with work to do would
launch a kernel on them if a GPU were present. As a second guard, independent of how the
library validates, the module runs only where no CUDA device is visible (the host-only test
run); with a GPU present its tests are skipped."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only checks on fake device addresses: run where no GPU is visible")
    from chunkwise_recurrent_prefill_gb300 import build_ext
    from chunkwise_recurrent_prefill_gb300.gla import load_library
    build_ext.build()
    return load_library()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b((?:gla|gdn)_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert {"gla_fwd", "gla_fwd_f32", "gla_fwd_ex", "gla_last_device_status", "gdn_fwd",
            "gdn_fwd_workspace_size"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"libgla.so does not export {name}"


def test_version_and_status_strings(lib):
    assert lib.gla_version() >= 100
    for code, name in [(0, b"GLA_OK"), (3, b"GLA_ERR_UNSUPPORTED_DIM"), (7, b"GLA_ERR_DEVICE_TIMEOUT")]:
        assert lib.gla_status_string(code) == name
    assert lib.gla_status_string(999) == b"GLA_ERR_UNKNOWN"


def _call(lib, q=0x10000, k=0x20000, v=0x30000, g=0x40000, h0=None, o=0x50000, hT=None,
          B=1, T=64, H=2, Dk=128, Dv=128, io=0, opt=None):
    from chunkwise_recurrent_prefill_gb300.gla import _Options
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    opt_p = ctypes.byref(opt) if opt is not None else ctypes.POINTER(_Options)()
    return lib.gla_fwd_ex(p(q), p(k), p(v), p(g), ctypes.c_float(1.0), p(h0), p(o), p(hT),
                          B, T, H, Dk, Dv, io, opt_p, None)


# fake device addresses far apart so that no range overlaps unless a test wants it
A = dict(q=0x1000000000, k=0x2000000000, v=0x3000000000, g=0x4000000000, o=0x5000000000)


def test_null_pointer(lib):
    assert _call(lib, **{**A, "q": None}) == 1
    assert _call(lib, **{**A, "o": None}) == 1


def test_bad_shape(lib):
    assert _call(lib, **A, B=-1) == 2
    assert _call(lib, **A, T=-5) == 2
    assert _call(lib, **A, B=1 << 40, T=1 << 40) == 2


def test_misaligned(lib):
    assert _call(lib, **{**A, "k": A["k"] + 2}) == 4
    assert _call(lib, **A, hT=0x6000000008) == 4


def test_alias(lib):
    assert _call(lib, **{**A, "o": A["q"] + 64}) == 5          # o overlaps q
    assert _call(lib, **A, h0=0x6000000000, hT=0x6000000000) == 5
    assert _call(lib, **A, hT=A["o"] + 1024) == 5              # hT inside o


def test_bad_io_and_options(lib):
    from chunkwise_recurrent_prefill_gb300.gla import options
    assert _call(lib, **A, io=7) == 10
    assert _call(lib, **A, opt=options("auto", -3)) == 10


def test_unsupported_dims(lib):
    from chunkwise_recurrent_prefill_gb300.gla import options
    assert _call(lib, **A, Dk=96, opt=options("exact")) == 3
    assert _call(lib, **A, Dk=0) == 3
    assert _call(lib, **A, io=1, opt=options("tc")) == 3       # tensor cores need bf16 I/O
    assert _call(lib, **A, Dk=96, Dv=96, opt=options("tc")) == 3      # 64 or 128 only


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from chunkwise_recurrent_prefill_gb300 import gla_fwd
    x = torch.zeros(1, 4, 1, 128)
    with pytest.raises(ValueError):
        gla_fwd(x, x, x, x, 1.0)


def _step(lib, q=0x1000000000, k=0x2000000000, v=0x3000000000, g=0x4000000000,
          S=0x5000000000, o=0x6000000000, B=1, H=2, Dk=128, Dv=128, io=0):
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.gla_step(p(q), p(k), p(v), p(g), ctypes.c_float(1.0), p(S), p(o), B, H, Dk, Dv,
                        io, None)


def test_step_validation(lib):
    from chunkwise_recurrent_prefill_gb300.gla import load_library
    load_library()   # sets the argument types
    assert _step(lib, q=None) == 1                      # GLA_ERR_NULL_ARG
    assert _step(lib, S=None) == 1
    assert _step(lib, B=-1) == 2                        # GLA_ERR_BAD_SHAPE
    assert _step(lib, Dk=0) == 3                        # GLA_ERR_UNSUPPORTED_DIM
    assert _step(lib, Dv=2048) == 3
    assert _step(lib, Dv=6) == 3                        # not a multiple of 4
    assert _step(lib, v=0x3000000008) == 4              # GLA_ERR_MISALIGNED
    assert _step(lib, o=0x5000000000 + 256) == 5        # o inside S: GLA_ERR_ALIAS
    assert _step(lib, S=0x4000000000) == 5              # S over g
    assert _step(lib, io=7) == 10                       # GLA_ERR_BAD_OPTION


def _varlen(lib, cu=0x7000000000, N=2, T=128, H=2, Dk=128, Dv=128, io=0, gate=0, h0=None,
            hT=None, o=0x5000000000):
    from chunkwise_recurrent_prefill_gb300.gla import _Options
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    opt = _Options()
    opt.gate = gate
    return lib.gla_fwd_varlen(p(A["q"]), p(A["k"]), p(A["v"]), p(A["g"]), ctypes.c_float(1.0),
                              p(h0), p(o), p(hT), p(cu), N, T, H, Dk, Dv, io,
                              ctypes.byref(opt), None)


def test_varlen_validation(lib):
    from chunkwise_recurrent_prefill_gb300.gla import load_library
    load_library()   # sets the argument types
    assert _varlen(lib, cu=None) == 1                    # offsets required when N > 0
    assert _varlen(lib, N=-1) == 2
    assert _varlen(lib, cu=0x7000000002) == 4            # int32 offsets: 4-byte aligned
    assert _varlen(lib, gate=5) == 10
    # a valid shape passes validation; with no sequences (N = 0) nothing is launched, so the
    # fake addresses above are never touched (0 with a GPU, 6 or 8 without an sm_103 device)
    assert _varlen(lib, N=0, Dk=64, Dv=64, io=0) in (0, 6, 8)
    assert _varlen(lib, hT=0x1000000000) == 5            # hT over q
    assert _varlen(lib, o=0x7000000000 - 64) == 5        # o over the offsets


def _gdn(lib, q=0x1000000000, k=0x2000000000, v=0x3000000000, g=0x4000000000,
         beta=0x4800000000, h0=None, o=0x5000000000, hT=None, B=1, T=64, H=2, Dk=128, Dv=128,
         io=0, ws=0x9000000000, ws_bytes=1 << 40):
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.gdn_fwd(p(q), p(k), p(v), p(g), p(beta), ctypes.c_float(1.0), p(h0), p(o), p(hT),
                       B, T, H, Dk, Dv, io, p(ws), ws_bytes, None)


def test_gdn_validation(lib):
    from chunkwise_recurrent_prefill_gb300.gla import load_library
    load_library()   # sets the argument types
    assert _gdn(lib, beta=None) == 1                    # GLA_ERR_NULL_ARG
    assert _gdn(lib, o=None) == 1
    assert _gdn(lib, T=-1) == 2                         # GLA_ERR_BAD_SHAPE
    assert _gdn(lib, Dk=130) == 3                       # GLA_ERR_UNSUPPORTED_DIM
    assert _gdn(lib, Dk=6) == 3                         # not a multiple of 4
    assert _gdn(lib, Dv=24) == 3                        # not a multiple of 16
    assert _gdn(lib, beta=0x4800000004) == 4            # GLA_ERR_MISALIGNED
    assert _gdn(lib, o=0x4800000000) == 5               # o over beta: GLA_ERR_ALIAS
    assert _gdn(lib, hT=0x3000000000) == 5              # hT over v
    assert _gdn(lib, ws_bytes=16) == 9                  # workspace too small
    assert _gdn(lib, ws=0x9000000008) == 9              # workspace misaligned
    assert _gdn(lib, ws=0x3000000000) == 9              # workspace over v
    assert _gdn(lib, io=3) == 10                        # GLA_ERR_BAD_OPTION
    # the workspace size grows with the number of 64-token chunks and is 0 when unsupported
    one = lib.gdn_fwd_workspace_size(1, 64, 1, 128, 128)
    assert one > 0 and lib.gdn_fwd_workspace_size(2, 65, 3, 128, 128) == 2 * 2 * 3 * one
    assert lib.gdn_fwd_workspace_size(1, 64, 1, 130, 128) == 0
    assert lib.gdn_fwd_workspace_size(1, 0, 1, 128, 128) == 0
