"""GB300 (sm_103a) gated linear attention (GLA) prefill forward.

The compute runs in ``_build/libgla.so`` (CUDA kernels behind the C ABI of
``include/gla.h``); ``gla.py`` only marshals torch tensors onto it.
"""
from .gla import (  # noqa: F401
    GLAError,
    gla_fwd,
    gla_fwd_noalloc,
    gla_fwd_varlen,
    gla_step,
    last_device_status,
    load_library,
    workspace_size,
)
from .workloads import BENCH_WORKLOAD, WORKLOADS, Workload, make_inputs  # noqa: F401
