"""GB300 (sm_103a) gated linear attention (GLA) prefill forward, and the gated delta
rule forward (gdn_fwd).

The compute runs in ``_build/libgla.so`` (CUDA kernels behind the C ABI of
``include/gla.h``); ``gla.py`` only marshals torch tensors onto it.
"""
from .gla import (  # noqa: F401
    GLAError,
    gdn_fwd,
    gdn_workspace_size,
    gla_fwd,
    gla_fwd_noalloc,
    gla_fwd_varlen,
    gla_step,
    last_device_status,
    load_library,
    workspace_size,
)
from .workloads import (  # noqa: F401
    BENCH_WORKLOAD,
    GDN_BENCH_WORKLOAD,
    GDN_WORKLOADS,
    WORKLOADS,
    Workload,
    make_gdn_inputs,
    make_inputs,
)
