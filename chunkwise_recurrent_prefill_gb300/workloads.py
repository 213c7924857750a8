"""Seeded synthetic inputs for the GLA prefill forward pass.

This module only draws random numbers and names workloads. It holds none of the
method's arithmetic, and it is the one module that both the CUDA path's tests/bench
and the oracle consume.

Recipe (the same for every workload; the pages measure on random shapes, not on a
dataset — "Linear Attention 在 GPU 上到底慢在哪", section 实验设计):

* ``torch.Generator('cpu').manual_seed(seed)``; draw order q, k, v, u, then h0, each a
  float32 ``randn`` of its full shape.
* q, k, v ~ N(0, 1), shapes [B, T, H, Dk] / [B, T, H, Dv].
* log-gate g = logsigmoid(u) / 16 with u ~ N(0, 1), one value per token, head and key
  dimension (one per token and head for the scalar-gate workloads), kept in float32.
* h0 = 0.02 * N(0, 1) (standard deviation 0.02) where a workload carries a state in.
* scale = Dk ** -0.5.
* bf16 workloads round q, k, v to bf16 after drawing; g and h0 stay float32.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    Dk: int = 128
    Dv: int = 128
    io: str = "bf16"          # dtype of q, k, v, o: "bf16" or "f32"
    seed: int = 0
    with_h0: bool = False     # draw a nonzero initial state
    want_hT: bool = False     # the workload returns the final state
    gate: str = "key"         # "key": g [B,T,H,Dk]; "scalar": g [B,T,H] (one gate per token/head)

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five parity workloads (sizes from the pages' test grid and latency table).
WORKLOADS = {
    "f32_B1_H2_T512": Workload("f32_B1_H2_T512", B=1, T=512, H=2, io="f32", seed=0),
    "bf16_B1_H16_T4096": Workload("bf16_B1_H16_T4096", B=1, T=4096, H=16, seed=1),
    "bf16_B1_H16_T16384": Workload("bf16_B1_H16_T16384", B=1, T=16384, H=16, seed=2),
    "bf16_B4_H16_T16384": Workload("bf16_B4_H16_T16384", B=4, T=16384, H=16, seed=2),
    "bf16_B16_H16_T4096": Workload("bf16_B16_H16_T4096", B=16, T=4096, H=16, seed=3),
    "bf16_B1_H16_T131072_h0": Workload("bf16_B1_H16_T131072_h0", B=1, T=131072, H=16, seed=4,
                                       with_h0=True, want_hT=True),
    # the scalar-per-head gate variant on the bench shape (one log-gate per token and head)
    "bf16_B1_H16_T16384_scalar": Workload("bf16_B1_H16_T16384_scalar", B=1, T=16384, H=16,
                                          seed=6, gate="scalar"),
    # head dims 64 on the bench shape (heads run in pairs on the tensor cores)
    "bf16_B1_H16_T16384_D64": Workload("bf16_B1_H16_T16384_D64", B=1, T=16384, H=16, Dk=64,
                                       Dv=64, seed=7, with_h0=True, want_hT=True),
}

# The workload the throughput metric is quoted on (B=1, H=16, T=16K, D=128, bf16).
BENCH_WORKLOAD = "bf16_B1_H16_T16384"


def make_inputs(w: Workload, device: str | torch.device = "cpu") -> dict:
    """Draw the inputs of workload ``w`` on the CPU generator and move them to ``device``.

    Returns a dict with q, k, v (bf16 or float32), g (float32), h0 (float32 or None)
    and scale (python float).
    """
    gen = torch.Generator("cpu").manual_seed(w.seed)
    io = torch.bfloat16 if w.io == "bf16" else torch.float32

    def draw(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    q = draw(w.B, w.T, w.H, w.Dk).to(io)
    k = draw(w.B, w.T, w.H, w.Dk).to(io)
    v = draw(w.B, w.T, w.H, w.Dv).to(io)
    g = F.logsigmoid(draw(w.B, w.T, w.H, w.Dk) if w.gate == "key" else draw(w.B, w.T, w.H)) / 16.0
    h0 = draw(w.B, w.H, w.Dk, w.Dv) * 0.02 if w.with_h0 else None
    out = dict(q=q, k=k, v=v, g=g, h0=h0, scale=float(w.Dk) ** -0.5)
    if str(device) != "cpu":
        for key in ("q", "k", "v", "g", "h0"):
            if out[key] is not None:
                out[key] = out[key].to(device)
    return out


def small(name: str, B: int, T: int, H: int, io: str = "bf16", seed: int = 0,
          with_h0: bool = False, Dk: int = 128, Dv: int = 128, gate: str = "key") -> Workload:
    """An ad-hoc workload with the same distributions (tests use these for edge cases)."""
    return Workload(name, B=B, T=T, H=H, Dk=Dk, Dv=Dv, io=io, seed=seed, with_h0=with_h0,
                    want_hT=True, gate=gate)


# Gated-delta-rule workloads (same shapes as the GLA bench and parity cases). Recipe:
# ``torch.Generator('cpu').manual_seed(seed)``; draw order q, k, v, u (gate), w (write
# strength), then h0. q and k ~ N(0, 1) rows divided by their L2 norm (unit-norm queries
# and keys, the regime the delta write assumes), v ~ N(0, 1), g = logsigmoid(u) / 16 and
# beta = sigmoid(w) with u, w ~ N(0, 1), one value each per token and head; h0 as above.
GDN_WORKLOADS = {
    "gdn_f32_B1_H2_T512": Workload("gdn_f32_B1_H2_T512", B=1, T=512, H=2, io="f32", seed=10),
    "gdn_bf16_B1_H16_T4096": Workload("gdn_bf16_B1_H16_T4096", B=1, T=4096, H=16, seed=11),
    "gdn_bf16_B1_H16_T16384": Workload("gdn_bf16_B1_H16_T16384", B=1, T=16384, H=16, seed=12),
    "gdn_bf16_B16_H16_T4096_h0": Workload("gdn_bf16_B16_H16_T4096_h0", B=16, T=4096, H=16,
                                          seed=13, with_h0=True, want_hT=True),
}
GDN_BENCH_WORKLOAD = "gdn_bf16_B1_H16_T16384"


def make_gdn_inputs(w: Workload, device: str | torch.device = "cpu") -> dict:
    """Inputs of a gated-delta-rule workload: q, k, v (io dtype), g, beta [B,T,H] float32,
    h0 (float32 or None), scale."""
    gen = torch.Generator("cpu").manual_seed(w.seed)
    io = torch.bfloat16 if w.io == "bf16" else torch.float32

    def draw(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True)

    q = unit(draw(w.B, w.T, w.H, w.Dk)).to(io)
    k = unit(draw(w.B, w.T, w.H, w.Dk)).to(io)
    v = draw(w.B, w.T, w.H, w.Dv).to(io)
    g = F.logsigmoid(draw(w.B, w.T, w.H)) / 16.0
    beta = torch.sigmoid(draw(w.B, w.T, w.H))
    h0 = draw(w.B, w.H, w.Dk, w.Dv) * 0.02 if w.with_h0 else None
    out = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, scale=float(w.Dk) ** -0.5)
    if str(device) != "cpu":
        for key in ("q", "k", "v", "g", "beta", "h0"):
            if out[key] is not None:
                out[key] = out[key].to(device)
    return out


# Decode-step workload: one token for each of B sequences and H heads on a resident state
# (the step after prefill). Same recipe: q, k, v, u, then the state S = 0.02 * N(0, 1).
# B = 256 makes the state (268 MB) larger than the 129 MB L2, so a step's state write-back
# cannot stay in L2 past the step.
STEP_WORKLOAD = dict(name="decode_B256_H16_D128", B=256, H=16, D=128, io="bf16", seed=5)


def make_step_inputs(B: int, H: int, D: int, io: str = "bf16", seed: int = 0,
                     device: torch.device | str = "cpu") -> dict:
    """q, k [B,H,D], v [B,H,D] (io dtype), g [B,H,D] float32, S [B,H,D,D] float32."""
    gen = torch.Generator("cpu").manual_seed(seed)
    dt = torch.bfloat16 if io == "bf16" else torch.float32
    q = torch.randn(B, H, D, generator=gen).to(dt)
    k = torch.randn(B, H, D, generator=gen).to(dt)
    v = torch.randn(B, H, D, generator=gen).to(dt)
    g = F.logsigmoid(torch.randn(B, H, D, generator=gen)) / 16
    S = 0.02 * torch.randn(B, H, D, D, generator=gen)
    x = dict(q=q, k=k, v=v, g=g, S=S, scale=D ** -0.5)
    return {n: (t.to(device) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}

