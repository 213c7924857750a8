"""GPU parity of the gated delta rule forward (gdn_fwd) against the fp64 oracle.

Small cases compare every output element; the full-size workloads compare sampled heads,
which the oracle's token loop runs one by one. Tolerances are those of ``tests/parity.py``.
"""
import numpy as np
import pytest
import torch

from parity import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(x, want_state=True, **kw):
    from chunkwise_recurrent_prefill_gb300 import gdn_fwd, last_device_status
    o, hT = gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"],
                    return_state=want_state, **kw)
    torch.cuda.synchronize()
    assert last_device_status() == 0
    return o, hT


def _oracle(x):
    from oracle import gdn_ref
    cpu = lambda t: None if t is None else t.cpu()   # noqa: E731
    return gdn_ref.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]), cpu(x["beta"]),
                             x["scale"], cpu(x["h0"]))


def _inputs(B, T, H, io, seed, h0=False, Dk=128, Dv=128):
    from chunkwise_recurrent_prefill_gb300.workloads import make_gdn_inputs, small
    return make_gdn_inputs(small("gdn", B=B, T=T, H=H, io=io, seed=seed, with_h0=h0, Dk=Dk, Dv=Dv),
                           DEV)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("B,T,H,h0", [(1, 64, 2, False), (1, 200, 3, True), (2, 129, 2, True),
                                      (1, 1, 2, True), (1, 63, 1, False), (2, 700, 4, True),
                                      (1, 1700, 1, True), (1, 2048, 2, True), (2, 1500, 1, False)])
def test_small_cases(io, B, T, H, h0):
    """bf16 at head dims 128 runs the tensor-core kernels; with few heads and enough chunks
    their scan splits the sequence (T=1700, H=1: 3 segments, the last ending in a ragged
    chunk; T=2048, H=2: 4 segments; B=2, T=1500: 3 segments per sequence, no h0)."""
    x = _inputs(B, T, H, io, seed=T * 7 + B + H, h0=h0)
    o, hT = _run(x)
    o_ref, h_ref = _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, io, "o")
    assert_close(hT.cpu().numpy(), h_ref, io, "hT")


@pytest.mark.parametrize("Dk,Dv", [(64, 64), (128, 64), (64, 128), (32, 48), (12, 16), (4, 16)])
def test_head_dims(Dk, Dv):
    x = _inputs(2, 150, 2, "f32", seed=Dk * 3 + Dv, h0=True, Dk=Dk, Dv=Dv)
    o, hT = _run(x)
    o_ref, h_ref = _oracle(x)
    assert_close(o.cpu().numpy(), o_ref, "f32", f"o[{Dk}x{Dv}]")
    assert_close(hT.cpu().numpy(), h_ref, "f32", f"hT[{Dk}x{Dv}]")


def test_f32_config_workload():
    """B=1, H=2, T=512, D=128, fp32 I/O: every element at the fp32 tolerance."""
    from chunkwise_recurrent_prefill_gb300.workloads import GDN_WORKLOADS, make_gdn_inputs
    x = make_gdn_inputs(GDN_WORKLOADS["gdn_f32_B1_H2_T512"], DEV)
    o, hT = _run(x)
    o_ref, h_ref = _oracle(x)
    assert_close(o.cpu().numpy(), o_ref, "f32", "o")
    assert_close(hT.cpu().numpy(), h_ref, "f32", "hT")


def test_bf16_T4096_workload():
    """B=1, H=16, T=4096 bf16: every element of every head."""
    from chunkwise_recurrent_prefill_gb300.workloads import GDN_WORKLOADS, make_gdn_inputs
    x = make_gdn_inputs(GDN_WORKLOADS["gdn_bf16_B1_H16_T4096"], DEV)
    o, hT = _run(x)
    o_ref, h_ref = _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", "o")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", "hT")


@pytest.mark.parametrize("name", ["gdn_bf16_B1_H16_T16384", "gdn_bf16_B16_H16_T4096_h0"])
def test_full_size_every_head(name):
    """The bench-size workloads in the bench's launch configuration: every output element of
    every (batch, head) against the C token loop of the oracle (fp64, OpenMP over the heads)."""
    from oracle import gdn_ref
    from chunkwise_recurrent_prefill_gb300.workloads import GDN_WORKLOADS, make_gdn_inputs
    x = make_gdn_inputs(GDN_WORKLOADS[name], DEV)
    o, hT = _run(x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    o_ref, h_ref = gdn_ref.recurrent_c(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]),
                                       cpu(x["beta"]), x["scale"], cpu(x["h0"]))
    eo = assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"{name} o")
    eh = assert_close(hT.cpu().numpy(), h_ref, "bf16", f"{name} hT")
    print(f"\nparity {name}: o max/mean rel {eo[0]:.3e}/{eo[1]:.3e}  "
          f"hT max/mean rel {eh[0]:.3e}/{eh[1]:.3e}")


def test_state_carry_on_gpu():
    """Running [0, T) equals running [0, T1) and then [T1, T) from the returned state."""
    x = _inputs(2, 300, 2, "f32", seed=5, h0=True)
    o, hT = _run(x)
    sl = lambda a, b: {**x, **{n: x[n][:, a:b].contiguous() for n in ("q", "k", "v", "g", "beta")}}  # noqa: E731
    xa = sl(0, 130)
    oa, ha = _run(xa)
    xb = {**sl(130, 300), "h0": ha}
    ob, hb = _run(xb)
    assert_close(torch.cat([oa, ob], 1).cpu().numpy(), o.cpu().numpy().astype(np.float64), "f32", "o")
    assert_close(hb.cpu().numpy(), hT.cpu().numpy().astype(np.float64), "f32", "hT")


def test_caller_workspace_and_determinism():
    from chunkwise_recurrent_prefill_gb300 import GLAError, gdn_fwd, gdn_workspace_size
    x = _inputs(1, 333, 3, "bf16", seed=21, h0=True)
    o1, h1 = _run(x)
    o2, h2 = _run(x)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)            # no atomics: bit-identical
    need = gdn_workspace_size(1, 333, 3, 128, 128)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    o3, h3 = _run(x, workspace=ws)
    assert torch.equal(o1, o3) and torch.equal(h1, h3)
    with pytest.raises(GLAError) as e:
        gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"],
                workspace=ws[: need - 16])
    assert e.value.status == 9                                   # GLA_ERR_WORKSPACE
    # a split scan (2 heads of 2048 tokens: 4 segments) keeps its segment arrays in the
    # caller's workspace too: the reported size holds them, and the results are identical
    x = _inputs(1, 2048, 2, "bf16", seed=22, h0=True)
    o1, h1 = _run(x)
    need = gdn_workspace_size(1, 2048, 2, 128, 128)
    ws = torch.full((need,), 255, dtype=torch.uint8, device=DEV)   # stale contents must not matter
    o3, h3 = _run(x, workspace=ws)
    assert torch.equal(o1, o3) and torch.equal(h1, h3)


def test_empty_and_no_state():
    from chunkwise_recurrent_prefill_gb300 import gdn_fwd
    x = _inputs(1, 0, 2, "bf16", seed=1)
    o, hT = gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"])
    assert o.shape == (1, 0, 2, 128) and hT is None
    # no tokens: hT is the initial state (zero without one)
    x = _inputs(2, 0, 3, "f32", seed=4, h0=True)
    o, hT = gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"],
                    return_state=True)
    torch.cuda.synchronize()
    assert o.shape == (2, 0, 3, 128) and torch.equal(hT, x["h0"])
    hT = torch.full((2, 3, 128, 128), 7.0, device=DEV)
    gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], None, hT=hT)
    torch.cuda.synchronize()
    assert not hT.any()
    x = _inputs(1, 96, 2, "bf16", seed=2)
    o, hT = _run(x, want_state=False)
    assert hT is None
    o_ref, _ = _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", "o")


def test_readback_property_on_gpu():
    """Unit keys, beta = 1, queries = keys, scale 1: each output returns its own value
    (the delta write's defining property), through the whole chunk machinery."""
    from chunkwise_recurrent_prefill_gb300 import gdn_fwd
    gen = torch.Generator("cpu").manual_seed(3)
    B, T, H, D = 1, 256, 2, 64
    k = torch.randn(B, T, H, D, generator=gen)
    k = (k / k.norm(dim=-1, keepdim=True)).to(DEV)
    v = torch.randn(B, T, H, D, generator=gen).to(DEV)
    g = (-0.1 * torch.rand(B, T, H, generator=gen)).to(DEV)
    beta = torch.ones(B, T, H, device=DEV)
    o, _ = gdn_fwd(k, k, v, g, beta, 1.0)
    torch.cuda.synchronize()
    err = (o - v).abs().max().item() / v.abs().max().item()
    assert err < 1e-4, err


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_degenerate_gates(io):
    """Full forgetting (g = -1e4: every in-chunk decay underflows to 0, and the masked
    exponentials above the diagonal overflow, which must never reach a product) and no
    writes (beta = 0: the state only decays), against the oracle."""
    x = _inputs(1, 1600, 2, io, seed=31, h0=True)   # bf16: a 3-segment split scan
    xf = {**x, "g": torch.full_like(x["g"], -1e4)}
    o, hT = _run(xf)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    o_ref, h_ref = _oracle(xf)
    assert_close(o.float().cpu().numpy(), o_ref, io, "o (g = -1e4)")
    assert_close(hT.cpu().numpy(), h_ref, io, "hT (g = -1e4)")
    xb = {**x, "beta": torch.zeros_like(x["beta"])}
    o, hT = _run(xb)
    o_ref, h_ref = _oracle(xb)
    assert_close(o.float().cpu().numpy(), o_ref, io, "o (beta = 0)")
    assert_close(hT.cpu().numpy(), h_ref, io, "hT (beta = 0)")
