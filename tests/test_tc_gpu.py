"""GPU parity of the tensor-core path (tcgen05/TMEM/TMA) against the fp64 oracle.

bf16 tolerances: max|d| <= 1.5e-2 max|ref|, sum|d| / sum|ref| <= 5e-3, for o and hT.
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


def _run(x, path="tc", seq_splits=0):
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                    path=path, seq_splits=seq_splits)
    torch.cuda.synchronize()
    assert last_device_status() == 0
    return o, hT


def _oracle(x):
    import oracle
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    return oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]), x["scale"],
                            cpu(x["h0"]))


def _inputs(B, T, H, seed=0, with_h0=True):
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    return make_inputs(small("tc", B=B, T=T, H=H, io="bf16", seed=seed, with_h0=with_h0), DEV)


def _check(x, seq_splits=0):
    o, hT = _run(x, seq_splits=seq_splits)
    o_ref, h_ref = _oracle(x)
    a = assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o(splits={seq_splits})")
    b = assert_close(hT.cpu().numpy(), h_ref, "bf16", f"hT(splits={seq_splits})")
    return a, b


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 512, 1000])
@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_tc_small_ragged(T, splits):
    _check(_inputs(B=2, T=T, H=2, seed=T + splits), seq_splits=splits)


@pytest.mark.parametrize("T", [1, 2, 5, 63])
def test_tc_few_tokens(T):
    """Fewer tokens than one chunk with the tensor-core path requested explicitly: the call
    runs the exact kernel (each output would otherwise be a handful of bf16-rounded decayed
    products with nothing to average the rounding), so the stated bf16 bounds hold."""
    _check(_inputs(B=2, T=T, H=2, seed=T + 1), seq_splits=1)


def test_default_path_short_sequences_exact():
    from chunkwise_recurrent_prefill_gb300.gla import path_for
    assert path_for(1, 63, 16) == "exact" and path_for(1, 64, 16) == "tc"


@pytest.mark.parametrize("B,T,H", [(1, 8192, 1), (1, 20000, 2), (3, 3000, 5)])
def test_tc_auto_split_many_segments(B, T, H):
    """Few heads: the automatic split gives many short segments (128 one-chunk segments at
    B*H = 1), so the state pass, the scan over up to 127 segment states and the output pass
    all run at their widest."""
    from chunkwise_recurrent_prefill_gb300.gla import workspace_size
    assert workspace_size(B, T, H) > 0
    _check(_inputs(B=B, T=T, H=H, seed=T + H), seq_splits=0)


def test_tc_no_h0():
    _check(_inputs(B=1, T=333, H=3, seed=8, with_h0=False), seq_splits=2)


def test_tc_split_invariance():
    """Different sequence splits give the same numbers up to bf16 operand rounding."""
    x = _inputs(B=1, T=2048, H=4, seed=21)
    o1, h1 = _run(x, seq_splits=1)
    for s in (2, 5, 16):
        o2, h2 = _run(x, seq_splits=s)
        d = (o1.float() - o2.float()).abs().max().item() / o1.float().abs().max().item()
        assert d < 1e-2, (s, d)
        dh = (h1 - h2).abs().max().item() / h1.abs().max().item()
        assert dh < 1e-2, (s, dh)


@pytest.mark.parametrize("name", ["bf16_B1_H16_T4096", "bf16_B1_H16_T16384",
                                  "bf16_B4_H16_T16384", "bf16_B16_H16_T4096",
                                  "bf16_B1_H16_T131072_h0"])
def test_tc_parity_workload(name):
    """Every output of the full-size parity workloads, element by element, in the launch
    configuration the bench times (automatic sequence split)."""
    from chunkwise_recurrent_prefill_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    x = make_inputs(w, DEV)
    o, hT = _run(x)
    o_ref, h_ref = _oracle(x)
    eo = assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"{name} o")
    eh = assert_close(hT.cpu().numpy(), h_ref, "bf16", f"{name} hT")
    print(f"\nparity {name}: o max/mean rel {eo[0]:.3e}/{eo[1]:.3e}  "
          f"hT max/mean rel {eh[0]:.3e}/{eh[1]:.3e}")


def _extreme(x, kind):
    g = x["g"]
    if kind == "forget":
        x["g"] = torch.full_like(g, -1e4)
    elif kind == "no_decay":
        x["g"] = torch.zeros_like(g)
    elif kind == "tiny":
        x["g"] = -1e-8 * torch.ones_like(g)
    elif kind == "strong":
        x["g"] = -5.0 * torch.rand_like(g)
    elif kind == "mixed":
        x["g"] = torch.where(torch.rand_like(g) < 0.02, torch.full_like(g, -200.0), g)
    elif kind == "renorm":       # ~-23 log2 units per chunk: renormalisation every ~3 chunks
        x["g"] = -0.5 * torch.rand_like(g)
    elif kind == "one_chunk_extreme":
        g[:, 64:128] = -3.0
        x["g"] = g
    elif kind == "big_values":
        for key in ("q", "k", "v"):
            x[key] = (x[key].float() * 30).to(x[key].dtype)
    return x


@pytest.mark.parametrize("kind", ["forget", "no_decay", "tiny", "strong", "mixed", "renorm",
                                  "one_chunk_extreme", "big_values"])
def test_tc_extreme_gates(kind):
    x = _extreme(_inputs(B=1, T=700, H=2, seed=3), kind)
    o, hT = _run(x, seq_splits=2)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    o_ref, h_ref = _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o[{kind}]")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", f"hT[{kind}]")


def test_tc_nan_propagates():
    """A NaN in v reaches every output it feeds and the final state. On the tensor-core
    path it also reaches the earlier tokens of its own 64-token chunk (the masked product
    0 * NaN inside the P.V MMA is NaN); outputs of earlier chunks stay finite."""
    x = _inputs(B=1, T=200, H=1, seed=1, with_h0=False)
    x["v"][0, 150, 0, 5] = float("nan")
    o, hT = _run(x, seq_splits=1)
    o = o.float().cpu()
    assert torch.isfinite(o[0, :128]).all()
    assert torch.isfinite(o[0, :, 0, :5]).all() and torch.isfinite(o[0, :, 0, 6:]).all()
    assert torch.isnan(o[0, 150:, 0, 5]).all()
    assert torch.isnan(hT.cpu()[0, 0, :, 5]).all()


def test_tc_caller_workspace_and_too_small():
    from chunkwise_recurrent_prefill_gb300 import GLAError, gla_fwd, workspace_size
    x = _inputs(B=1, T=1024, H=2, seed=4)
    need = workspace_size(1, 1024, 2, path="tc", seq_splits=4)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                    path="tc", seq_splits=4, workspace=ws)
    torch.cuda.synchronize()
    o_ref, h_ref = _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", "o(ws)")
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(GLAError) as e:
        gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], path="tc", seq_splits=4,
                workspace=small)
    assert e.value.status == 9


def test_tc_default_path_is_tensor_cores():
    from chunkwise_recurrent_prefill_gb300.gla import path_for
    assert path_for(1, 16384, 16) == "tc"
    assert path_for(1, 512, 2, io="f32") == "exact"


# ---------------------------------------------------------------- scalar-per-head gate

def _oracle_scalar(x):
    """The oracle takes per-key gates: a scalar gate is the same in every key dimension."""
    import oracle
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    g = x["g"].cpu()
    gk = g[..., None].expand(*g.shape, x["q"].shape[-1]).contiguous()
    return oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), gk, x["scale"], cpu(x["h0"]))


def _scalar_inputs(B, T, H, io="bf16", seed=0, with_h0=True):
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    return make_inputs(small("scalar", B=B, T=T, H=H, io=io, seed=seed, with_h0=with_h0,
                             gate="scalar"), DEV)


@pytest.mark.parametrize("T", [64, 65, 200, 1000])
@pytest.mark.parametrize("splits", [1, 3])
def test_tc_scalar_gate(T, splits):
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status
    x = _scalar_inputs(B=2, T=T, H=3, seed=T + 5 * splits)
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                    path="tc", seq_splits=splits, gate="scalar")
    torch.cuda.synchronize()
    assert last_device_status() == 0
    o_ref, h_ref = _oracle_scalar(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o(scalar, splits={splits})")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", f"hT(scalar, splits={splits})")


@pytest.mark.parametrize("kind", ["forget", "strong", "renorm"])
def test_tc_scalar_gate_extremes(kind):
    from chunkwise_recurrent_prefill_gb300 import gla_fwd
    x = _scalar_inputs(B=1, T=700, H=2, seed=9)
    g = x["g"]
    x["g"] = {"forget": torch.full_like(g, -1e4), "strong": -5.0 * torch.rand_like(g),
              "renorm": -0.5 * torch.rand_like(g)}[kind]
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                    path="tc", seq_splits=2, gate="scalar")
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    o_ref, h_ref = _oracle_scalar(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o[scalar {kind}]")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", f"hT[scalar {kind}]")


def test_exact_scalar_gate_f32():
    from chunkwise_recurrent_prefill_gb300 import gla_fwd
    x = _scalar_inputs(B=1, T=333, H=2, io="f32", seed=12)
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                    gate="scalar")
    torch.cuda.synchronize()
    o_ref, h_ref = _oracle_scalar(x)
    assert_close(o.cpu().numpy(), o_ref, "f32", "o(exact scalar)")
    assert_close(hT.cpu().numpy(), h_ref, "f32", "hT(exact scalar)")


def test_tc_scalar_gate_workload():
    """The scalar-gate bench shape (B=1, H=16, T=16384), every output, automatic split."""
    from chunkwise_recurrent_prefill_gb300 import gla_fwd
    from chunkwise_recurrent_prefill_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS["bf16_B1_H16_T16384_scalar"]
    x = make_inputs(w, DEV)
    o, _ = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                   gate="scalar")
    torch.cuda.synchronize()
    o_ref, _ = _oracle_scalar(x)
    eo = assert_close(o.float().cpu().numpy(), o_ref, "bf16", "scalar workload o")
    print(f"\nparity {w.name}: o max/mean rel {eo[0]:.3e}/{eo[1]:.3e}")


# ---------------------------------------------------------------- head dim 64

@pytest.mark.parametrize("Dk,Dv", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("gate", ["key", "scalar"])
def test_tc_head_dim_64(Dk, Dv, splits, gate):
    """Head dims of 64 on the tensor-core path (the kernels pad to 128 with zeros)."""
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status
    from chunkwise_recurrent_prefill_gb300.gla import path_for
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    assert path_for(1, 512, 2, Dk=Dk, Dv=Dv) == "tc"
    x = make_inputs(small("d64", B=2, T=700, H=3, seed=Dk + Dv + splits, with_h0=True, Dk=Dk,
                          Dv=Dv, gate=gate), DEV)
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                    path="tc", seq_splits=splits, gate=gate)
    torch.cuda.synchronize()
    assert last_device_status() == 0
    o_ref, h_ref = _oracle_scalar(x) if gate == "scalar" else _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o(D={Dk}x{Dv})")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", f"hT(D={Dk}x{Dv})")


def _d64_inputs(B, T, H, seed, with_h0=True):
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    return make_inputs(small("d64p", B=B, T=T, H=H, io="bf16", seed=seed, with_h0=with_h0, Dk=64,
                             Dv=64), DEV)


@pytest.mark.parametrize("B,T,H,splits", [(2, 700, 4, 1), (2, 700, 4, 3), (1, 1000, 2, 0),
                                          (1, 64, 2, 1), (3, 321, 6, 0), (1, 4100, 8, 0)])
def test_tc_head_pairs_d64(B, T, H, splits):
    """Head dims 64 with an even number of heads: two heads run as one of dims 128 with a
    block-diagonal state. Every element of o and hT (h0 given) against the oracle."""
    x = _d64_inputs(B, T, H, seed=B * 31 + T + H)
    o, hT = _run(x, seq_splits=splits)
    o_ref, h_ref = _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o(pairs B={B} T={T} H={H})")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", f"hT(pairs B={B} T={T} H={H})")


@pytest.mark.parametrize("kind", ["forget", "strong", "mixed", "renorm", "one_chunk_extreme",
                                  "one_head_extreme", "big_values"])
def test_tc_head_pairs_d64_extreme(kind):
    """Extreme gates on head pairs: chunks flagged extreme compute each head's P on the exact
    route from that head's own key dims; a chunk extreme in one head only flags the pair."""
    x = _d64_inputs(1, 700, 4, seed=7)
    if kind == "one_head_extreme":
        x["g"][:, 64:128, 1] = -3.0   # head 1 (second of the first pair) only
    else:
        x = _extreme(x, kind)
    o, hT = _run(x, seq_splits=2)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    o_ref, h_ref = _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o[pairs {kind}]")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", f"hT[pairs {kind}]")


def test_tc_head_pairs_d64_bench_shape():
    """The D = 64 bench shape (B=1, H=16, T=16384, h0 and hT) in its launch configuration:
    every output of every head against the C oracle."""
    from chunkwise_recurrent_prefill_gb300.workloads import WORKLOADS, make_inputs
    x = make_inputs(WORKLOADS["bf16_B1_H16_T16384_D64"], DEV)
    o, hT = _run(x)
    o_ref, h_ref = _oracle(x)
    eo = assert_close(o.float().cpu().numpy(), o_ref, "bf16", "D64 o")
    eh = assert_close(hT.cpu().numpy(), h_ref, "bf16", "D64 hT")
    print(f"\nparity D64 bench shape: o max/mean rel {eo[0]:.3e}/{eo[1]:.3e}  "
          f"hT max/mean rel {eh[0]:.3e}/{eh[1]:.3e}")
