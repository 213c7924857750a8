"""GPU parity: the CUDA paths through the C ABI against the fp64 oracle on the same
seeded inputs (element by element), plus edge cases and status codes."""
import numpy as np
import pytest
import torch

from parity import assert_close, errors

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(x, path="auto", seq_splits=0, want_state=True):
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"],
                    return_state=want_state, path=path, seq_splits=seq_splits)
    torch.cuda.synchronize()
    assert last_device_status() == 0
    return o, hT


def _oracle(x):
    import oracle
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    return oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]), x["scale"],
                            cpu(x["h0"]))


def _check(x, io, path="auto", seq_splits=0):
    o, hT = _run(x, path, seq_splits)
    o_ref, h_ref = _oracle(x)
    r1 = assert_close(o.float().cpu().numpy(), o_ref, io, f"o[{path}]")
    r2 = assert_close(hT.cpu().numpy(), h_ref, io, f"hT[{path}]")
    return r1, r2


def _inputs(name, B, T, H, io="bf16", seed=0, with_h0=True, Dk=128, Dv=128):
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    return make_inputs(small(name, B=B, T=T, H=H, io=io, seed=seed, with_h0=with_h0, Dk=Dk,
                             Dv=Dv), DEV)


# ---------------- exact fp32 CUDA-core path ----------------

def test_exact_f32_workload():
    """fp32 I/O parity workload (B=1, H=2, T=512, D=128, seed 0) on every output."""
    from chunkwise_recurrent_prefill_gb300.workloads import WORKLOADS, make_inputs
    x = make_inputs(WORKLOADS["f32_B1_H2_T512"], DEV)
    _check(x, "f32", path="exact")


@pytest.mark.parametrize("T", [0, 1, 3, 63, 64, 65, 127, 200])
def test_exact_f32_ragged(T):
    _check(_inputs("r", B=2, T=T, H=3, io="f32", seed=T), "f32", path="exact")


@pytest.mark.parametrize("dims", [(64, 64), (64, 128), (128, 64)])
def test_exact_head_dims(dims):
    _check(_inputs("d", B=1, T=150, H=2, io="f32", seed=9, Dk=dims[0], Dv=dims[1]), "f32",
           path="exact")


def test_exact_bf16_io():
    _check(_inputs("b", B=2, T=300, H=2, io="bf16", seed=4), "bf16", path="exact")


def _extreme(x, kind):
    g = x["g"]
    if kind == "forget":         # exp(g) underflows to 0: each token sees only itself
        x["g"] = torch.full_like(g, -1e4)
    elif kind == "no_decay":     # g = 0: plain causal linear attention
        x["g"] = torch.zeros_like(g)
    elif kind == "tiny":
        x["g"] = -1e-8 * torch.ones_like(g)
    elif kind == "strong":       # |g| ~ 5 per token: in-chunk cumulative gates reach ~-300
        x["g"] = -5.0 * torch.rand_like(g)
    elif kind == "mixed":        # a few columns and tokens forget completely, rest mild
        x["g"] = torch.where(torch.rand_like(g) < 0.02, torch.full_like(g, -200.0), g)
    elif kind == "big_values":
        for key in ("q", "k", "v"):
            x[key] = (x[key].float() * 30).to(x[key].dtype)
    return x


@pytest.mark.parametrize("kind", ["forget", "no_decay", "tiny", "strong", "mixed", "big_values"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_exact_extreme_gates(kind, io):
    x = _extreme(_inputs("e", B=1, T=160, H=2, io=io, seed=3), kind)
    o, hT = _run(x, path="exact")
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    o_ref, h_ref = _oracle(x)
    assert_close(o.float().cpu().numpy(), o_ref, io, f"o[{kind}]")
    assert_close(hT.cpu().numpy(), h_ref, io, f"hT[{kind}]")


def test_exact_nan_propagates():
    x = _inputs("n", B=1, T=100, H=1, io="f32", seed=1, with_h0=False)
    x["v"][0, 70, 0, 5] = float("nan")
    o, hT = _run(x, path="exact")
    o = o.cpu()
    assert torch.isfinite(o[0, :70]).all()
    assert torch.isnan(o[0, 70:, 0, 5]).all()
    assert torch.isnan(hT.cpu()[0, 0, :, 5]).all()


def test_empty_batch_is_noop():
    from chunkwise_recurrent_prefill_gb300 import gla_fwd
    x = _inputs("z", B=0, T=64, H=2, io="bf16")
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], 1.0, None, return_state=True)
    torch.cuda.synchronize()
    assert o.shape == (0, 64, 2, 128) and hT.shape == (0, 2, 128, 128)


def test_status_codes_on_device():
    from chunkwise_recurrent_prefill_gb300 import GLAError, gla_fwd
    x = _inputs("s", B=1, T=64, H=1, io="bf16", with_h0=False)
    buf = torch.empty(64 * 128 + 8, dtype=torch.bfloat16, device=DEV)
    mis = buf[1:1 + 64 * 128].view(1, 64, 1, 128)            # 2-byte offset
    with pytest.raises(GLAError) as e:
        gla_fwd(mis, x["k"], x["v"], x["g"], 1.0)
    assert e.value.status == 4
    with pytest.raises(GLAError) as e:                     # o aliases q
        gla_fwd(x["q"], x["k"], x["v"], x["g"], 1.0, o=x["q"])
    assert e.value.status == 5
