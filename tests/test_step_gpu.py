"""GPU parity of the decode step (gla_step) against the fp64 oracle.

One step is the oracle's recurrence over a single token starting from the state S. A
prefill followed by decode steps must match the oracle run over all the tokens at once.
"""
import pytest
import torch

from parity import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _oracle_step(x):
    import oracle
    c = lambda t: t.cpu()[:, None]  # noqa: E731  one token: [B, 1, H, D]
    o, hT = oracle.recurrent(c(x["q"]), c(x["k"]), c(x["v"]), c(x["g"]), x["scale"],
                             x["S"].cpu())
    return o[:, 0], hT


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("B,H,D", [(2, 3, 128), (4, 16, 128), (1, 2, 64), (3, 1, 96)])
def test_step_matches_oracle(io, B, H, D):
    from chunkwise_recurrent_prefill_gb300 import gla_step, last_device_status
    from chunkwise_recurrent_prefill_gb300.workloads import make_step_inputs
    x = make_step_inputs(B, H, D, io, seed=B * 100 + H + D, device=DEV)
    o_ref, s_ref = _oracle_step(x)
    S = x["S"].clone()
    o = gla_step(x["q"], x["k"], x["v"], x["g"], x["scale"], S)
    torch.cuda.synchronize()
    assert last_device_status() == 0
    # the state is fp32 arithmetic on exactly representable inputs: fp32 class either way
    assert_close(S.cpu().numpy(), s_ref, "f32", f"S[{io}]")
    assert_close(o.float().cpu().numpy(), o_ref, io, f"o[{io}]")


def test_prefill_then_decode_matches_oracle():
    """hT of a tensor-core prefill, then eight decode steps, against the oracle over all
    the tokens (bf16 tolerance: the prefill's state is bf16-operand class)."""
    import oracle
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, gla_step
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    T, K = 1000, 8
    x = make_inputs(small("dec", B=2, T=T + K, H=4, io="bf16", seed=77, with_h0=True), DEV)
    pre = {n: x[n][:, :T].contiguous() for n in ("q", "k", "v", "g")}
    _, S = gla_fwd(pre["q"], pre["k"], pre["v"], pre["g"], x["scale"], x["h0"],
                   return_state=True)
    outs = []
    for t in range(T, T + K):
        outs.append(gla_step(x["q"][:, t].contiguous(), x["k"][:, t].contiguous(),
                             x["v"][:, t].contiguous(), x["g"][:, t].contiguous(), x["scale"],
                             S))
    torch.cuda.synchronize()
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    o_ref, h_ref = oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]),
                                    x["scale"], cpu(x["h0"]))
    o_dec = torch.stack(outs, dim=1).float().cpu().numpy()
    assert_close(o_dec, o_ref[:, T:], "bf16", "decoded o")
    assert_close(S.cpu().numpy(), h_ref, "bf16", "state after decode")


def test_step_empty_batch_and_zero_gate():
    """B = 0 launches nothing; g = -inf-like forgetting leaves exactly k^T v."""
    from chunkwise_recurrent_prefill_gb300 import gla_step
    from chunkwise_recurrent_prefill_gb300.workloads import make_step_inputs
    e = make_step_inputs(0, 2, 128, "f32", device=DEV)
    gla_step(e["q"], e["k"], e["v"], e["g"], e["scale"], e["S"])
    x = make_step_inputs(1, 2, 128, "f32", seed=3, device=DEV)
    x["g"] = torch.full_like(x["g"], -1e4)
    S = x["S"].clone()
    gla_step(x["q"], x["k"], x["v"], x["g"], x["scale"], S)
    torch.cuda.synchronize()
    kv = x["k"][..., :, None] * x["v"][..., None, :]
    assert torch.equal(S, kv)
