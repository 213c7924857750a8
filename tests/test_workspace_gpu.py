"""The library's own scratch (the sequence split's segment states) is kept per stream.

Two calls of different shapes issued back to back on two streams, with no ordering between
them, must each match the fp64 oracle (they would race if they shared one buffer), and
repeating a call of the same shape on the same stream must allocate nothing.
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


def _inputs(B, T, H, seed):
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    return make_inputs(small("ws", B=B, T=T, H=H, io="bf16", seed=seed, with_h0=True), DEV)


def _oracle(x):
    import oracle
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    return oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]), x["scale"],
                            cpu(x["h0"]))


def test_two_streams_concurrently():
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status
    from chunkwise_recurrent_prefill_gb300.gla import workspace_size
    xa, xb = _inputs(1, 4096, 4, seed=71), _inputs(2, 3000, 3, seed=72)
    assert workspace_size(1, 4096, 4) > 0 and workspace_size(2, 3000, 3) > 0
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):   # several rounds, each pair issued without any ordering between them
        with torch.cuda.stream(sa):
            oa = gla_fwd(xa["q"], xa["k"], xa["v"], xa["g"], xa["scale"], xa["h0"],
                         return_state=True, stream=sa)
        with torch.cuda.stream(sb):
            ob = gla_fwd(xb["q"], xb["k"], xb["v"], xb["g"], xb["scale"], xb["h0"],
                         return_state=True, stream=sb)
        outs.append((oa, ob))
    torch.cuda.synchronize()
    assert last_device_status() == 0
    ra, rb = _oracle(xa), _oracle(xb)
    for oa, ob in outs:
        for (o, h), (o_ref, h_ref), name in ((oa, ra, "a"), (ob, rb, "b")):
            assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o {name}")
            assert_close(h.cpu().numpy(), h_ref, "bf16", f"hT {name}")


def test_repeated_calls_allocate_nothing():
    from chunkwise_recurrent_prefill_gb300 import gla_fwd
    from chunkwise_recurrent_prefill_gb300.gla import workspace_allocations, workspace_size
    x = _inputs(1, 8192, 8, seed=73)
    assert workspace_size(1, 8192, 8) > 0
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], stream=s)
        n0 = workspace_allocations()
        for _ in range(5):
            gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], stream=s)
        # a smaller problem on the same stream fits the buffer it already has
        y = _inputs(1, 2048, 4, seed=74)
        gla_fwd(y["q"], y["k"], y["v"], y["g"], y["scale"], y["h0"], stream=s)
    torch.cuda.synchronize()
    assert workspace_allocations() == n0
