"""CUDA graph capture of the forward calls.

A call is a short chain of kernel launches on one stream (the tensor-core GLA forward: state
pass, segment scan and output kernel, chained with programmatic dependent launch; the gated
delta rule: prep, and its scan in one or three launches). Captured into a graph, the chain
replays with whatever the captured input buffers hold at replay time. Each capture passes a
caller workspace, so nothing is allocated while the stream is capturing.
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


def _copy_into(dst: dict, src: dict):
    for k_, v_ in src.items():
        if isinstance(v_, torch.Tensor):
            dst[k_].copy_(v_)


@pytest.mark.parametrize("T,H,D", [(4096, 4, 128), (2048, 4, 64)])
def test_gla_graph_replay(T, H, D):
    """The GLA forward captured once (sequence split on: 4 heads of T tokens, or 2 head pairs
    at head dims 64) and replayed on two fresh inputs: each replay equals an eager call on the
    same inputs, bit for bit, and the oracle within the bf16 bounds."""
    import oracle
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status, workspace_size
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    mk = lambda seed: make_inputs(small("graph", B=1, T=T, H=H, io="bf16", seed=seed,  # noqa: E731
                                        with_h0=True, Dk=D, Dv=D), DEV)
    x = mk(61)
    need = workspace_size(1, T, H, Dk=D, Dv=D)
    assert need > 0                                      # the split is on
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    o = torch.empty((1, T, H, D), dtype=torch.bfloat16, device=DEV)
    hT = torch.empty((1, H, D, D), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up on the capture stream (per-device setup)
        gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], o=o, hT=hT, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], o=o, hT=hT, workspace=ws)
    for seed in (62, 63):
        y = mk(seed)
        _copy_into(x, y)
        o.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert last_device_status() == 0
        oe, he = gla_fwd(y["q"], y["k"], y["v"], y["g"], y["scale"], y["h0"], return_state=True,
                         workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o, oe) and torch.equal(hT, he)
        cpu = lambda t: t.cpu()  # noqa: E731
        o_ref, h_ref = oracle.recurrent(cpu(y["q"]), cpu(y["k"]), cpu(y["v"]), cpu(y["g"]),
                                        y["scale"], cpu(y["h0"]))
        assert_close(o.float().cpu().numpy(), o_ref, "bf16", f"o(graph, seed {seed})")
        assert_close(hT.cpu().numpy(), h_ref, "bf16", f"hT(graph, seed {seed})")


def test_gdn_graph_replay():
    """The gated delta rule forward captured once with its split scan on (2 heads of 2048
    tokens: prep and three scan launches) and replayed on a fresh input: bit for bit the eager
    result, and the oracle within the bf16 bounds."""
    from oracle import gdn_ref
    from chunkwise_recurrent_prefill_gb300 import gdn_fwd, gdn_workspace_size, last_device_status
    from chunkwise_recurrent_prefill_gb300.workloads import make_gdn_inputs, small
    mk = lambda seed: make_gdn_inputs(small("gdn_graph", B=1, T=2048, H=2, io="bf16",  # noqa: E731
                                            seed=seed, with_h0=True), DEV)
    x = mk(71)
    ws = torch.empty(gdn_workspace_size(1, 2048, 2, 128, 128), dtype=torch.uint8, device=DEV)
    o = torch.empty((1, 2048, 2, 128), dtype=torch.bfloat16, device=DEV)
    hT = torch.empty((1, 2, 128, 128), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], o=o, hT=hT,
                workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], o=o, hT=hT,
                workspace=ws)
    y = mk(72)
    _copy_into(x, y)
    g.replay()
    torch.cuda.synchronize()
    assert last_device_status() == 0
    oe, he = gdn_fwd(y["q"], y["k"], y["v"], y["g"], y["beta"], y["scale"], y["h0"],
                     return_state=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o, oe) and torch.equal(hT, he)
    cpu = lambda t: t.cpu()  # noqa: E731
    o_ref, h_ref = gdn_ref.recurrent(cpu(y["q"]), cpu(y["k"]), cpu(y["v"]), cpu(y["g"]),
                                     cpu(y["beta"]), y["scale"], cpu(y["h0"]))
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", "gdn o(graph)")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", "gdn hT(graph)")
