"""Numerical error against sequence length on the tensor-core path.

"面向长序列大模型的线性注意力算子性能评测方法与优化实践", section 七 (5.), warns that the
error of a recurrent operator can grow faster as sequences get longer. This runs the bench's
input recipe (bf16 q/k/v ~ N(0,1), fp32 log-gates logsigmoid(N(0,1))/16, h0 = 0.02 N(0,1),
B = 1, H = 16, D = 128) at T = 512 ... 131072 in the launch configuration gla_fwd picks, and
compares o and hT with the fp64 oracle: every length within the bf16 bounds, and the error
growing no faster than linearly in T (each step's error ratio at most twice the length ratio).
The measured table is printed (run with -s to see it).
"""
import pytest
import torch

from parity import TOL, errors

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
LENGTHS = [512, 4096, 16384, 65536, 131072]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_error_against_length():
    import oracle
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    rows = []
    for T in LENGTHS:
        x = make_inputs(small("growth", B=1, T=T, H=16, io="bf16", seed=100 + T % 97,
                              with_h0=True), DEV)
        o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True)
        torch.cuda.synchronize()
        assert last_device_status() == 0
        cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
        o_ref, h_ref = oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]),
                                        x["scale"], cpu(x["h0"]))
        eo = errors(o.float().cpu().numpy(), o_ref)
        eh = errors(hT.cpu().numpy(), h_ref)
        rows.append((T, eo, eh))
        del x, o, hT, o_ref, h_ref
    print("\n   T      o max     o mean    hT max    hT mean")
    for T, eo, eh in rows:
        print(f"{T:7d}  {eo[0]:.3e}  {eo[1]:.3e}  {eh[0]:.3e}  {eh[1]:.3e}")
    tol = TOL["bf16"]
    for T, eo, eh in rows:
        for e in (eo, eh):
            assert e[0] <= tol["max"] and e[1] <= tol["mean"], (T, e)
    for (T1, eo1, eh1), (T2, eo2, eh2) in zip(rows[:-1], rows[1:]):
        for a, b in ((eo1, eo2), (eh1, eh2)):
            for i in (0, 1):
                assert b[i] <= 2.0 * (T2 / T1) * max(a[i], 1e-7), (T1, T2, a, b)
