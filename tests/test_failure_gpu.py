"""Failure detection without a GPU fault: a bounded pipeline wait that runs out.

With GLA_TEST_STALL_ONE_LOAD set, the output kernel's TMA producer never issues the q/k/v
load of one chunk. Every wait that depends on it gives up after its bounded limit, the
kernel raises the library's device error word, drains what it issued, frees its TMEM and
returns. The host then reads GLA_ERR_DEVICE_TIMEOUT, and the next call on the same context
is correct.
"""
import time

import pytest
import torch

from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_bounded_wait_times_out_and_context_survives(monkeypatch):
    import oracle
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    x = make_inputs(small("stall", B=1, T=512, H=2, io="bf16", seed=6, with_h0=True),
                    torch.device("cuda:0"))
    assert last_device_status() == 0
    monkeypatch.setenv("GLA_TEST_STALL_ONE_LOAD", "1")
    t0 = time.time()
    gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True, path="tc",
            seq_splits=1)
    status = last_device_status()
    waited = time.time() - t0
    monkeypatch.delenv("GLA_TEST_STALL_ONE_LOAD")
    assert status == 7, status                      # GLA_ERR_DEVICE_TIMEOUT
    assert 1.0 < waited < 30.0, waited              # the waits are bounded (~2 s each)
    assert last_device_status() == 0                # reading the status cleared it
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                    path="tc", seq_splits=1)
    torch.cuda.synchronize()
    assert last_device_status() == 0
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    o_ref, h_ref = oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]),
                                    x["scale"], cpu(x["h0"]))
    assert_close(o.float().cpu().numpy(), o_ref, "bf16", "o after timeout")
    assert_close(hT.cpu().numpy(), h_ref, "bf16", "hT after timeout")
