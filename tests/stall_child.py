"""Child process of test_failure_gpu.py (run as a script, never collected by pytest).

It starts with GLA_TEST_STALL_ONE_LOAD set, so the library's first tensor-core launch of
this process skips one chunk's load: that call must report GLA_ERR_DEVICE_TIMEOUT after its
bounded waits run out, and the next call on the same context must match the oracle.
Prints one JSON line with what it saw.
"""
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))


def main():
    import torch
    import oracle
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, last_device_status
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    from parity import errors
    assert os.environ.get("GLA_TEST_STALL_ONE_LOAD")
    x = make_inputs(small("stall", B=1, T=512, H=2, io="bf16", seed=6, with_h0=True),
                    torch.device("cuda:0"))
    out = {"status_before": last_device_status()}
    t0 = time.time()
    gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True, path="tc",
            seq_splits=1)
    out["status_stalled"] = last_device_status()
    out["waited_s"] = time.time() - t0
    out["status_cleared"] = last_device_status()
    o, hT = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                    path="tc", seq_splits=1)
    torch.cuda.synchronize()
    out["status_after"] = last_device_status()
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    o_ref, h_ref = oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]),
                                    x["scale"], cpu(x["h0"]))
    out["o_err"] = errors(o.float().cpu().numpy(), o_ref)
    out["hT_err"] = errors(hT.cpu().numpy(), h_ref)
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
