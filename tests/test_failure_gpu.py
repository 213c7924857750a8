"""Failure detection without a GPU fault: a bounded pipeline wait that runs out.

With GLA_TEST_STALL_ONE_LOAD set when a process starts, the library's first tensor-core
launch in that process has its TMA producer skip the q/k/v load of one chunk. Every wait that
depends on it gives up after its bounded limit, the kernel raises the library's device error
word, drains what it issued, frees its TMEM and returns. The host then reads
GLA_ERR_DEVICE_TIMEOUT, and the next call on the same context is correct. The library reads
the variable once per process, so the scenario runs in a child process (tests/stall_child.py).
"""
import json
import os
import subprocess
import sys

import pytest

from parity import TOL

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_bounded_wait_times_out_and_context_survives():
    env = dict(os.environ, GLA_TEST_STALL_ONE_LOAD="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "stall_child.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["status_before"] == 0
    assert out["status_stalled"] == 7, out            # GLA_ERR_DEVICE_TIMEOUT
    assert 1.0 < out["waited_s"] < 30.0, out          # the waits are bounded (~2 s each)
    assert out["status_cleared"] == 0                 # reading the status cleared it
    assert out["status_after"] == 0
    for name in ("o_err", "hT_err"):
        mx, mean = out[name]
        assert mx <= TOL["bf16"]["max"] and mean <= TOL["bf16"]["mean"], (name, mx, mean)
