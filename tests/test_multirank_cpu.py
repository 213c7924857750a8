"""Multi-rank host logic of bench.py on CPU (gloo, world_size 2): every rank runs its own
copy of the workload (weak scaling, no data-path collective); the job time is the max over
ranks and the job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        m = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        v = bench.weak_scaling_value(16384, 10, world, m)
        dist.barrier()
        out[rank] = (m, v)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    world, port = 2, _free_port()
    times = [1.25, 2.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        m, v = res[r]
        assert m == pytest.approx(2.5)
        assert v == pytest.approx(2 * 16384 * 10 / 2.5)


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, None, None) == 3.0
    assert bench.weak_scaling_value(100, 5, 1, 2.0) == pytest.approx(250.0)


def test_reference_arm_nonzero_rank_does_no_work(capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from chunkwise_recurrent_prefill_gb300.workloads import WORKLOADS

    class A:
        steps, warmup = 1, 0
    bench.run_reference(A, WORKLOADS["bf16_B1_H16_T16384"], rank=1, world=2)
    assert capsys.readouterr().out == ""
