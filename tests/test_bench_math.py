"""The bench's workload arithmetic (CPU only): the algorithmic bytes and flops its roofline
fractions divide by, the derived fp32 peak, and the committed traffic lookup."""
import json
import os

import bench


def test_gla_algorithmic_bytes_and_flops():
    from chunkwise_recurrent_prefill_gb300.workloads import WORKLOADS
    w = WORKLOADS["bf16_B1_H16_T16384"]
    # q, k, v, o in bf16 (4 x 128 x 2 B) + g in fp32 (128 x 4 B) = 1536 B per token and head
    assert bench.algorithmic_bytes(w) == 16384 * 16 * 1536 == 402_653_184
    # 4 Dk Dv + (C + 1)(Dk + Dv) = 82,176 flops per token and head at C = 64
    assert bench.algorithmic_flops(w) == 16384 * 16 * 82_176
    # a scalar gate is 4 B per token and head; h0 and hT add 64 KiB per (b, h) each
    ws = WORKLOADS["bf16_B1_H16_T16384_scalar"]
    assert bench.algorithmic_bytes(ws) == 16384 * 16 * (1024 + 4)
    wh = WORKLOADS["bf16_B1_H16_T131072_h0"]
    assert bench.algorithmic_bytes(wh) == 131072 * 16 * 1536 + 2 * 16 * 128 * 128 * 4


def test_gdn_flops_and_peak():
    # 2 C Dk + C (Dk + Dv) + 6 Dk Dv + C Dv at C = 64, Dk = Dv = 128
    assert bench.gdn_flops_per_token_head(128, 128) == 16384 + 16384 + 98304 + 8192 == 139_264
    peak, src = bench.fp32_alu_peak_tflops(None)
    assert abs(peak - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9 and "2070 MHz" in src
    assert abs(bench.fp32_alu_peak_tflops(1000.0)[0] - 152 * 128 * 2 * 1e9 / 1e12) < 1e-9
    # the tensor-core path's tf32 peak: the measured bf16 peak x the nominal dense ratio
    assert abs(bench.TF32_PER_BF16 - 1.1 / 2.25) < 1e-12


def test_weak_scaling_value():
    # every rank processed `steps` of its own workload; the slowest rank's time counts
    assert bench.weak_scaling_value(16384, 10, 4, 2.0) == 4 * 16384 * 10 / 2.0


def test_committed_traffic_is_keyed_by_source():
    path = os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")
    with open(path) as f:
        entries = json.load(f)
    for e in entries:
        got = bench.committed_traffic(e["kernel_kind"], e["workload"])
        # the entry applies exactly when the kernel source still has the recorded hash
        if bench.source_sha(e["kernel_kind"]) == e["source_sha256"]:
            assert got == e["dram_bytes_per_launch"]
        else:
            assert got is None
    assert bench.committed_traffic("tc", "no_such_workload") is None
