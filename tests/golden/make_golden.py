"""Write the oracle's golden regression values (calls only ``oracle/`` and the seeded
input generator). Run from the repo root:  python tests/golden/make_golden.py

The pages print no worked numeric example of GLA or of the gated delta rule, so these
values are not the pages': they are the pinned oracles' outputs on the fp32 parity
workloads (B=1, H=2, T=512, D=128; seed 0 for GLA, seed 10 for the gated delta rule) at
fixed sampled positions, stored so that a later change to an oracle's arithmetic shows up
as a diff here.
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import gdn_ref  # noqa: E402
from chunkwise_recurrent_prefill_gb300.workloads import (  # noqa: E402
    GDN_WORKLOADS, WORKLOADS, make_gdn_inputs, make_inputs)


def sampled(w, o, hT, name, seed):
    rng = np.random.default_rng(seed)
    idx_o = [(0, int(t), int(h), int(e)) for t, h, e in
             zip(rng.integers(0, w.T, 48), rng.integers(0, w.H, 48), rng.integers(0, w.Dv, 48))]
    idx_o += [(0, w.T - 1, 1, 0), (0, 0, 0, 0), (0, 63, 0, 5), (0, 64, 1, 127)]
    idx_h = [(0, int(h), int(d), int(e)) for h, d, e in
             zip(rng.integers(0, w.H, 16), rng.integers(0, w.Dk, 16), rng.integers(0, w.Dv, 16))]
    out = {
        "about": "oracle outputs (fp64) at sampled positions; written by make_golden.py",
        "workload": w.name,
        "o": [[list(i), float(o[i])] for i in idx_o],
        "hT": [[list(i), float(hT[i])] for i in idx_h],
        "o_abs_max": float(np.abs(o).max()),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), name)
    with open(path, "w") as f:
        json.dump(out, f)
        f.write("\n")
    print("wrote", path)


def main():
    w = WORKLOADS["f32_B1_H2_T512"]
    x = make_inputs(w)
    o, hT = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"])
    sampled(w, o, hT, "oracle_f32_B1_H2_T512.json", 2024)
    w = GDN_WORKLOADS["gdn_f32_B1_H2_T512"]
    x = make_gdn_inputs(w)
    o, hT = gdn_ref.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    sampled(w, o, hT, "gdn_oracle_f32_B1_H2_T512.json", 2025)


if __name__ == "__main__":
    main()
