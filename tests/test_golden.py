"""The oracle still reproduces its stored golden values (regression anchor)."""
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_reproduces_golden(oracle_lib):
    from chunkwise_recurrent_prefill_gb300.workloads import WORKLOADS, make_inputs
    with open(os.path.join(HERE, "golden", "oracle_f32_B1_H2_T512.json")) as f:
        gold = json.load(f)
    x = make_inputs(WORKLOADS[gold["workload"]])
    o, hT = oracle_lib.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"])
    for idx, val in gold["o"]:
        assert abs(o[tuple(idx)] - val) <= 1e-12 * gold["o_abs_max"], idx
    for idx, val in gold["hT"]:
        assert abs(hT[tuple(idx)] - val) <= 1e-12 * max(1.0, abs(val)), idx
    assert np.isclose(np.abs(o).max(), gold["o_abs_max"], rtol=1e-12)


def test_gdn_oracle_reproduces_golden():
    from oracle import gdn_ref
    from chunkwise_recurrent_prefill_gb300.workloads import GDN_WORKLOADS, make_gdn_inputs
    with open(os.path.join(HERE, "golden", "gdn_oracle_f32_B1_H2_T512.json")) as f:
        gold = json.load(f)
    x = make_gdn_inputs(GDN_WORKLOADS[gold["workload"]])
    o, hT = gdn_ref.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    for idx, val in gold["o"]:
        assert abs(o[tuple(idx)] - val) <= 1e-12 * gold["o_abs_max"], idx
    for idx, val in gold["hT"]:
        assert abs(hT[tuple(idx)] - val) <= 1e-12 * max(1.0, abs(val)), idx
    assert np.isclose(np.abs(o).max(), gold["o_abs_max"], rtol=1e-12)
