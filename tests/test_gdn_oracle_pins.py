"""Pins for the gated-delta-rule oracle (CPU only).

Every oracle function (the numpy token loop, the C token loop, and the fp64 chunk algebra
at several chunk sizes, ragged tails included) must pass every check in
``tests/gdn_pins.py``; copies of the token loop with a planted mistake must each fail at
least one.
"""
import numpy as np
import pytest

import gdn_pins
from pins import rel


def _impls():
    from oracle import gdn_ref
    return {
        "recurrent": gdn_ref.recurrent,
        "c_recurrent": gdn_ref.recurrent_c,
        "chunk_C1": lambda *a: gdn_ref.chunkwise(*a, C=1),
        "chunk_C4": lambda *a: gdn_ref.chunkwise(*a, C=4),
        "chunk_C5": lambda *a: gdn_ref.chunkwise(*a, C=5),
        "chunk_C64": lambda *a: gdn_ref.chunkwise(*a, C=64),
    }


@pytest.mark.parametrize("check", sorted(gdn_pins.ALL_CHECKS))
@pytest.mark.parametrize("impl", ["recurrent", "c_recurrent", "chunk_C1", "chunk_C4", "chunk_C5",
                                  "chunk_C64"])
def test_pin(impl, check):
    fn = _impls()[impl]
    rng = np.random.default_rng(4321)
    err, tol = gdn_pins.ALL_CHECKS[check](fn, rng)
    assert err <= tol, f"{impl}/{check}: err {err:.3e} > {tol:.1e}"


def _broken(kind):
    """The token loop with one planted mistake."""
    def fn(q, k, v, g, beta, scale, h0=None):
        q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
        B, T, H, Dk = q.shape
        Dv = v.shape[-1]
        S = np.zeros((B, H, Dk, Dv)) if h0 is None else np.asarray(h0, np.float64).copy()
        o = np.empty((B, T, H, Dv))
        for t in range(T):
            kt, vt = k[:, t], v[:, t]
            a = np.exp(-g[:, t] if kind == "gate_sign" else g[:, t])[..., None, None]
            bt = beta[:, t][..., None, None]
            kS = np.einsum("bhd,bhde->bhe", kt, S)
            outer = lambda x, y: x[..., :, None] * y[..., None, :]   # noqa: E731
            if kind == "read_before_write":
                o[:, t] = scale * np.einsum("bhd,bhde->bhe", q[:, t], S)
            if kind == "undecayed_error":      # error term taken from the undecayed state
                S = a * S + bt * outer(kt, vt - kS)
            elif kind == "projection_sign":
                S = a * (S + bt * outer(kt, kS)) + bt * outer(kt, vt)
            elif kind == "beta_on_value_only":
                S = a * (S - outer(kt, kS)) + bt * outer(kt, vt)
            elif kind == "no_decay_on_projection":
                S = a * S - bt * outer(kt, kS) + bt * outer(kt, vt)
            else:
                S = a * (S - bt * outer(kt, kS)) + bt * outer(kt, vt)
            if kind != "read_before_write":
                o[:, t] = scale * np.einsum("bhd,bhde->bhe", q[:, t], S)
        return o, S
    return fn


@pytest.mark.parametrize("kind", ["gate_sign", "read_before_write", "undecayed_error",
                                  "projection_sign", "beta_on_value_only",
                                  "no_decay_on_projection"])
def test_planted_mistakes_are_caught(kind):
    fn = _broken(kind)
    caught = []
    for name, check in gdn_pins.ALL_CHECKS.items():
        err, tol = check(fn, np.random.default_rng(4321))
        if not err <= tol:
            caught.append(name)
    assert caught, f"no pin catches the planted mistake {kind}"


def test_unbroken_copy_passes():
    """The planted-mistake harness itself is correct when nothing is planted."""
    fn = _broken("none")
    for name, check in gdn_pins.ALL_CHECKS.items():
        err, tol = check(fn, np.random.default_rng(4321))
        assert err <= tol, name


@pytest.mark.parametrize("C", [1, 3, 16, 64, 100])
def test_chunk_algebra_ragged(C):
    """The chunk algebra reaches the token loop at any chunk size, ragged tail included,
    at the workloads' distributions (unit-norm keys, gates logsigmoid(u)/16)."""
    from oracle import gdn_ref
    from chunkwise_recurrent_prefill_gb300.workloads import make_gdn_inputs, small
    x = make_gdn_inputs(small("t", B=2, T=100, H=2, io="f32", seed=9, with_h0=True, Dk=32, Dv=24))
    o, hT = gdn_ref.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    oc, hc = gdn_ref.chunkwise(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], C=C)
    assert rel(oc, o) < 1e-11 and rel(hc, hT) < 1e-11


def test_head_entry_matches_batch():
    from oracle import gdn_ref
    q, k, v, g, beta, h0 = gdn_pins.rand_case(np.random.default_rng(3), B=2, T=17, H=3)
    o, hT = gdn_ref.recurrent(q, k, v, g, beta, 0.4, h0)
    for b in range(2):
        for h in range(3):
            oh, hh = gdn_ref.recurrent_head(q, k, v, g, beta, 0.4, h0, b, h)
            assert np.array_equal(oh, o[b, :, h]) and np.array_equal(hh, hT[b, h])
            oh, _ = gdn_ref.recurrent_head(q, k, v, g, beta, 0.4, h0, b, h, t_end=9)
            assert np.allclose(oh, o[b, :9, h], rtol=0, atol=0)


def test_c_and_numpy_loops_agree():
    """The C token loop and the numpy one, written independently, agree to fp64 rounding on
    the workload distributions (D = 128, ragged T, h0) and on the pins' small cases."""
    from oracle import gdn_ref
    from chunkwise_recurrent_prefill_gb300.workloads import make_gdn_inputs, small
    x = make_gdn_inputs(small("t", B=2, T=77, H=3, io="bf16", seed=12, with_h0=True))
    o1, h1 = gdn_ref.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    o2, h2 = gdn_ref.recurrent_c(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    assert rel(o2, o1) < 1e-13 and rel(h2, h1) < 1e-13
    q, k, v, g, beta, _ = gdn_pins.rand_case(np.random.default_rng(8), B=1, T=30, H=2, Dk=7, Dv=5,
                                             with_h0=False)
    o1, h1 = gdn_ref.recurrent(q, k, v, g, beta, 0.9)
    o2, h2 = gdn_ref.recurrent_c(q, k, v, g, beta, 0.9)
    assert rel(o2, o1) < 1e-13 and rel(h2, h1) < 1e-13
