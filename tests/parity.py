"""Error metrics and tolerances for GPU-vs-oracle parity.

Tolerances (fixed for this method's workloads):
* fp32 I/O:  max|out - ref| <= 1e-4 * max|ref|
* bf16 I/O:  max|out - ref| <= 1.5e-2 * max|ref|  and  sum|out - ref| / sum|ref| <= 5e-3
Both apply to o and, separately, to the returned state hT.
The "mean relative error" is the L1 ratio sum|d| / sum|ref|; an elementwise mean of
|d| / |ref| is undefined near zero outputs.
"""
import numpy as np

TOL = {"f32": dict(max=1e-4, mean=1e-4), "bf16": dict(max=1.5e-2, mean=5e-3)}


def errors(out, ref):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(out - ref)
    mx = float(d.max() / max(np.abs(ref).max(), 1e-300)) if d.size else 0.0
    mean = float(d.sum() / max(np.abs(ref).sum(), 1e-300)) if d.size else 0.0
    return mx, mean


def assert_close(out, ref, io, what=""):
    out = np.asarray(out, np.float64)
    assert not np.isnan(out).any() or np.isnan(ref).any(), f"{what}: NaN in output"
    mx, mean = errors(out, ref)
    tol = TOL[io]
    assert mx <= tol["max"] and mean <= tol["mean"], \
        f"{what}: max rel {mx:.3e} (tol {tol['max']:.1e}), mean rel {mean:.3e} (tol {tol['mean']:.1e})"
    return mx, mean
