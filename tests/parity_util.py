"""Shared tolerances and comparison helpers for the GPU parity tests.

Tolerances (fixed by the target statement of the path): f16 K/V outputs must
match the fp64 oracle to max-abs <= 2e-3 and relative L2 <= 1e-3; int8 K/V
outputs to 5e-3 against the oracle run on the dequantised values (the oracle
dequantises from the same codes and scales).  The int8 figure stands in the
target beside both the max-abs and the relative-L2 bound, so both are applied:
max-abs <= 5e-3 and relative L2 <= 5e-3.
"""
import numpy as np

F16_MAX_ABS = 2e-3
F16_REL_L2 = 1e-3
INT8_MAX_ABS = 5e-3
INT8_REL_L2 = 5e-3
LSE_MAX_ABS = 2e-3


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff)) / denom if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(got, ref, int8=False, what=""):
    max_abs, rel = errors(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), "%s: non-finite output" % what
    tol_abs, tol_rel = (INT8_MAX_ABS, INT8_REL_L2) if int8 else (F16_MAX_ABS, F16_REL_L2)
    assert max_abs <= tol_abs and rel <= tol_rel, \
        "%s: max-abs %.3g (<= %.3g), rel-L2 %.3g (<= %.3g)" % (what, max_abs, tol_abs, rel, tol_rel)


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "%s: lse finiteness differs" % what
    if fin.any():
        err = float(np.abs(got[fin] - ref[fin]).max())
        assert err <= LSE_MAX_ABS, "%s: lse max-abs %.3g" % (what, err)
