"""Acceptance test for FP32 products against the FP64 oracle (test helper).

An FP32 result C of C = A.B is accepted when, elementwise,
    |C - C_ref| <= 4 * K * 2**-24 * (|A|.|B|)_ij
and the relative Frobenius error ||C - C_ref||_F / ||C_ref||_F <= 1e-5.
The elementwise bound is the standard a-priori bound for a K-term FP32 dot
product in any summation order (gamma_K ~ K * 2**-24), with a factor 4 of
margin; the Frobenius limit is the stated FP32 tolerance.  NaN positions
must agree exactly.  For K == 0 the bound is 0: the result must be exactly 0.
"""
import numpy as np

FROB_LIMIT = 1e-5


def bound(S_ref: np.ndarray, K: int) -> np.ndarray:
    return 4.0 * K * 2.0 ** -24 * S_ref


def check(C, C_ref, S_ref, K, frob_limit=FROB_LIMIT):
    """Return (ok, report) for an FP32 result against the oracle."""
    C = np.asarray(C, dtype=np.float64)
    C_ref = np.asarray(C_ref, dtype=np.float64)
    nan_c, nan_r = np.isnan(C), np.isnan(C_ref)
    if not np.array_equal(nan_c, nan_r):
        return False, {"reason": "NaN positions differ",
                       "nan_result": int(nan_c.sum()), "nan_ref": int(nan_r.sum())}
    ok_mask = ~nan_r
    err = np.abs(C - C_ref)[ok_mask]
    lim = bound(np.asarray(S_ref, dtype=np.float64), K)[ok_mask]
    elem_ok = bool(np.all(err <= lim))
    worst = float(np.max(err / np.where(lim > 0, lim, 1.0))) if err.size else 0.0
    if np.any((lim == 0) & (err > 0)):
        worst = float("inf")
    ref = C_ref[ok_mask]
    den = float(np.sqrt(np.sum(ref * ref)))
    num = float(np.sqrt(np.sum(err * err)))
    frob = num / den if den > 0 else (0.0 if num == 0 else float("inf"))
    ok = elem_ok and frob <= frob_limit
    return ok, {"max_err_over_bound": worst, "frob_rel": frob, "n": int(err.size)}


def assert_close(C, C_ref, S_ref, K, what=""):
    ok, rep = check(C, C_ref, S_ref, K)
    assert ok, f"{what}: {rep}"
    return rep
