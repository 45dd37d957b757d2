"""Parity tolerances, one place for every test.

fp32 path: max |x - x_ref| <= 1e-5 against the fp64 oracle (O and LSE; same bound for the
gradients).

bf16-in / fp32-accumulate path, for O, dQ, dK, dV, each tensor on its own:
  * mean |x - x_ref| / rms(x_ref) <= 2e-3            (as stated for this path)
  * max  |x - x_ref| / max |x_ref| <= 2e-2            (the 2e-2 max bound, normalised by the
                                                       tensor's peak magnitude)
  * LSE: max |LSE - LSE_ref| <= 2e-2 on finite rows; -inf exactly where the oracle has -inf.
Normalising the max error by the RMS instead cannot be met by any kernel that rounds P (or dS)
to bf16 before the tensor-core product and rounds its outputs to bf16: the rounding of the
largest outputs alone exceeds 2e-2 of the RMS on causal shapes.  test_tolerance_reading.py
measures this on an emulated kernel that is exact apart from those roundings.
"""
import numpy as np

FP32_MAX_ABS = 1e-5
BF16_MEAN_OVER_RMS = 2e-3
BF16_MAX_OVER_PEAK = 2e-2
BF16_LSE_MAX_ABS = 2e-2


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    e = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    peak = float(np.max(np.abs(ref))) if ref.size else 0.0
    return dict(max_abs=float(e.max()) if e.size else 0.0,
                mean_over_rms=float(e.mean() / rms) if rms > 0 else float(e.mean()),
                max_over_peak=float(e.max() / peak) if peak > 0 else float(e.max() if e.size else 0.0),
                max_over_rms=float(e.max() / rms) if rms > 0 else float(e.max() if e.size else 0.0))


def assert_bf16_close(name, got, ref):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    r = errors(got, ref)
    assert r["mean_over_rms"] <= BF16_MEAN_OVER_RMS, (name, r)
    assert r["max_over_peak"] <= BF16_MAX_OVER_PEAK, (name, r)
    return r


def assert_lse_close(got, ref, tol):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    neg = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), neg), "LSE: -inf rows differ"
    if (~neg).any():
        err = float(np.max(np.abs(got[~neg] - ref[~neg])))
        assert err <= tol, ("LSE", err)
        return err
    return 0.0


def assert_fp32_close(name, got, ref, tol=FP32_MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= tol, (name, err)
    return err
