"""Shared helpers of the GPU parity tests (no method arithmetic here)."""
import numpy as np

TOL_F32 = 1e-4   # max|err| / RMS(ref), fp32 path
TOL_BF16 = 2e-2  # max|err| / RMS(ref), bf16 path


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    err = np.max(np.abs(got - ref))
    rms = np.sqrt(np.mean(ref * ref))
    if rms == 0.0:
        return err / 1e-6 * 1e-6 if err > 1e-6 else 0.0
    return err / rms


def assert_close(got, ref, tol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    err = np.max(np.abs(got - ref)) if ref.size else 0.0
    if rms == 0.0:
        assert err <= 1e-6, f"{what}: max|err| {err:.3e} with zero reference"
    else:
        assert err / rms <= tol, f"{what}: max|err|/RMS = {err / rms:.3e} > {tol:.1e} (max|err| {err:.3e}, RMS {rms:.3e})"
    return err / rms if rms else err


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
