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


BF16_U = 2.0 ** -8   # unit roundoff of bf16 (half an ulp, relative)


def bf16_excess(got, ref):
    """max_i max(|got_i - ref_i| - u|ref_i|, 0) / RMS(ref): the error beyond one
    rounding of the exact value to bf16."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0, 0.0
    err = np.abs(got - ref)
    rms = np.sqrt(np.mean(ref * ref))
    exc = np.maximum(err - BF16_U * np.abs(ref), 0.0).max()
    if rms == 0.0:
        return exc, err.max()
    return exc / rms, err.max() / rms


def assert_close_bf16(got, ref, tol=TOL_BF16, what=""):
    """bf16-path bound: max|err|/RMS(ref) <= tol for the part of the error that
    exceeds one rounding of the exact value to bf16 (u = 2^-8 relative).  A bf16
    result stored exactly rounded already carries |err| up to u|ref|, which for
    tensors with max|ref|/RMS(ref) > tol/u = 5 alone would exceed tol."""
    got = np.asarray(got, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    exc, lit = bf16_excess(got, ref)
    rms = float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2))) if np.size(ref) else 0.0
    if rms == 0.0:
        assert exc <= 1e-6, f"{what}: max|err| {exc:.3e} with zero reference"
    else:
        assert exc <= tol, f"{what}: error beyond bf16 rounding {exc:.3e}/RMS > {tol:.1e} (plain max|err|/RMS {lit:.3e})"
    return exc, lit
