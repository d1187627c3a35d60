"""Shared helpers of the GPU parity tests (no method arithmetic here).

The bound is max|err|/RMS(ref) <= 1e-4 (fp32 path) and <= 2e-2 (bf16 path) on
every output and gradient.  How a result is stored decides what it is held to:

* fp32-stored results (weight gradients, dγ/dβ, statistics) and every result
  of the fp32 path: the plain ratio;
* results stored in a 16-bit type (bf16 activations and gradients, the f16
  attention output O): the part of the error beyond one rounding of the exact
  value to that type, max_i max(|got_i - ref_i| - u|ref_i|, 0) / RMS(ref), with
  u = 2^-8 (bf16) or 2^-11 (f16).  An exactly rounded bf16 tensor whose
  max|ref|/RMS(ref) exceeds tol/u = 5 would fail the plain ratio by itself.

Every check records the plain ratio and the allowance figure; with
MTGR_PARITY_LOG set they are appended to that file as JSON lines.
"""
import json
import os

import numpy as np

TOL_F32 = 1e-4   # max|err| / RMS(ref), fp32 path
TOL_BF16 = 2e-2  # max|err| / RMS(ref), bf16 path

BF16_U = 2.0 ** -8   # unit roundoff of bf16 (half an ulp, relative)
F16_U = 2.0 ** -11   # unit roundoff of f16
_U = {"fp32": 0.0, "bf16": BF16_U, "f16": F16_U}


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


def _record(what, stored, tol, plain, excess, rms):
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "tensor": what, "stored": stored,
           "tol": tol, "plain": plain, "beyond_rounding": excess, "rms": rms}
    path = os.environ.get("MTGR_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
    print(f"PARITY {rec['test']} {what} [{stored}] plain {plain:.3e} beyond-rounding {excess:.3e} (tol {tol:.0e})")


def check(got, ref, tol, what="", stored="fp32"):
    """Assert the bound for a result stored as `stored` ("fp32", "bf16" or
    "f16"); returns (figure held to tol, plain ratio)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    if ref.size == 0:
        return 0.0, 0.0
    u = _U[stored]
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    exc = float(np.maximum(err - u * np.abs(ref), 0.0).max())
    plain = float(err.max())
    if rms == 0.0:
        _record(what, stored, tol, plain, exc, rms)
        assert exc <= 1e-6, f"{what}: max|err| {exc:.3e} with zero reference"
        return exc, plain
    _record(what, stored, tol, plain / rms, exc / rms, rms)
    if stored == "fp32":
        assert plain / rms <= tol, (f"{what}: max|err|/RMS = {plain / rms:.3e} > {tol:.1e} "
                                    f"(max|err| {plain:.3e}, RMS {rms:.3e})")
    else:
        assert exc / rms <= tol, (f"{what}: error beyond {stored} rounding {exc / rms:.3e}/RMS > {tol:.1e} "
                                  f"(plain max|err|/RMS {plain / rms:.3e})")
    return exc / rms, plain / rms


def assert_close(got, ref, tol, what=""):
    """Plain max|err|/RMS(ref) <= tol (fp32-stored results)."""
    return check(got, ref, tol, what, "fp32")[1]


def assert_close_bf16(got, ref, tol=TOL_BF16, what=""):
    """Bound for a bf16-stored result: error beyond one bf16 rounding."""
    return check(got, ref, tol, what, "bf16")


def assert_close_f16(got, ref, tol=TOL_BF16, what=""):
    """Bound for an f16-stored result: error beyond one f16 rounding."""
    return check(got, ref, tol, what, "f16")


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
