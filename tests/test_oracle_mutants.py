"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source to a temporary directory, plants one
plausible mistake there (a dropped term, a wrong sign or comparison, a wrong
index or operand), compiles it, and runs every pin of test_oracle_pins.py
against the mutant: at least one pin has to fail.  The committed oracle is
never modified.
"""
import importlib.util
import inspect
import os
import shutil

import pytest

import tests.test_oracle_pins as pins

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")

MUTANTS = {
    "rt_rows_strict": ("if (gi == G_RT) return ts[j] <= ts[i];", "if (gi == G_RT) return ts[j] < ts[i];"),
    "cand_rows_not_strict": ("if (gi == G_CAND) return ts[j] < ts[i];", "if (gi == G_CAND) return ts[j] <= ts[i];"),
    "static_rows_see_rt": ("        return 0;                          /* User/Seq rows", "        return 1;                          /* User/Seq rows"),
    "cand_sees_all_cands": ("return i == j;", "return 1;"),
    "no_score_scale": ("const double c = 1.0 / sqrt((double)dh);\n#pragma omp parallel for schedule(dynamic, 1)\n    for (int b = 0; b < B; ++b) {\n        const int64_t s0 = offsets[b], s1 = offsets[b + 1];\n        const double nu = n_override > 0 ? n_override : (double)(s1 - s0);\n        double* acc",
                       "const double c = 1.0;\n#pragma omp parallel for schedule(dynamic, 1)\n    for (int b = 0; b < B; ++b) {\n        const int64_t s0 = offsets[b], s1 = offsets[b + 1];\n        const double nu = n_override > 0 ? n_override : (double)(s1 - s0);\n        double* acc"),
    "n_u_off_by_one": ("const double nu = n_override > 0 ? n_override : (double)(s1 - s0);\n        double* acc",
                       "const double nu = n_override > 0 ? n_override : (double)(s1 - s0 + 1);\n        double* acc"),
    "silu_grad_sign": ("const double ds = dA * sg * (1.0 + s * (1.0 - sg)) / nu;", "const double ds = dA * sg * (1.0 - s * (1.0 - sg)) / nu;"),
    "dk_wrong_operand": ("dk[j * ldg + h * dh + d] += ds * c * qi[d];", "dk[j * ldg + h * dh + d] += ds * c * kj[d];"),
    "gate_bwd_drops_term": ("dO[t * n + f] = r * (g - m1 - oh * m2);", "dO[t * n + f] = r * (g - m1);"),
    "gln_shared_gamma": ("y[t * D + f] = (xr[f] - mu) * r * gamma[g * D + f] + beta[g * D + f];",
                         "y[t * D + f] = (xr[f] - mu) * r * gamma[f] + beta[g * D + f];"),
    "gln_var_unbiased": ("    var /= D;\n        const double r = 1.0 / sqrt(var + eps);\n        for (int f = 0; f < D; ++f) y[",
                         "    var /= (D - 1);\n        const double r = 1.0 / sqrt(var + eps);\n        for (int f = 0; f < D; ++f) y["),
    "layer_no_residual": ("for (int64_t e = 0; e < T * D; ++e) x_out[e] += x[e];", ""),
    "layer_uqkv_order": ("a + HD, a + 2 * HD, a + 3 * HD, 4 * HD, 0.0, O);", "a + 2 * HD, a + HD, a + 3 * HD, 4 * HD, 0.0, O);"),
    "dgamma_wrong_group": ("sg[g] += dy[t * D + f] * (x[t * D + f] - mus[t]) * rs[t];",
                           "sg[0] += dy[t * D + f] * (x[t * D + f] - mus[t]) * rs[t];"),
    "dv_without_1_over_n": ("const double a = s * sg / nu;", "const double a = s * sg;"),
    "dv_wrong_operand": ("dv[j * ldg + h * dh + d] += a * gi[d];", "dv[j * ldg + h * dh + d] += a * qi[d];"),
    "dq_without_scale": ("dq[i * ldg + h * dh + d] += ds * c * kj[d];", "dq[i * ldg + h * dh + d] += ds * kj[d];"),
    "gate_eps_outside_sqrt": ("        var /= n;\n        const double r = 1.0 / sqrt(var + eps);\n        for (int f = 0; f < n; ++f) Y[",
                              "        var /= n;\n        const double r = 1.0 / (sqrt(var) + eps);\n        for (int f = 0; f < n; ++f) Y["),
    "gate_bwd_du_unnormalised": ("dU[t * ldg + f] = dY[t * n + f] * oh;", "dU[t * ldg + f] = dY[t * n + f] * o[f];"),
    "gln_bwd_drops_term": ("dx[t * D + f] = r * (gx - m1 - xh * m2);", "dx[t * D + f] = r * (gx - m1);"),
    "dbeta_wrong_group": ("sb[g] += dy[t * D + f];", "sb[0] += dy[t * D + f];"),
    "u_block_without_silu": ("for (int64_t e = 0; e < T * 4 * HD; ++e) a[e] = silu(z[e]);",
                             "for (int64_t e = 0; e < T * 4 * HD; ++e) a[e] = e % (4 * HD) < HD ? z[e] : silu(z[e]);"),
    "layer_bwd_silu_grad_is_sigmoid": ("da[e] *= sg * (1.0 + z[e] * (1.0 - sg));", "da[e] *= sg;"),
    "layer_bwd_no_residual_grad": ("for (int64_t e = 0; e < T * D; ++e) dx[e] += dx_out[e];", ""),
}


def _load_mutant(tmp_path, name, old, new):
    src = open(os.path.join(ORACLE_DIR, "mtgr_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    d = tmp_path / name
    d.mkdir()
    shutil.copy(os.path.join(ORACLE_DIR, "__init__.py"), d / "__init__.py")
    (d / "mtgr_oracle.c").write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}", d / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    return mod


def _pin_calls():
    calls = []
    for fname, fn in inspect.getmembers(pins, inspect.isfunction):
        if not fname.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        combos = [{}]
        for m in params:
            argnames = [a.strip() for a in m.args[0].split(",")] if isinstance(m.args[0], str) else m.args[0]
            new = []
            for c in combos:
                for val in m.args[1]:
                    vals = val if len(argnames) > 1 else (val,)
                    cc = dict(c)
                    cc.update(zip(argnames, vals))
                    new.append(cc)
            combos = new
        for c in combos[:1]:     # first parameter combination is enough here
            calls.append((fname, fn, c))
    return calls


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    mod = _load_mutant(tmp_path, name, old, new)
    failed = []
    for fname, fn, kw in _pin_calls():
        try:
            fn(orc=mod, **kw)
        except AssertionError:
            failed.append(fname)
        except Exception:   # a crash on the mutant counts as a catch too
            failed.append(fname)
    assert failed, f"no pin caught mutant {name}"
