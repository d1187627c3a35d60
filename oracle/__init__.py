"""fp64 CPU oracle of the MTGR HSTU layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path.

``liboracle.so`` is compiled from ``mtgr_oracle.c`` (plain C, fp64, OpenMP);
this module marshals numpy arrays into it and, for batches too large for the
C loops' index-order products, composes the layer from the same C steps with
numpy's matmul (``layer_fwd_blas`` / ``layer_bwd_blas``, pinned to the C layer).
``bruteforce.py`` is an independent NumPy restatement used to pin the C code.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mtgr_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

EPS_GLN = 1e-5
EPS_LN = 1e-5


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (no CUDA involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        P = C.c_void_p
        i64, i32, dbl = C.c_int64, C.c_int, C.c_double
        sig = {
            "orc_visible": (C.c_int, [i64, i64, P, P]),
            "orc_visible_counts": (None, [i32, P, P, P, P, P]),
            "orc_attn_core_fwd": (None, [i32, P, P, P, i32, i32, P, P, P, i64, dbl, P]),
            "orc_attn_core_bwd": (None, [i32, P, P, P, i32, i32, P, P, P, i64, dbl, P, P, P, P, i64]),
            "orc_ln_gate_fwd": (None, [i64, i32, P, P, i64, dbl, P, P, P]),
            "orc_ln_gate_bwd": (None, [i64, i32, P, P, P, i64, dbl, P, P, i64]),
            "orc_gln_fwd": (None, [i64, i32, P, P, P, P, dbl, P, P, P]),
            "orc_gln_bwd": (None, [i64, i32, P, P, P, P, dbl, P, P, P]),
            "orc_matmul": (None, [i64, i64, i64, P, P, P]),
            "orc_matmul_nt": (None, [i64, i64, i64, P, P, P]),
            "orc_matmul_tn": (None, [i64, i64, i64, P, P, P]),
            "orc_layer_fwd": (None, [i32, P, P, P, i64, i32, i32, i32, P, P, P, P, P, dbl, dbl,
                                     P, P, P, P, P]),
            "orc_layer_bwd": (None, [i32, P, P, P, i64, i32, i32, i32, P, P, P, P, P, dbl, dbl,
                                     P, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(_lib, name)
            f.restype = res
            f.argtypes = args
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _meta(batch):
    off = np.ascontiguousarray(batch.offsets, np.int32)
    gid = np.ascontiguousarray(batch.gid, np.uint8)
    ts = np.ascontiguousarray(batch.ts, np.int64)
    return off, gid, ts


# ---------------------------------------------------------------------------
def visible(i, j, batch) -> int:
    off, gid, ts = _meta(batch)
    return int(_load().orc_visible(i, j, _p(gid), _p(ts)))


def visible_counts(batch):
    off, gid, ts = _meta(batch)
    cnt = np.zeros(batch.T, np.int32)
    tot = np.zeros(1, np.int64)
    _load().orc_visible_counts(batch.B, _p(off), _p(gid), _p(ts), _p(cnt), _p(tot))
    return cnt, int(tot[0])


def attn_core_fwd(batch, H, dh, q, k, v, n_override=0.0):
    """q, k, v: [T, ld] with head h in columns h*dh..; returns O [T, H*dh]."""
    off, gid, ts = _meta(batch)
    q, k, v = _f64(q), _f64(k), _f64(v)
    assert q.shape == k.shape == v.shape
    O = np.zeros((batch.T, H * dh))
    _load().orc_attn_core_fwd(batch.B, _p(off), _p(gid), _p(ts), H, dh, _p(q), _p(k), _p(v),
                              q.shape[1] if q.ndim == 2 else H * dh, float(n_override), _p(O))
    return O


def attn_core_bwd(batch, H, dh, q, k, v, dO, n_override=0.0):
    off, gid, ts = _meta(batch)
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    HD = H * dh
    dq, dk, dv = (np.zeros((batch.T, HD)) for _ in range(3))
    _load().orc_attn_core_bwd(batch.B, _p(off), _p(gid), _p(ts), H, dh, _p(q), _p(k), _p(v),
                              q.shape[1], float(n_override), _p(dO), _p(dq), _p(dk), _p(dv), HD)
    return dq, dk, dv


def ln_gate_fwd(O, U, eps=EPS_LN):
    O, U = _f64(O), _f64(U)
    T, n = O.shape
    Y = np.zeros((T, n))
    mean, rstd = np.zeros(T), np.zeros(T)
    _load().orc_ln_gate_fwd(T, n, _p(O), _p(U), U.shape[1], eps, _p(Y), _p(mean), _p(rstd))
    return Y, mean, rstd


def ln_gate_bwd(dY, O, U, eps=EPS_LN):
    dY, O, U = _f64(dY), _f64(O), _f64(U)
    T, n = O.shape
    dO, dU = np.zeros((T, n)), np.zeros((T, n))
    _load().orc_ln_gate_bwd(T, n, _p(dY), _p(O), _p(U), U.shape[1], eps, _p(dO), _p(dU), n)
    return dO, dU


def attn_fwd(batch, H, dh, q, k, v, u, eps=EPS_LN, n_override=0.0):
    """Full attention op: Y = LN(A·V) ⊙ U.  Returns (Y, O, mean, rstd)."""
    O = attn_core_fwd(batch, H, dh, q, k, v, n_override)
    Y, mean, rstd = ln_gate_fwd(O, u, eps)
    return Y, O, mean, rstd


def attn_bwd(batch, H, dh, q, k, v, u, dY, eps=EPS_LN, n_override=0.0):
    """Returns (dq, dk, dv, du) for the full attention op."""
    O = attn_core_fwd(batch, H, dh, q, k, v, n_override)
    dO, du = ln_gate_bwd(dY, O, u, eps)
    dq, dk, dv = attn_core_bwd(batch, H, dh, q, k, v, dO, n_override)
    return dq, dk, dv, du


def gln_fwd(x, gid, gamma, beta, eps=EPS_GLN):
    x, gamma, beta = _f64(x), _f64(gamma), _f64(beta)
    gid = np.ascontiguousarray(gid, np.uint8)
    T, D = x.shape
    y = np.zeros((T, D))
    mean, rstd = np.zeros(T), np.zeros(T)
    _load().orc_gln_fwd(T, D, _p(x), _p(gid), _p(gamma), _p(beta), eps, _p(y), _p(mean), _p(rstd))
    return y, mean, rstd


def gln_bwd(dy, x, gid, gamma, eps=EPS_GLN):
    dy, x, gamma = _f64(dy), _f64(x), _f64(gamma)
    gid = np.ascontiguousarray(gid, np.uint8)
    T, D = x.shape
    dx = np.zeros((T, D))
    dg, db = np.zeros((4, D)), np.zeros((4, D))
    _load().orc_gln_bwd(T, D, _p(dy), _p(x), _p(gid), _p(gamma), eps, _p(dx), _p(dg), _p(db))
    return dx, dg, db


def matmul(A, B):
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    Cm = np.zeros((M, N))
    _load().orc_matmul(M, N, K, _p(A), _p(B), _p(Cm))
    return Cm


def matmul_nt(A, B):
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    Cm = np.zeros((M, N))
    _load().orc_matmul_nt(M, N, K, _p(A), _p(B), _p(Cm))
    return Cm


def matmul_tn(A, B):
    A, B = _f64(A), _f64(B)
    K, M = A.shape
    K2, N = B.shape
    assert K == K2
    Cm = np.zeros((M, N))
    _load().orc_matmul_tn(M, N, K, _p(A), _p(B), _p(Cm))
    return Cm


def layer_fwd(batch, D, H, dh, x, w_uqkv, w_o, gamma, beta, eps_gln=EPS_GLN, eps_ln=EPS_LN):
    """Returns dict with x_out and the saved intermediates xn, z, o, y."""
    off, gid, ts = _meta(batch)
    x, w_uqkv, w_o, gamma, beta = map(_f64, (x, w_uqkv, w_o, gamma, beta))
    T, HD = batch.T, H * dh
    out = dict(x_out=np.zeros((T, D)), xn=np.zeros((T, D)), z=np.zeros((T, 4 * HD)),
               o=np.zeros((T, HD)), y=np.zeros((T, HD)))
    _load().orc_layer_fwd(batch.B, _p(off), _p(gid), _p(ts), T, D, H, dh, _p(x), _p(w_uqkv),
                          _p(w_o), _p(gamma), _p(beta), eps_gln, eps_ln, _p(out["x_out"]),
                          _p(out["xn"]), _p(out["z"]), _p(out["o"]), _p(out["y"]))
    return out


def layer_bwd(batch, D, H, dh, x, w_uqkv, w_o, gamma, beta, dx_out, eps_gln=EPS_GLN, eps_ln=EPS_LN):
    """Returns dict dx, dw_uqkv, dw_o, dgamma, dbeta."""
    off, gid, ts = _meta(batch)
    x, w_uqkv, w_o, gamma, beta, dx_out = map(_f64, (x, w_uqkv, w_o, gamma, beta, dx_out))
    T, HD = batch.T, H * dh
    out = dict(dx=np.zeros((T, D)), dw_uqkv=np.zeros((D, 4 * HD)), dw_o=np.zeros((HD, D)),
               dgamma=np.zeros((4, D)), dbeta=np.zeros((4, D)))
    _load().orc_layer_bwd(batch.B, _p(off), _p(gid), _p(ts), T, D, H, dh, _p(x), _p(w_uqkv),
                          _p(w_o), _p(gamma), _p(beta), eps_gln, eps_ln, _p(dx_out),
                          _p(out["dx"]), _p(out["dw_uqkv"]), _p(out["dw_o"]), _p(out["dgamma"]),
                          _p(out["dbeta"]))
    return out


def silu(z):
    """Elementwise SiLU in fp64 (σ written out), for composing oracle steps."""
    z = _f64(z)
    return z / (1.0 + np.exp(-z))


def silu_grad(z):
    z = _f64(z)
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def layer_fwd_blas(batch, D, H, dh, x, w_uqkv, w_o, gamma, beta, eps_gln=EPS_GLN, eps_ln=EPS_LN):
    """The layer forward of ``layer_fwd`` (paper-daily "模型怎么搭": GLN, UQKV +
    SiLU, masked SiLU attention, LN(O) ⊙ U, output linear + residual) composed
    from the same pinned steps (``gln_fwd``, ``attn_core_fwd``, ``ln_gate_fwd``),
    with its two products taken by numpy's matmul (a library primitive).  The
    plain C loops sum in index order and need hours for a 60k-token batch at
    d_model 1024; this differs from ``layer_fwd`` only in summation order.
    Returns the same dict (x_out, xn, z, o, y)."""
    x, w_uqkv, w_o = _f64(x), _f64(w_uqkv), _f64(w_o)
    HD = H * dh
    xn, _, _ = gln_fwd(x, batch.gid, gamma, beta, eps_gln)
    z = xn @ w_uqkv
    a = silu(z)
    O = attn_core_fwd(batch, H, dh, a[:, HD:2 * HD], a[:, 2 * HD:3 * HD], a[:, 3 * HD:])
    Y, _, _ = ln_gate_fwd(O, a[:, :HD], eps_ln)
    return dict(x_out=x + Y @ w_o, xn=xn, z=z, o=O, y=Y)


def layer_bwd_blas(batch, D, H, dh, x, w_uqkv, w_o, gamma, beta, dx_out, eps_gln=EPS_GLN, eps_ln=EPS_LN):
    """The layer backward of ``layer_bwd`` composed from the pinned steps with
    numpy's matmul for the four products (see ``layer_fwd_blas``):
    dY = dx'·W_oᵀ, dW_o = Yᵀ·dx', gate and attention backward,
    dz = [dU|dQ|dK|dV] ⊙ silu'(z), dW_uqkv = xnᵀ·dz, dxn = dz·W_uqkvᵀ, GLN
    backward plus the residual.  Returns dict dx, dw_uqkv, dw_o, dgamma, dbeta."""
    x, w_uqkv, w_o, dx_out = _f64(x), _f64(w_uqkv), _f64(w_o), _f64(dx_out)
    HD = H * dh
    f = layer_fwd_blas(batch, D, H, dh, x, w_uqkv, w_o, gamma, beta, eps_gln, eps_ln)
    a = silu(f["z"])
    dY = dx_out @ w_o.T
    dw_o = f["y"].T @ dx_out
    dO, du = ln_gate_bwd(dY, f["o"], a[:, :HD], eps_ln)
    del dY
    dq, dk, dv = attn_core_bwd(batch, H, dh, a[:, HD:2 * HD], a[:, 2 * HD:3 * HD], a[:, 3 * HD:], dO)
    del dO, a
    dz = np.concatenate([du, dq, dk, dv], axis=1)
    del du, dq, dk, dv
    dz *= silu_grad(f["z"])
    dw_uqkv = f["xn"].T @ dz
    dxn = dz @ w_uqkv.T
    del dz
    dx, dg, db = gln_bwd(dxn, x, batch.gid, gamma, eps_gln)
    return dict(dx=dx + dx_out, dw_uqkv=dw_uqkv, dw_o=dw_o, dgamma=dg, dbeta=db)
