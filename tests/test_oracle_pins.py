"""Pins of the fp64 oracle against what the pages and mathematics fix.

None of these tests re-types the oracle's formulas: each compares it with an
independent restatement (explicit mask matrix + numpy.matmul), a worked example
written by hand from the pages, a closed form, a library routine the oracle
does not call (torch layer_norm, numpy matmul), an invariant that the mask
rules imply, or central finite differences of the oracle's own forward.
"""
import math
import os

import numpy as np
import pytest

from hstu_attention_attn_b300 import synth
from oracle import bruteforce

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _batch_from(gid, ts, offsets=None):
    gid = np.asarray(gid, np.uint8)
    ts = np.asarray(ts, np.int64)
    if offsets is None:
        offsets = [0, len(gid)]
    return synth.Batch(np.asarray(offsets, np.int32), gid, ts)


# ---------------------------------------------------------------------------
# 1. brute force on tiny inputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("ts_hi", [86400, 16])   # 16: many equal stamps (<= vs <)
def test_core_matches_bruteforce(orc, seed, ts_hi):
    a = synth.tiny_attn(seed, ts_hi=ts_hi)
    b = a.batch
    O = orc.attn_core_fwd(b, a.H, a.dh, a.q, a.k, a.v)
    Ob = bruteforce.attn_core(b.offsets, b.gid, b.ts, a.H, a.dh, a.q, a.k, a.v)
    assert np.max(np.abs(O - Ob)) <= 1e-12 * max(1.0, np.abs(Ob).max())


@pytest.mark.parametrize("seed", [0, 5])
def test_visible_counts_match_bruteforce(orc, seed):
    a = synth.tiny_attn(seed, ts_hi=16)
    cnt, tot = orc.visible_counts(a.batch)
    ref = bruteforce.visible_counts(a.batch.offsets, a.batch.gid, a.batch.ts)
    assert np.array_equal(cnt, ref)
    assert tot == int(ref.sum())


# ---------------------------------------------------------------------------
# 2. the pages' worked example (fun-rec §7.3.4; paper-daily mask section)
# ---------------------------------------------------------------------------
def _read_golden_mask():
    toks, rows, mode = [], [], None
    with open(os.path.join(GOLD, "worked_example_mask.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line in ("tokens", "mask"):
                mode = line
                continue
            if mode == "tokens":
                i, g, t = line.split()
                toks.append((int(g), int(t)))
            else:
                rows.append([int(c) for c in line])
    return toks, np.array(rows)


def test_worked_example_mask(orc):
    toks, expect = _read_golden_mask()
    b = _batch_from([g for g, _ in toks], [t for _, t in toks])
    got = np.array([[orc.visible(i, j, b) for j in range(b.T)] for i in range(b.T)])
    assert np.array_equal(got, expect)
    cnt, tot = orc.visible_counts(b)
    assert np.array_equal(cnt, expect.sum(1)) and tot == expect.sum()


# ---------------------------------------------------------------------------
# 3. complexity exercise (fun-rec Problem 7.3.2): n = 1000 history tokens,
#    m = 200 candidates, no realtime -> n^2 + m*n + m visible pairs.
# ---------------------------------------------------------------------------
def test_visible_pairs_closed_form(orc):
    n, m = 1000, 200
    gid = [0] * 8 + [1] * (n - 8) + [3] * m
    ts = list(range(n + m))
    _, tot = orc.visible_counts(_batch_from(gid, ts))
    assert tot == n * n + m * n + m == 1_200_200


# ---------------------------------------------------------------------------
# 4. invariants of the mask (checked on O with n_u held fixed)
# ---------------------------------------------------------------------------
def _user(rng, nU, nS, nR, K, dh=16, H=2, rt_ts=None, c_ts=None):
    gid = [0] * nU + [1] * nS + [2] * nR + [3] * K
    ts = [0] * nU + list(range(-nS, 0)) \
        + (sorted(rng.integers(0, 1000, nR)) if rt_ts is None else list(rt_ts)) \
        + (sorted(rng.integers(0, 1000, K)) if c_ts is None else list(c_ts))
    T = len(gid)
    q, k, v = (rng.standard_normal((T, H * dh)) for _ in range(3))
    return np.array(gid, np.uint8), np.array(ts, np.int64), q, k, v


def _core(orc, gid, ts, q, k, v, H=2, dh=16, n=50.0):
    return orc.attn_core_fwd(_batch_from(gid, ts), H, dh, q, k, v, n_override=n)


def test_invariant_candidates_independent(orc):
    rng = np.random.default_rng(11)
    gid, ts, q, k, v = _user(rng, 3, 10, 6, 8)
    base = _core(orc, gid, ts, q, k, v)
    cand = np.where(gid == 3)[0]
    # remove two other candidates
    keep = np.array([i for i in range(len(gid)) if i not in (cand[1], cand[5])])
    O2 = _core(orc, gid[keep], ts[keep], q[keep], k[keep], v[keep])
    for new_i, old_i in enumerate(keep):
        if gid[old_i] == 3:
            assert np.allclose(O2[new_i], base[old_i], rtol=1e-13, atol=1e-15)
    # permute candidates
    perm = np.concatenate([np.arange(cand[0]), rng.permutation(cand)])
    O3 = _core(orc, gid[perm], ts[perm], q[perm], k[perm], v[perm])
    assert np.allclose(O3, base[perm], rtol=1e-13, atol=1e-15)
    # add three candidates with arbitrary stamps and values
    extra = 3
    gid4 = np.concatenate([gid, [3] * extra]).astype(np.uint8)
    ts4 = np.concatenate([ts, [5, 500, 999]])
    q4, k4, v4 = (np.concatenate([m, rng.standard_normal((extra, m.shape[1]))]) for m in (q, k, v))
    O4 = _core(orc, gid4, ts4, q4, k4, v4)
    assert np.allclose(O4[: len(gid)], base, rtol=1e-13, atol=1e-15)


def test_invariant_static_rows_ignore_realtime_and_candidates(orc):
    rng = np.random.default_rng(12)
    gid, ts, q, k, v = _user(rng, 3, 10, 6, 8)
    base = _core(orc, gid, ts, q, k, v)
    us = gid <= 1
    # edit every RealTime / candidate value and stamp
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for m in (q2, k2, v2):
        m[~us] = rng.standard_normal(m[~us].shape)
    ts2 = ts.copy()
    ts2[~us] = rng.integers(0, 1000, (~us).sum())
    O2 = _core(orc, gid, ts2, q2, k2, v2)
    assert np.allclose(O2[us], base[us], rtol=1e-13, atol=1e-15)
    # drop all RealTime and candidate tokens
    O3 = _core(orc, gid[us], ts[us], q[us], k[us], v[us])
    assert np.allclose(O3, base[us], rtol=1e-13, atol=1e-15)


def test_invariant_candidate_ignores_later_realtime(orc):
    rng = np.random.default_rng(13)
    gid, ts, q, k, v = _user(rng, 2, 6, 4, 3, rt_ts=[10, 20, 30, 40], c_ts=[25, 35, 50])
    base = _core(orc, gid, ts, q, k, v)
    # insert RealTime tokens stamped at or after the first candidate (25)
    ins = 2
    pos = np.where(gid == 2)[0][-1] + 1
    gid2 = np.insert(gid, pos, [2] * ins).astype(np.uint8)
    ts2 = np.insert(ts, pos, [25, 60])
    q2, k2, v2 = (np.insert(m, pos, rng.standard_normal((ins, m.shape[1])), axis=0) for m in (q, k, v))
    O2 = _core(orc, gid2, ts2, q2, k2, v2)
    first_c_old = np.where(gid == 3)[0][0]
    first_c_new = np.where(gid2 == 3)[0][0]
    assert np.allclose(O2[first_c_new], base[first_c_old], rtol=1e-13, atol=1e-15)
    # ... but the candidate at 35 sees the RT at 25 and must change
    assert not np.allclose(O2[first_c_new + 1], base[first_c_old + 1])


# ---------------------------------------------------------------------------
# 5. textbook special cases
# ---------------------------------------------------------------------------
def test_all_seq_segment_is_dense_bidirectional(orc):
    rng = np.random.default_rng(21)
    n, H, dh = 37, 2, 8
    q, k, v = (rng.standard_normal((n, H * dh)) for _ in range(3))
    O = orc.attn_core_fwd(_batch_from([1] * n, [0] * n), H, dh, q, k, v)
    for h in range(H):
        c = slice(h * dh, (h + 1) * dh)
        S = np.matmul(q[:, c], k[:, c].T) / math.sqrt(dh)
        ref = np.matmul(S * (1.0 / (1.0 + np.exp(-S))), v[:, c]) / n
        assert np.allclose(O[:, c], ref, rtol=1e-12, atol=1e-14)


def test_constant_rows_closed_form(orc):
    """Every row holds the same q and every key the same k (all static tokens):
    O_i = silu(q·k/sqrt(d)) * mean_j v_j (n_u = n, all pairs visible)."""
    rng = np.random.default_rng(22)
    n, dh = 9, 4
    qrow, krow = rng.standard_normal(dh), rng.standard_normal(dh)
    v = rng.standard_normal((n, dh))
    q = np.tile(qrow, (n, 1))
    k = np.tile(krow, (n, 1))
    O = orc.attn_core_fwd(_batch_from([0] * 3 + [1] * 6, [0] * n), 1, dh, q, k, v)
    s = float(qrow @ krow) / math.sqrt(dh)
    silu = s / (1.0 + math.exp(-s))
    assert np.allclose(O, silu * v.mean(0)[None, :], rtol=1e-12, atol=1e-14)


def test_empty_and_single_token_users(orc):
    gid = [1, 3, 0, 2]
    ts = [0, 5, 0, 9]
    b = _batch_from(gid, ts, offsets=[0, 0, 1, 1, 2, 4, 4])
    rng = np.random.default_rng(23)
    q, k, v = (rng.standard_normal((4, 4)) for _ in range(3))
    O = orc.attn_core_fwd(b, 1, 4, q, k, v)
    Ob = bruteforce.attn_core(b.offsets, b.gid, b.ts, 1, 4, q, k, v)
    assert np.allclose(O, Ob, rtol=1e-12, atol=1e-15)
    # a lone token sees itself: O = silu(q·k/2) v / 1
    s = q[0] @ k[0] / 2.0
    assert np.allclose(O[0], s / (1 + math.exp(-s)) * v[0])


def test_gln_equal_groups_is_layer_norm(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    T, D = 50, 24
    x = rng.standard_normal((T, D)) * 3 + 1
    gid = rng.integers(0, 4, T).astype(np.uint8)
    g1, b1 = rng.standard_normal(D), rng.standard_normal(D)
    y, mean, rstd = orc.gln_fwd(x, gid, np.tile(g1, (4, 1)), np.tile(b1, (4, 1)))
    ref = torch.nn.functional.layer_norm(torch.tensor(x), (D,), torch.tensor(g1), torch.tensor(b1), eps=1e-5)
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_gln_groups_use_their_own_parameters(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(32)
    T, D = 40, 16
    x = rng.standard_normal((T, D))
    gid = rng.integers(0, 4, T).astype(np.uint8)
    gam, bet = rng.standard_normal((4, D)), rng.standard_normal((4, D))
    y, _, _ = orc.gln_fwd(x, gid, gam, bet)
    for g in range(4):
        rows = gid == g
        ref = torch.nn.functional.layer_norm(torch.tensor(x[rows]), (D,), torch.tensor(gam[g]),
                                             torch.tensor(bet[g]), eps=1e-5)
        assert np.allclose(y[rows], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_ln_gate_is_layer_norm_times_u(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(33)
    O = rng.standard_normal((30, 64)) * 0.01
    U = rng.standard_normal((30, 64))
    Y, _, _ = orc.ln_gate_fwd(O, U)
    ref = torch.nn.functional.layer_norm(torch.tensor(O), (64,), eps=1e-5).numpy() * U
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_matmuls_match_numpy(orc):
    rng = np.random.default_rng(34)
    A, Bm = rng.standard_normal((7, 5)), rng.standard_normal((5, 9))
    assert np.allclose(orc.matmul(A, Bm), A @ Bm, rtol=1e-13)
    assert np.allclose(orc.matmul_nt(A, Bm.T.copy()), A @ Bm, rtol=1e-13)
    assert np.allclose(orc.matmul_tn(A.T.copy(), Bm), A @ Bm, rtol=1e-13)


# ---------------------------------------------------------------------------
# 6. gradients: central finite differences of the oracle's own forward
# ---------------------------------------------------------------------------
def _fd_dir(f, x, d, h=1e-5):
    return (f(x + h * d) - f(x - h * d)) / (2 * h)


def _check_grad(f, x, g, rng, n_dirs=4, n_coords=3):
    for _ in range(n_dirs):
        d = rng.standard_normal(x.shape)
        fd = _fd_dir(f, x, d)
        an = float(np.sum(g * d))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)
    flat = x.reshape(-1)
    for idx in rng.choice(flat.size, n_coords, replace=False):
        d = np.zeros_like(flat)
        d[idx] = 1.0
        d = d.reshape(x.shape)
        fd = _fd_dir(f, x, d)
        an = float(g.reshape(-1)[idx])
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (idx, fd, an)


@pytest.mark.parametrize("ts_hi", [86400, 16])
def test_attention_grads_finite_difference(orc, ts_hi):
    a = synth.tiny_attn(4, ts_hi=ts_hi)
    b, H, dh = a.batch, a.H, a.dh
    rng = np.random.default_rng(41)
    dY = rng.standard_normal((b.T, H * dh))
    q, k, v, u = (np.asarray(m, np.float64) for m in (a.q, a.k, a.v, a.u))
    dq, dk, dv, du = orc.attn_bwd(b, H, dh, q, k, v, u, dY)

    def loss(qq=q, kk=k, vv=v, uu=u):
        Y, _, _, _ = orc.attn_fwd(b, H, dh, qq, kk, vv, uu)
        return float(np.sum(Y * dY))

    _check_grad(lambda t: loss(qq=t), q, dq, rng)
    _check_grad(lambda t: loss(kk=t), k, dk, rng)
    _check_grad(lambda t: loss(vv=t), v, dv, rng)
    _check_grad(lambda t: loss(uu=t), u, du, rng)


def test_gln_grads_finite_difference(orc):
    rng = np.random.default_rng(42)
    T, D = 20, 12
    x = rng.standard_normal((T, D))
    gid = rng.integers(0, 4, T).astype(np.uint8)
    gam, bet = rng.standard_normal((4, D)), rng.standard_normal((4, D))
    dy = rng.standard_normal((T, D))
    dx, dg, db = orc.gln_bwd(dy, x, gid, gam)

    def loss(xx=x, gg=gam, bb=bet):
        return float(np.sum(orc.gln_fwd(xx, gid, gg, bb)[0] * dy))

    _check_grad(lambda t: loss(xx=t), x, dx, rng)
    _check_grad(lambda t: loss(gg=t), gam, dg, rng)
    _check_grad(lambda t: loss(bb=t), bet, db, rng)


def test_layer_grads_finite_difference(orc):
    L = synth.tiny_layer(5)
    b = L.batch
    args = dict(D=L.D, H=L.H, dh=L.dh)
    p = {k: np.asarray(getattr(L, k), np.float64) for k in ("x", "w_uqkv", "w_o", "gamma", "beta")}
    dxo = np.asarray(L.dx_out, np.float64)
    g = orc.layer_bwd(b, **args, **p, dx_out=dxo)
    rng = np.random.default_rng(43)

    def loss(**kw):
        pp = dict(p)
        pp.update(kw)
        return float(np.sum(orc.layer_fwd(b, **args, **pp)["x_out"] * dxo))

    _check_grad(lambda t: loss(x=t), p["x"], g["dx"], rng, n_dirs=2, n_coords=2)
    _check_grad(lambda t: loss(w_uqkv=t), p["w_uqkv"], g["dw_uqkv"], rng, n_dirs=2, n_coords=2)
    _check_grad(lambda t: loss(w_o=t), p["w_o"], g["dw_o"], rng, n_dirs=2, n_coords=2)
    _check_grad(lambda t: loss(gamma=t), p["gamma"], g["dgamma"], rng, n_dirs=2, n_coords=2)
    _check_grad(lambda t: loss(beta=t), p["beta"], g["dbeta"], rng, n_dirs=2, n_coords=2)


def test_layer_forward_composes_documented_steps(orc):
    """The layer equals GLN -> x·W -> SiLU -> attention -> LN⊙U -> ·W_o + x,
    each step checked against numpy / torch rather than the oracle itself."""
    torch = pytest.importorskip("torch")
    L = synth.tiny_layer(6)
    b = L.batch
    HD = L.H * L.dh
    out = orc.layer_fwd(b, L.D, L.H, L.dh, L.x, L.w_uqkv, L.w_o, L.gamma, L.beta)
    x = np.asarray(L.x, np.float64)
    xn = np.zeros_like(x)
    for g in range(4):
        r = b.gid == g
        xn[r] = torch.nn.functional.layer_norm(torch.tensor(x[r]), (L.D,), torch.tensor(L.gamma[g], dtype=torch.float64),
                                               torch.tensor(L.beta[g], dtype=torch.float64), eps=1e-5).numpy()
    z = xn @ np.asarray(L.w_uqkv, np.float64)
    a = z * (1.0 / (1.0 + np.exp(-z)))
    U, Q, K, V = (a[:, i * HD:(i + 1) * HD] for i in range(4))
    O = bruteforce.attn_core(b.offsets, b.gid, b.ts, L.H, L.dh, Q, K, V)
    Y = torch.nn.functional.layer_norm(torch.tensor(O), (HD,), eps=1e-5).numpy() * U
    xo = x + Y @ np.asarray(L.w_o, np.float64)
    assert np.allclose(out["xn"], xn, rtol=1e-11, atol=1e-11)
    assert np.allclose(out["z"], z, rtol=1e-11, atol=1e-11)
    assert np.allclose(out["o"], O, rtol=1e-10, atol=1e-12)
    assert np.allclose(out["x_out"], xo, rtol=1e-10, atol=1e-10)


def test_attention_grads_match_torch_autograd(orc):
    """Second, independent check of the analytic backward: torch autograd on an
    fp64 restatement (explicit mask matrix) of the attention op."""
    torch = pytest.importorskip("torch")
    a = synth.tiny_attn(7, ts_hi=16)
    b, H, dh = a.batch, a.H, a.dh
    rng = np.random.default_rng(44)
    dY = rng.standard_normal((b.T, H * dh))
    dq, dk, dv, du = orc.attn_bwd(b, H, dh, a.q, a.k, a.v, a.u, dY)
    q, k, v, u = (torch.tensor(np.asarray(m, np.float64), requires_grad=True) for m in (a.q, a.k, a.v, a.u))
    Os = []
    for s in range(b.B):
        s0, s1 = int(b.offsets[s]), int(b.offsets[s + 1])
        M = torch.tensor(bruteforce.mask_matrix(b.gid[s0:s1], b.ts[s0:s1]), dtype=torch.float64)
        heads = []
        for h in range(H):
            c = slice(h * dh, (h + 1) * dh)
            S = q[s0:s1, c] @ k[s0:s1, c].T / math.sqrt(dh)
            heads.append((torch.nn.functional.silu(S) * M / (s1 - s0)) @ v[s0:s1, c])
        Os.append(torch.cat(heads, 1))
    O = torch.cat(Os, 0)
    Y = torch.nn.functional.layer_norm(O, (H * dh,), eps=1e-5) * u
    (Y * torch.tensor(dY)).sum().backward()
    for mine, ref in ((dq, q.grad), (dk, k.grad), (dv, v.grad), (du, u.grad)):
        assert np.allclose(mine, ref.numpy(), rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_layer_blas_composition_equals_c_layer(orc, case):
    """``layer_fwd_blas`` / ``layer_bwd_blas`` (the pinned steps with numpy's
    matmul for the products, used where the C layer's index-order loops are too
    slow) equal the C layer, which the finite-difference and composition pins
    above hold, on every output and gradient to fp64 summation-order noise."""
    if case == "tiny":
        L = synth.tiny_layer(8)
    else:
        L = synth.layer_inputs(9, lambda r: [(8, 150, 20, 20), (4, 40, 0, 3), (0, 0, 5, 2)], 64, 2, 32)
    b = L.batch
    args = (b, L.D, L.H, L.dh, L.x, L.w_uqkv, L.w_o, L.gamma, L.beta)
    f_c, f_b = orc.layer_fwd(*args), orc.layer_fwd_blas(*args)
    for k in ("x_out", "xn", "z", "o", "y"):
        assert np.allclose(f_b[k], f_c[k], rtol=1e-11, atol=1e-12 * max(1.0, np.abs(f_c[k]).max())), k
    g_c, g_b = orc.layer_bwd(*args, L.dx_out), orc.layer_bwd_blas(*args, L.dx_out)
    for k in ("dx", "dw_uqkv", "dw_o", "dgamma", "dbeta"):
        assert np.allclose(g_b[k], g_c[k], rtol=1e-10, atol=1e-11 * max(1.0, np.abs(g_c[k]).max())), k
