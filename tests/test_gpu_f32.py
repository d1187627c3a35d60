"""fp32 path vs the fp64 oracle: max|err|/RMS(ref) <= 1e-4 on every output and gradient."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import mtgr, synth
from hstu_attention_attn_b300.layer import HstuAttention, HstuLayer, device_batch
from tests.gpu_common import dev, need_gpu, ragged_users
from tests.util import TOL_F32, assert_close, to_np

pytestmark = pytest.mark.gpu
F32 = torch.float32


def _attn_case(seed, ts_hi):
    return synth.tiny_attn(seed, ts_hi=ts_hi)


@pytest.mark.parametrize("seed,ts_hi", [(0, 86400), (1, 16), (2, 86400)])
def test_attention_fwd_bwd_f32(orc, seed, ts_hi):
    need_gpu()
    a = _attn_case(seed, ts_hi)
    b, H, dh = a.batch, a.H, a.dh
    db = device_batch(b)
    q, k, v, u = (dev(m, F32) for m in (a.q, a.k, a.v, a.u))
    op = HstuAttention(H, dh, F32)
    y, saved = op.forward(q, k, v, u, db)
    Y, O, mean, rstd = orc.attn_fwd(b, H, dh, a.q, a.k, a.v, a.u)
    torch.cuda.synchronize()
    assert_close(to_np(saved[0]), O, TOL_F32, "O")
    assert_close(to_np(y), Y, TOL_F32, "Y")
    assert_close(to_np(saved[1]), mean, TOL_F32, "ln mean")
    assert_close(to_np(saved[2]), rstd, TOL_F32, "ln rstd")
    rng = np.random.default_rng(100 + seed)
    dY = rng.standard_normal(y.shape).astype(np.float32)
    dq, dk, dv, du = op.backward(dev(dY, F32), q, k, v, u, saved, db)
    ref = orc.attn_bwd(b, H, dh, a.q, a.k, a.v, a.u, dY)
    torch.cuda.synchronize()
    for name, got, r in zip(("dq", "dk", "dv", "du"), (dq, dk, dv, du), ref):
        assert_close(to_np(got), r, TOL_F32, name)


def test_attention_f32_ragged_and_degenerate_users(orc):
    need_gpu()
    rng = np.random.default_rng(5)
    b = synth.make_batch(rng, ragged_users(), ts_hi=200)
    H, dh = 2, 32
    q, k, v, u = (rng.standard_normal((b.T, H * dh)).astype(np.float32) for _ in range(4))
    db = device_batch(b)
    op = HstuAttention(H, dh, F32)
    y, saved = op.forward(dev(q, F32), dev(k, F32), dev(v, F32), dev(u, F32), db)
    Y, O, _, _ = orc.attn_fwd(b, H, dh, q, k, v, u)
    torch.cuda.synchronize()
    assert_close(to_np(saved[0]), O, TOL_F32, "O")
    assert_close(to_np(y), Y, TOL_F32, "Y")


def test_gln_f32(orc):
    need_gpu()
    rng = np.random.default_rng(9)
    T, D = 300, 64
    x = (rng.standard_normal((T, D)) * 2 + 0.5).astype(np.float32)
    gid = rng.integers(0, 4, T).astype(np.uint8)
    gam, bet = synth.gln_params(rng, D)
    y = torch.empty(T, D, device="cuda")
    mean = torch.empty(T, device="cuda")
    rstd = torch.empty(T, device="cuda")
    xt, gt = dev(x, F32), dev(gid, torch.uint8)
    gamt, bett = dev(gam, F32), dev(bet, F32)
    mtgr.mtgr_group_layernorm_fwd(xt, y, mean, rstd, gt, gamt, bett, 1e-5)
    ry, rm, rr = orc.gln_fwd(x, gid, gam, bet)
    torch.cuda.synchronize()
    assert_close(to_np(y), ry, TOL_F32, "y")
    dy = rng.standard_normal((T, D)).astype(np.float32)
    dx = torch.empty(T, D, device="cuda")
    dg = torch.empty(4, D, device="cuda")
    dbt = torch.empty(4, D, device="cuda")
    ws = torch.empty(mtgr.mtgr_group_layernorm_bwd_workspace_size(T, D), dtype=torch.uint8, device="cuda")
    mtgr.mtgr_group_layernorm_bwd(dev(dy, F32), xt, mean, rstd, gt, gamt, None, dx, dg, dbt, ws)
    rdx, rdg, rdb = orc.gln_bwd(dy, x, gid, gam)
    torch.cuda.synchronize()
    assert_close(to_np(dx), rdx, TOL_F32, "dx")
    assert_close(to_np(dg), rdg, TOL_F32, "dgamma")
    assert_close(to_np(dbt), rdb, TOL_F32, "dbeta")


@pytest.mark.parametrize("seed", [0, 3])
def test_layer_f32(orc, seed):
    need_gpu()
    L = synth.tiny_layer(seed)
    b = L.batch
    db = device_batch(b)
    layer = HstuLayer(L.D, L.H, L.dh, torch.from_numpy(L.w_uqkv), torch.from_numpy(L.w_o),
                      torch.from_numpy(L.gamma), torch.from_numpy(L.beta), dtype=F32)
    x = dev(L.x, F32)
    x_out, saved = layer.forward(x, db)
    ref = orc.layer_fwd(b, L.D, L.H, L.dh, L.x, L.w_uqkv, L.w_o, L.gamma, L.beta)
    torch.cuda.synchronize()
    assert_close(to_np(saved["xn"]), ref["xn"], TOL_F32, "xn")
    assert_close(to_np(saved["dsilu"]), orc.silu_grad(ref["z"]), TOL_F32, "silu'(z)")
    assert_close(to_np(saved["o"]), ref["o"], TOL_F32, "o")
    assert_close(to_np(saved["y"]), ref["y"], TOL_F32, "y")
    assert_close(to_np(x_out), ref["x_out"], TOL_F32, "x_out")
    dx, g = layer.backward(x, saved, dev(L.dx_out, F32), db)
    rb = orc.layer_bwd(b, L.D, L.H, L.dh, L.x, L.w_uqkv, L.w_o, L.gamma, L.beta, L.dx_out)
    torch.cuda.synchronize()
    assert_close(to_np(dx), rb["dx"], TOL_F32, "dx")
    for n in ("dw_uqkv", "dw_o", "dgamma", "dbeta"):
        assert_close(to_np(g[n]), rb[n], TOL_F32, n)
