"""bf16 HSTU layer (tcgen05 GEMMs + attention) vs the fp64 oracle.

Each step is checked against the oracle applied to the GPU's own 16-bit input of
that step (the oracle is fed what the kernel consumed), so that the rounding of
earlier steps does not accumulate into the tolerance; the whole layer is also
compared end to end at the same bound, on whole batches up to the
MTGR-large-like one."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import mtgr, synth
from hstu_attention_attn_b300.layer import HstuLayer, device_batch
from tests.gpu_common import bf16_round, dev, need_gpu, ragged_users
from tests.util import TOL_BF16, assert_close, assert_close_bf16, assert_close_f16, to_np

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def _layer_case(seed, D, H, dh, users):
    rng = np.random.default_rng(seed)
    return synth.layer_inputs(seed, lambda r: users, D, H, dh)


@pytest.mark.parametrize("D,H,dh", [(256, 2, 128), (512, 4, 128), (256, 4, 64)])
def test_layer_fwd_bf16_steps(orc, D, H, dh):
    need_gpu()
    L = _layer_case(31 + D + dh, D, H, dh, ragged_users())
    b = L.batch
    db = device_batch(b)
    layer = HstuLayer(D, H, dh, torch.from_numpy(L.w_uqkv), torch.from_numpy(L.w_o), torch.from_numpy(L.gamma),
                      torch.from_numpy(L.beta), dtype=BF)
    x = dev(L.x, BF)
    x_out, sv = layer.forward(x, db)
    torch.cuda.synchronize()
    HD = H * dh
    xb = bf16_round(L.x)
    wu, wo = bf16_round(L.w_uqkv), bf16_round(L.w_o)
    # GLN on the bf16 input (xn kept in f16)
    xn_ref, _, _ = orc.gln_fwd(xb, b.gid, L.gamma, L.beta)
    assert_close_f16(to_np(sv["xn"]), xn_ref, TOL_BF16, "xn")
    # projection on the GPU's xn
    xn = to_np(sv["xn"])
    z_ref = orc.matmul(xn, wu)
    # silu(z) and silu'(z) stored in f16, each one rounding of a function of the
    # fp32 accumulation of z.  Elementwise: half an ulp of f16 (2^-11) with a
    # factor-2 margin, plus the accumulation error of z (bounded generously by
    # 2e-4) times the slopes |silu'| <= 1.1 and |silu''| <= 0.5.
    s_ref, ds_ref = orc.silu(z_ref), orc.silu_grad(z_ref)
    sg, dsg = to_np(sv["uqkv"]), to_np(sv["dsilu"])
    assert np.all(np.abs(sg - s_ref) <= 2.0 ** -10 * np.abs(s_ref) + 2.2e-4), "silu(z)"
    assert np.all(np.abs(dsg - ds_ref) <= 2.0 ** -10 * np.abs(ds_ref) + 1e-4), "silu'(z)"
    assert_close_f16(dsg, ds_ref, TOL_BF16, "silu'(z)")
    assert_close_f16(sg, s_ref, TOL_BF16, "silu(z)")

    # attention on the GPU's uqkv
    a = to_np(sv["uqkv"])
    U, Q, K, V = (a[:, i * HD:(i + 1) * HD] for i in range(4))
    Y_ref, O_ref, _, _ = orc.attn_fwd(b, H, dh, Q, K, V, U)
    assert_close_f16(to_np(sv["o"]), O_ref, TOL_BF16, "o")
    assert_close_f16(to_np(sv["y"]), Y_ref, TOL_BF16, "y")
    # output projection + residual on the GPU's Y
    xo_ref = xb + orc.matmul(to_np(sv["y"]), wo)
    assert_close_bf16(to_np(x_out), xo_ref, TOL_BF16, "x_out")
    # end to end against the oracle layer on the bf16 inputs
    ref = orc.layer_fwd(b, D, H, dh, xb, wu, wo, L.gamma, L.beta)
    assert_close_bf16(to_np(x_out), ref["x_out"], TOL_BF16, "x_out end-to-end")


@pytest.mark.parametrize("D,H,dh", [(256, 2, 128), (256, 4, 64)])
def test_layer_bwd_bf16_steps(orc, D, H, dh):
    """Layer backward: the oracle's chain of steps fed with the GPU's saved
    forward state (the f16 xn, [U|Q|K|V], y and silu'(z)) and the bf16
    upstream gradient; then the whole backward end to end."""
    need_gpu()
    L = _layer_case(57 + D + dh, D, H, dh, ragged_users())
    b = L.batch
    db = device_batch(b)
    layer = HstuLayer(D, H, dh, torch.from_numpy(L.w_uqkv), torch.from_numpy(L.w_o), torch.from_numpy(L.gamma),
                      torch.from_numpy(L.beta), dtype=BF)
    x = dev(L.x, BF)
    _, sv = layer.forward(x, db)
    dx, g = layer.backward(x, sv, dev(L.dx_out, BF), db)
    torch.cuda.synchronize()
    # the layer lends its backward a store for the dS tiles (by default): dQ came from them
    assert mtgr.mtgr_debug_plan_counts(layer._ws, b.B)[3] == 1
    HD = H * dh
    xb, dxo = bf16_round(L.x), bf16_round(L.dx_out)
    wu, wo = bf16_round(L.w_uqkv), bf16_round(L.w_o)
    xn, a, y, ds = (to_np(sv[n]) for n in ("xn", "uqkv", "y", "dsilu"))
    # dW_o = yᵀ · dx_out (fp32-stored)
    assert_close(to_np(g["dw_o"]), orc.matmul_tn(y, dxo), TOL_BF16, "dw_o")
    # dY = dx_out · W_oᵀ; attention backward; dZ = [dU|dQ|dK|dV] ⊙ silu'(z)
    dY = orc.matmul_nt(dxo, wo)
    U, Q, K, V = (a[:, i * HD:(i + 1) * HD] for i in range(4))
    dq, dk, dv, du = orc.attn_bwd(b, H, dh, Q, K, V, U, dY)
    dZ = np.concatenate([du, dq, dk, dv], axis=1) * ds
    assert_close(to_np(g["dw_uqkv"]), orc.matmul_tn(xn, dZ), TOL_BF16, "dw_uqkv")
    # dxn = dZ · W_uqkvᵀ; GLN backward; plus the residual path
    rdx, rdg, rdb = orc.gln_bwd(orc.matmul_nt(dZ, wu), xb, b.gid, L.gamma)
    assert_close_bf16(to_np(dx), rdx + dxo, TOL_BF16, "dx")
    assert_close(to_np(g["dgamma"]), rdg, TOL_BF16, "dgamma")
    assert_close(to_np(g["dbeta"]), rdb, TOL_BF16, "dbeta")
    # end to end against the oracle layer backward on the bf16 inputs, at the same bound
    rb = orc.layer_bwd(b, D, H, dh, xb, wu, wo, L.gamma, L.beta, dxo)
    assert_close_bf16(to_np(dx), rb["dx"], TOL_BF16, "dx end-to-end")
    for n in ("dw_uqkv", "dw_o", "dgamma", "dbeta"):
        assert_close(to_np(g[n]), rb[n], TOL_BF16, n + " end-to-end")


def _check_layer_end_to_end(orc, L, rows=None, sub=None):
    """Run the layer forward + backward on the GPU over the whole batch of L;
    compare with the oracle end to end (whole batch, or the users of `sub`
    whose rows are `rows`) at the bf16-path bound."""
    b = L.batch
    db = device_batch(b)
    layer = HstuLayer(L.D, L.H, L.dh, torch.from_numpy(L.w_uqkv), torch.from_numpy(L.w_o),
                      torch.from_numpy(L.gamma), torch.from_numpy(L.beta), dtype=BF)
    x = dev(L.x, BF)
    x_out, sv = layer.forward(x, db)
    dx, g = layer.backward(x, sv, dev(L.dx_out, BF), db)
    torch.cuda.synchronize()
    got = {"x_out": to_np(x_out), "dx": to_np(dx), "xn": to_np(sv["xn"]), "o": to_np(sv["o"]),
           "y": to_np(sv["y"])}
    wu, wo = bf16_round(L.w_uqkv), bf16_round(L.w_o)
    if rows is None:
        xb, dxo, bb = bf16_round(L.x), bf16_round(L.dx_out), b
    else:
        xb, dxo, bb = bf16_round(L.x[rows]), bf16_round(L.dx_out[rows]), sub
        got = {k: v[rows] for k, v in got.items()}
    ref = orc.layer_fwd_blas(bb, L.D, L.H, L.dh, xb, wu, wo, L.gamma, L.beta)
    assert_close_f16(got["xn"], ref["xn"], TOL_BF16, "xn end-to-end")
    assert_close_f16(got["o"], ref["o"], TOL_BF16, "o end-to-end")
    assert_close_f16(got["y"], ref["y"], TOL_BF16, "y end-to-end")
    assert_close_bf16(got["x_out"], ref["x_out"], TOL_BF16, "x_out end-to-end")
    del ref
    rb = orc.layer_bwd_blas(bb, L.D, L.H, L.dh, xb, wu, wo, L.gamma, L.beta, dxo)
    assert_close_bf16(got["dx"], rb["dx"], TOL_BF16, "dx end-to-end")
    if rows is None:   # weight gradients sum over every user: whole batches only
        for n in ("dw_uqkv", "dw_o", "dgamma", "dbeta"):
            assert_close(to_np(g[n]), rb[n], TOL_BF16, n + " end-to-end")


def test_layer_fwd_bwd_large_batch_whole(orc):
    """One whole MTGR-large-like batch (128 users, about 63k tokens, d_model
    1024, 8 heads x 128, dense upstream gradient): forward and backward end to
    end against the oracle on every output and gradient, the weight gradients
    included (their split-K slices run only at this size)."""
    need_gpu()
    L = synth.large_layer(2)
    assert L.batch.B == 128 and L.D == 1024 and L.H == 8 and L.dh == 128
    _check_layer_end_to_end(orc, L)


def test_layer_training_step_full_size_sampled_users(orc):
    """The benchmark's own training step (262,171 tokens, d_model 1024, 8 heads
    x 128, upstream gradient on candidates only), run whole on the GPU; a user's
    x_out and dx rows depend on that user alone (given the weights), so sampled
    whole users are checked against the oracle run on them alone."""
    need_gpu()
    from tests.gpu_common import sub_batch
    L = synth.large_train_layer(3)
    b = L.batch
    n = np.diff(b.offsets)
    rt = np.array([c[2] for c in b.counts]) if b.counts else np.zeros(b.B)
    rng = np.random.default_rng(0)
    users = sorted({int(np.argmax(n)), int(np.argmin(n)), int(np.argmax(rt)), *rng.choice(b.B, 2, replace=False).tolist()})
    sb, rows = sub_batch(b, users)
    _check_layer_end_to_end(orc, L, rows, sb)
