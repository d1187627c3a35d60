"""bf16 HSTU layer (tcgen05 GEMMs + attention) vs the fp64 oracle.

Each step is checked against the oracle applied to the GPU's own bf16 input of
that step (the oracle is fed what the kernel consumed), so that bf16 rounding of
earlier steps does not accumulate into the tolerance; the whole layer output is
also compared end to end."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import synth
from hstu_attention_attn_b300.layer import HstuLayer, device_batch
from tests.gpu_common import bf16_round, dev, need_gpu, ragged_users
from tests.util import TOL_BF16, assert_close, assert_close_bf16, to_np

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
    # GLN on the bf16 input
    xn_ref, _, _ = orc.gln_fwd(xb, b.gid, L.gamma, L.beta)
    assert_close_bf16(to_np(sv["xn"]), xn_ref, TOL_BF16, "xn")
    # projection on the GPU's xn
    xn = to_np(sv["xn"])
    z_ref = orc.matmul(xn, wu)
    assert_close_bf16(to_np(sv["z"]), z_ref, TOL_BF16, "z")
    # silu of the stored z, rounded once to bf16: elementwise relative check
    sz = orc.silu(to_np(sv["z"]))
    assert np.all(np.abs(to_np(sv["uqkv"]) - sz) <= 2.0 ** -8 * np.abs(sz) + 1e-6), "silu(z)"

    # attention on the GPU's uqkv
    a = to_np(sv["uqkv"])
    U, Q, K, V = (a[:, i * HD:(i + 1) * HD] for i in range(4))
    Y_ref, O_ref, _, _ = orc.attn_fwd(b, H, dh, Q, K, V, U)
    assert_close_bf16(to_np(sv["o"]), O_ref, TOL_BF16, "o")
    assert_close_bf16(to_np(sv["y"]), Y_ref, TOL_BF16, "y")
    # output projection + residual on the GPU's Y
    xo_ref = xb + orc.matmul(to_np(sv["y"]), wo)
    assert_close_bf16(to_np(x_out), xo_ref, TOL_BF16, "x_out")
    # end to end against the oracle layer on the bf16 inputs
    ref = orc.layer_fwd(b, D, H, dh, xb, wu, wo, L.gamma, L.beta)
    assert_close_bf16(to_np(x_out), ref["x_out"], TOL_BF16, "x_out end-to-end")
