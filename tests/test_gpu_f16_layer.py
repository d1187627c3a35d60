"""f16 inference variant of the layer forward (MTGR_F16) vs the fp64 oracle,
step by step on the GPU's own f16 input of each step, then end to end, at the
2e-2 bound on the error beyond one f16 rounding (2^-11) of every stored result."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import synth
from hstu_attention_attn_b300.layer import HstuLayer, HstuStack, device_batch
from tests.gpu_common import dev, f16_round, need_gpu, ragged_users
from tests.util import TOL_BF16, assert_close_f16, to_np

pytestmark = pytest.mark.gpu
F16 = torch.float16


@pytest.mark.parametrize("D,H,dh", [(256, 2, 128), (256, 4, 64)])
def test_layer_fwd_f16_steps(orc, D, H, dh):
    need_gpu()
    L = synth.layer_inputs(41 + D + dh, lambda r: ragged_users(), D, H, dh)
    b = L.batch
    db = device_batch(b)
    layer = HstuLayer(D, H, dh, torch.from_numpy(L.w_uqkv), torch.from_numpy(L.w_o), torch.from_numpy(L.gamma),
                      torch.from_numpy(L.beta), dtype=F16)
    x = dev(L.x, F16)
    x_out, sv = layer.forward(x, db)
    torch.cuda.synchronize()
    HD = H * dh
    xh, wu, wo = f16_round(L.x), f16_round(L.w_uqkv), f16_round(L.w_o)
    xn_ref, _, _ = orc.gln_fwd(xh, b.gid, L.gamma, L.beta)
    assert_close_f16(to_np(sv["xn"]), xn_ref, TOL_BF16, "xn")
    z_ref = orc.matmul(to_np(sv["xn"]), wu)
    s_ref, ds_ref = orc.silu(z_ref), orc.silu_grad(z_ref)
    assert np.all(np.abs(to_np(sv["uqkv"]) - s_ref) <= 2.0 ** -10 * np.abs(s_ref) + 2.2e-4), "silu(z)"
    assert np.all(np.abs(to_np(sv["dsilu"]) - ds_ref) <= 2.0 ** -10 * np.abs(ds_ref) + 1e-4), "silu'(z)"
    a = to_np(sv["uqkv"])
    U, Q, K, V = (a[:, i * HD:(i + 1) * HD] for i in range(4))
    Y_ref, O_ref, _, _ = orc.attn_fwd(b, H, dh, Q, K, V, U)
    assert_close_f16(to_np(sv["o"]), O_ref, TOL_BF16, "o")
    assert_close_f16(to_np(sv["y"]), Y_ref, TOL_BF16, "y")
    assert_close_f16(to_np(x_out), xh + orc.matmul(to_np(sv["y"]), wo), TOL_BF16, "x_out")
    ref = orc.layer_fwd(b, D, H, dh, xh, wu, wo, L.gamma, L.beta)
    assert_close_f16(to_np(x_out), ref["x_out"], TOL_BF16, "x_out end-to-end")


def test_stack_f16_graph_equals_eager_and_backward_is_refused():
    need_gpu()
    from hstu_attention_attn_b300 import mtgr
    D, H, dh = 256, 2, 128
    L = synth.layer_inputs(7, lambda r: ragged_users()[:5], D, H, dh)
    layers = [HstuLayer(D, H, dh, torch.from_numpy(L.w_uqkv), torch.from_numpy(L.w_o), torch.from_numpy(L.gamma),
                        torch.from_numpy(L.beta), dtype=F16) for _ in range(3)]
    db = device_batch(L.batch)
    x = dev(L.x, F16)
    stack = HstuStack(layers)
    y_eager = stack.forward(x, db, native=False).clone()
    assert torch.equal(stack.forward(x, db).clone(), y_eager)
    stack.capture(x, db)
    assert torch.equal(stack.replay().clone(), y_eager)
    with pytest.raises(mtgr.MtgrError, match="forward"):
        _, sv = layers[0].forward(x, db)
        layers[0].backward(x, sv, x, db)
