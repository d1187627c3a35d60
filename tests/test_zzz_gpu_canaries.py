"""Canary pads (tests/canary.py) around every buffer a bf16 layer step hands
to the library: input, output, saved state, workspace, upstream gradient,
input gradient and weight gradients.  After the forward and the backward on
ragged users (tails of every tile size, empty and one-token users) no pad may
have changed, and the results must match a run on plain allocations."""
import pytest
import torch

from hstu_attention_attn_b300 import mtgr, synth
from hstu_attention_attn_b300.layer import HstuLayer, device_batch
from tests.canary import Canaries
from tests.gpu_common import dev, need_gpu, ragged_users

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def _layer(L, D, H, dh):
    return HstuLayer(D, H, dh, *(torch.from_numpy(a) for a in (L.w_uqkv, L.w_o, L.gamma, L.beta)), dtype=BF)


@pytest.mark.parametrize("D,H,dh", [(256, 2, 128), (256, 4, 64)])
def test_layer_step_writes_stay_inside_their_buffers(D, H, dh):
    need_gpu()
    L = synth.layer_inputs(71 + D + dh, lambda r: ragged_users(), D, H, dh)
    db = device_batch(L.batch)
    T, HD = L.batch.T, H * dh
    c = Canaries("cuda")
    layer = _layer(L, D, H, dh)
    layer._ws = c.tensor((mtgr.mtgr_layer_workspace_size(db.B, db.T, D, H, dh, mtgr.MTGR_BF16),), torch.uint8)
    x = c.tensor((T, D), BF)
    x.copy_(dev(L.x, BF))
    saved = {n: c.like(t) for n, t in layer.alloc_saved(T).items()}
    x_out = c.tensor((T, D), BF)
    layer.forward(x, db, saved, x_out)
    dxo = c.tensor((T, D), BF)
    dxo.copy_(dev(L.dx_out, BF))
    dx = c.tensor((T, D), BF)
    grads = {n: c.tensor(s, torch.float32)
             for n, s in (("dw_uqkv", (D, 4 * HD)), ("dw_o", (HD, D)), ("dgamma", (4, D)), ("dbeta", (4, D)))}
    layer.backward(x, saved, dxo, db, dx, grads)
    torch.cuda.synchronize()
    assert c.broken() == [], "a write landed outside its buffer"
    ref = _layer(L, D, H, dh)
    x_ref = dev(L.x, BF)
    xo_ref, sv_ref = ref.forward(x_ref, db)
    dx_ref, g_ref = ref.backward(x_ref, sv_ref, dev(L.dx_out, BF), db)
    torch.cuda.synchronize()
    torch.testing.assert_close(x_out.float(), xo_ref.float(), rtol=1e-2, atol=1e-2)
    torch.testing.assert_close(dx.float(), dx_ref.float(), rtol=1e-2, atol=1e-2)
    for n, g in grads.items():
        torch.testing.assert_close(g, g_ref[n], rtol=1e-3, atol=1e-3 * float(g_ref[n].abs().max()))
