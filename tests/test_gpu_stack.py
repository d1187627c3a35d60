"""Layer stack for ranking: eager forward vs the replay of one captured CUDA
Graph (bit-exact: every forward kernel writes each output element from one
place in a fixed order), and every layer against the fp64 oracle fed that
layer's own GPU input (parity per layer; the stack's end-to-end drift is not a
parity claim)."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import synth
from hstu_attention_attn_b300.layer import HstuLayer, HstuStack, device_batch
from tests.gpu_common import bf16_round, dev, need_gpu
from tests.util import TOL_BF16, assert_close_bf16, to_np

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def _stack(D, H, dh, n_layers, users, seed):
    base = synth.layer_inputs(seed, lambda r: users, D, H, dh)
    ws = [synth.layer_inputs(seed + 100 + l, lambda r: users[:1], D, H, dh) for l in range(n_layers)]
    layers = [HstuLayer(D, H, dh, torch.from_numpy(w.w_uqkv), torch.from_numpy(w.w_o), torch.from_numpy(w.gamma),
                        torch.from_numpy(w.beta), dtype=BF) for w in ws]
    return base, ws, HstuStack(layers)


# a ranking-like user (history + RealTime + candidates), a multi-tile user, a short one
USERS = [(8, 300, 40, 12), (4, 117, 10, 3), (8, 600, 20, 30), (1, 5, 0, 1)]


def test_stack_graph_replay_equals_eager(orc):
    need_gpu()
    D, H, dh, n_layers = 256, 2, 128, 3
    base, ws, stack = _stack(D, H, dh, n_layers, USERS, 71)
    db = device_batch(base.batch)
    x = dev(base.x, BF)
    outs = []
    y_eager = stack.forward(x, db, outs=outs).clone()          # layer by layer
    y_native = HstuStack(stack.layers).forward(x, db).clone()  # one library call, one work-list build
    assert torch.equal(y_native, y_eager)
    stack.capture(x, db)
    torch.cuda.synchronize()
    assert torch.equal(stack.replay().clone(), y_eager)
    # a new request through the same graph: refill the static input, replay
    x2 = dev(np.random.default_rng(5).standard_normal(base.x.shape).astype(np.float32), BF)
    y2_eager = HstuStack(stack.layers).forward(x2, db).clone()
    x.copy_(x2)
    y2_graph = stack.replay().clone()
    torch.cuda.synchronize()
    assert torch.equal(y2_graph, y2_eager)
    assert not torch.equal(y2_eager, y_eager)

    # every layer against the oracle on that layer's GPU input
    inp = bf16_round(base.x)
    for l in range(n_layers):
        w = ws[l]
        ref = orc.layer_fwd(base.batch, D, H, dh, inp, bf16_round(w.w_uqkv), bf16_round(w.w_o), w.gamma, w.beta)
        got = to_np(outs[l])
        assert_close_bf16(got, ref["x_out"], TOL_BF16, f"layer {l}")
        inp = got


def test_kept_f16_weights_give_identical_results():
    """A bf16 layer reading f16 copies of its weights made once
    (mtgr_layer_weights_to_f16) returns what it returns when every call
    converts them (bit for bit, except the order of the dγ/dβ atomics);
    setting only one copy is refused."""
    need_gpu()
    from hstu_attention_attn_b300 import mtgr
    D, H, dh = 256, 2, 128
    base, ws, stack = _stack(D, H, dh, 1, USERS, 81)
    layer = stack.layers[0]
    db = device_batch(base.batch)
    x = dev(base.x, BF)
    dxo = dev(np.random.default_rng(3).standard_normal(base.x.shape).astype(np.float32), BF)
    layer.drop_f16_weights()
    y0, sv0 = layer.forward(x, db)
    y0 = y0.clone()
    dx0, g0 = layer.backward(x, sv0, dxo, db)
    dx0, g0 = dx0.clone(), {k: v.clone() for k, v in g0.items()}
    layer.keep_f16_weights()
    y1, sv1 = layer.forward(x, db)
    dx1, g1 = layer.backward(x, sv1, dxo, db)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(dx0, dx1)
    for k in ("dw_uqkv", "dw_o"):
        assert torch.equal(g0[k], g1[k]), k
    # dγ and dβ are summed through shared-memory atomics, whose order varies
    for k in ("dgamma", "dbeta"):
        assert torch.allclose(g0[k], g1[k], rtol=1e-5, atol=1e-5), k
    w16 = layer._w16
    assert torch.equal(w16[0], layer.w_uqkv.to(torch.float16)) and torch.equal(w16[1], layer.w_o.to(torch.float16))
    layer.weights.w_o_f16 = None
    with pytest.raises(mtgr.MtgrError, match="both f16 weight copies"):
        layer.forward(x, db)
    layer.drop_f16_weights()
