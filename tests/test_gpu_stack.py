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
