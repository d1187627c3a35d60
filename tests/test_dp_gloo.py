"""Data-parallel training step on CPU with two gloo ranks.

Each rank takes its token-balanced share of a step's users, computes the layer's
weight gradients of the mean loss over its own users (the fp64 oracle stands in
for the rank's GPU), and joins the weighted all-reduce; the result must be the
gradient of the mean loss over all users of the step, computed in one process.
The users are independent and every weight gradient is a sum over tokens, so
the two agree up to fp64 rounding."""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _case():
    from hstu_attention_attn_b300 import synth
    return synth.layer_inputs(5, lambda r: synth.tiny_users(r, 7), 64, 2, 32)


def _worker(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import oracle as orc
        from hstu_attention_attn_b300 import dp, synth
        L = _case()
        b = L.batch
        first, rank_tokens, weight = dp.rank_users(np.diff(b.offsets), WORLD)
        u0, u1 = int(first[rank]), int(first[rank + 1])
        r0, r1, off = dp.user_rows(b.offsets, u0, u1)
        local = synth.Batch(off, b.gid[r0:r1], b.ts[r0:r1])
        n_users = u1 - u0
        g = orc.layer_bwd(local, L.D, L.H, L.dh, L.x[r0:r1], L.w_uqkv, L.w_o, L.gamma, L.beta,
                          L.dx_out[r0:r1].astype(np.float64) / n_users)   # mean over this rank's users
        grads = {k: torch.from_numpy(np.ascontiguousarray(g[k])) for k in ("dw_uqkv", "dw_o", "dgamma", "dbeta")}
        dp.allreduce_weighted(grads, float(weight[rank]))
        if rank == 0:
            np.savez(os.path.join(out_dir, "dp.npz"), **{k: v.numpy() for k, v in grads.items()},
                     tokens=rank_tokens, first=first)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_data_parallel_step_equals_single_process():
    import oracle as orc
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(_free_port(), d), nprocs=WORLD, join=True)
        got = dict(np.load(os.path.join(d, "dp.npz")))
    L = _case()
    ref = orc.layer_bwd(L.batch, L.D, L.H, L.dh, L.x, L.w_uqkv, L.w_o, L.gamma, L.beta,
                        L.dx_out.astype(np.float64) / L.batch.B)
    for k in ("dw_uqkv", "dw_o", "dgamma", "dbeta"):
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-10, atol=1e-12 * np.abs(ref[k]).max())
    # both ranks got users, and every user exactly one rank
    assert got["first"][0] == 0 and got["first"][-1] == L.batch.B and np.all(np.diff(got["first"]) > 0)
    assert got["tokens"].sum() == L.batch.T
