"""bf16 tcgen05 attention vs the fp64 oracle (fed the same bf16-rounded inputs):
the 2e-2 bound on O (f16-stored), Y and every gradient (bf16-stored)."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import mtgr, synth
from hstu_attention_attn_b300.layer import HstuAttention, device_batch, workspace
from tests.gpu_common import bf16_round, dev, need_gpu, ragged_users, sub_batch
from tests.util import TOL_BF16, assert_close_bf16, assert_close_f16, to_np

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def _inputs(rng, batch, H, dh, scale=1.0, packed=False):
    T, HD = batch.T, H * dh
    if packed:   # q/k/v/u as column blocks of one [T, 4*HD] buffer, like the layer
        big = (rng.standard_normal((T, 4 * HD)) * scale).astype(np.float32)
        t = dev(big, BF)
        views = [t[:, i * HD:(i + 1) * HD] for i in (1, 2, 3, 0)]   # q, k, v, u
        host = [bf16_round(big[:, i * HD:(i + 1) * HD]) for i in (1, 2, 3, 0)]
        return views, host, 4 * HD
    mats = [(rng.standard_normal((T, HD)) * scale).astype(np.float32) for _ in range(4)]
    return [dev(m, BF) for m in mats], [bf16_round(m) for m in mats], HD


def _run_fwd(batch, H, dh, rng, scale=1.0, packed=False):
    db = device_batch(batch)
    (q, k, v, u), host, ld = _inputs(rng, batch, H, dh, scale, packed)
    op = HstuAttention(H, dh, BF)
    y, saved = op.forward(q, k, v, u, db, ld=ld)
    torch.cuda.synchronize()
    return op, db, (q, k, v, u), host, ld, y, saved


@pytest.mark.parametrize("dh", [128, 64])
@pytest.mark.parametrize("ts_hi", [86400, 40])
def test_attention_fwd_bf16_ragged(orc, dh, ts_hi):
    need_gpu()
    rng = np.random.default_rng(11 + dh + ts_hi)
    batch = synth.make_batch(rng, ragged_users(), ts_hi=ts_hi)
    H = 2
    _, _, _, host, _, y, saved = _run_fwd(batch, H, dh, rng)
    Y, O, mean, rstd = orc.attn_fwd(batch, H, dh, *host)
    assert_close_f16(to_np(saved[0]), O, TOL_BF16, "O")
    assert_close_bf16(to_np(y), Y, TOL_BF16, "Y")


def test_attention_fwd_bf16_ragged_paired_items(orc):
    """Enough ragged users (about 41k tokens) that the forward plans pairs of
    query tiles per item (short requests get one tile per item instead)."""
    need_gpu()
    rng = np.random.default_rng(31)
    batch = synth.make_batch(rng, ragged_users() * 24, ts_hi=3000)
    H, dh = 2, 128
    assert (batch.T // 128 + batch.B) * H > 4 * 148
    _, _, _, host, _, y, saved = _run_fwd(batch, H, dh, rng)
    Y, O, _, _ = orc.attn_fwd(batch, H, dh, *host)
    assert_close_f16(to_np(saved[0]), O, TOL_BF16, "O")
    assert_close_bf16(to_np(y), Y, TOL_BF16, "Y")


def test_attention_fwd_bf16_packed_layout(orc):
    need_gpu()
    rng = np.random.default_rng(21)
    batch = synth.make_batch(rng, ragged_users()[:4], ts_hi=500)
    H, dh = 4, 128
    _, _, _, host, _, y, saved = _run_fwd(batch, H, dh, rng, packed=True)
    Y, O, _, _ = orc.attn_fwd(batch, H, dh, *host)
    assert_close_f16(to_np(saved[0]), O, TOL_BF16, "O")
    assert_close_bf16(to_np(y), Y, TOL_BF16, "Y")


def test_attention_fwd_bf16_small_workload_sampled(orc):
    """The MTGR-small-like workload at full size (64 users, d_model 512, 4 heads x 128);
    the oracle recomputes a sample of whole users (users are independent)."""
    need_gpu()
    a = synth.small_attn(1)
    batch, H, dh = a.batch, a.H, a.dh
    db = device_batch(batch)
    q, k, v, u = (dev(m, BF) for m in (a.q, a.k, a.v, a.u))
    op = HstuAttention(H, dh, BF)
    y, saved = op.forward(q, k, v, u, db)
    torch.cuda.synchronize()
    lens = np.diff(batch.offsets)
    order = np.argsort(lens)
    pick = sorted(set([int(order[0]), int(order[len(order) // 2]), int(order[-1])] +
                      [int(i) for i in np.where(lens <= 1200)[0][:5]]))
    sb, rows = sub_batch(batch, pick)
    host = [bf16_round(m[rows]) for m in (a.q, a.k, a.v, a.u)]
    Y, O, _, _ = orc.attn_fwd(sb, H, dh, *host)
    assert_close_f16(to_np(saved[0])[rows], O, TOL_BF16, "O")
    assert_close_bf16(to_np(y)[rows], Y, TOL_BF16, "Y")


@pytest.mark.parametrize("dh", [128, 64])
@pytest.mark.parametrize("ts_hi", [86400, 40])
def test_attention_bwd_bf16_ragged(orc, dh, ts_hi):
    need_gpu()
    rng = np.random.default_rng(51 + dh + ts_hi)
    batch = synth.make_batch(rng, ragged_users(), ts_hi=ts_hi)
    H = 2
    op, db, (q, k, v, u), host, ld, y, saved = _run_fwd(batch, H, dh, rng)
    dY = rng.standard_normal(tuple(y.shape)).astype(np.float32)
    dq, dk, dv, du = op.backward(dev(dY, BF), q, k, v, u, saved, db, ld=ld)
    torch.cuda.synchronize()
    assert op.device_status() == 0
    ref = orc.attn_bwd(batch, H, dh, *host, bf16_round(dY))
    for name, got, r in zip(("dq", "dk", "dv", "du"), (dq, dk, dv, du), ref):
        assert_close_bf16(to_np(got), r, TOL_BF16, name)


@pytest.mark.parametrize("dh", [128, 64])
def test_attention_bwd_bf16_many_items_per_cta(orc, dh):
    """About 41k ragged tokens: several query-tile and key-tile items per CTA,
    so the TMEM accumulators, the score buffers and the Q/dO stage are reused
    across items (one dQ accumulator per CTA for d_h = 128, two for d_h = 64)."""
    need_gpu()
    rng = np.random.default_rng(71 + dh)
    batch = synth.make_batch(rng, ragged_users() * 24, ts_hi=3000)
    H = 2
    assert sum((int(n) + 127) // 128 for n in np.diff(batch.offsets)) * H > 2 * 148
    op, db, (q, k, v, u), host, ld, y, saved = _run_fwd(batch, H, dh, rng)
    dY = rng.standard_normal(tuple(y.shape)).astype(np.float32)
    dq, dk, dv, du = op.backward(dev(dY, BF), q, k, v, u, saved, db, ld=ld)
    torch.cuda.synchronize()
    assert op.device_status() == 0
    ref = orc.attn_bwd(batch, H, dh, *host, bf16_round(dY))
    for name, got, r in zip(("dq", "dk", "dv", "du"), (dq, dk, dv, du), ref):
        assert_close_bf16(to_np(got), r, TOL_BF16, name)


def test_attention_bwd_bf16_small_workload_sampled(orc):
    """Backward at the MTGR-small-like size; sampled whole users recomputed by the oracle."""
    need_gpu()
    a = synth.small_attn(1)
    batch, H, dh = a.batch, a.H, a.dh
    db = device_batch(batch)
    q, k, v, u = (dev(m, BF) for m in (a.q, a.k, a.v, a.u))
    op = HstuAttention(H, dh, BF)
    y, saved = op.forward(q, k, v, u, db)
    rng = np.random.default_rng(5)
    dY = rng.standard_normal(tuple(y.shape)).astype(np.float32)
    dq, dk, dv, du = op.backward(dev(dY, BF), q, k, v, u, saved, db)
    torch.cuda.synchronize()
    assert op.device_status() == 0
    lens = np.diff(batch.offsets)
    pick = sorted(set([int(np.argmin(lens)), int(np.argsort(lens)[len(lens) // 2])] +
                      [int(i) for i in np.where(lens <= 1000)[0][:4]]))
    sb, rows = sub_batch(batch, pick)
    host = [bf16_round(m[rows]) for m in (a.q, a.k, a.v, a.u)]
    ref = orc.attn_bwd(sb, H, dh, *host, bf16_round(dY[rows]))
    for name, got, r in zip(("dq", "dk", "dv", "du"), (dq, dk, dv, du), ref):
        assert_close_bf16(to_np(got)[rows], r, TOL_BF16, name)


def test_attention_bf16_longest_user(orc):
    """One 4,112-token user (33 tiles: its tile cost passes the planner's
    1023-bucket clamp, and each of its items streams up to 33 K/V tiles
    through the ring) beside the ragged users; forward and backward against
    the oracle on every user."""
    need_gpu()
    rng = np.random.default_rng(61)
    batch = synth.make_batch(rng, [(8, 4020, 64, 20)] + ragged_users(), ts_hi=86400)
    H, dh = 1, 128
    assert int(np.diff(batch.offsets).max()) == 4112
    op, db, (q, k, v, u), host, ld, y, saved = _run_fwd(batch, H, dh, rng)
    Y, O, _, _ = orc.attn_fwd(batch, H, dh, *host)
    assert_close_f16(to_np(saved[0]), O, TOL_BF16, "O")
    assert_close_bf16(to_np(y), Y, TOL_BF16, "Y")
    dY = rng.standard_normal(tuple(y.shape)).astype(np.float32)
    dq, dk, dv, du = op.backward(dev(dY, BF), q, k, v, u, saved, db, ld=ld)
    torch.cuda.synchronize()
    assert op.device_status() == 0
    ref = orc.attn_bwd(batch, H, dh, *host, bf16_round(dY))
    for name, got, r in zip(("dq", "dk", "dv", "du"), (dq, dk, dv, du), ref):
        assert_close_bf16(to_np(got), r, TOL_BF16, name)


@pytest.mark.parametrize("dh", [128, 64])
def test_attention_bwd_bf16_ds_store_and_recompute(orc, dh):
    """The two dQ passes of the backward: with a store for the dS tiles (the
    dK/dV pass keeps them and dQ = dS K reads them back), without one, and
    with a store too small for the batch (the plan falls back to recomputing
    S and dP on the device).  Each against the oracle; the plan's flag says
    which pass ran."""
    need_gpu()
    rng = np.random.default_rng(81 + dh)
    batch = synth.make_batch(rng, ragged_users() * 6, ts_hi=3000)
    H = 2
    op, db, (q, k, v, u), host, ld, y, saved = _run_fwd(batch, H, dh, rng)
    dY = rng.standard_normal(tuple(y.shape)).astype(np.float32)
    ref = orc.attn_bwd(batch, H, dh, *host, bf16_round(dY))
    need = mtgr.mtgr_attn_ds_store_size(batch.offsets, H, dh, mtgr.MTGR_BF16)
    tiles = sum(((int(n) + 127) // 128) ** 2 for n in np.diff(batch.offsets))
    assert need == H * tiles * 128 * 128 * 2 + 1024
    base = mtgr.mtgr_attn_workspace_size(batch.B, batch.T, H, dh, mtgr.MTGR_BF16)
    runs = {}
    for name, extra, kept in (("store", need, 1), ("none", 0, 0), ("short", need // 2, 0)):
        run = HstuAttention(H, dh, BF, ds_store=False)
        run._ws = workspace(base + extra)
        dq, dk, dv, du = run.backward(dev(dY, BF), q, k, v, u, saved, db, ld=ld)
        torch.cuda.synchronize()
        assert run.device_status() == 0
        assert mtgr.mtgr_debug_plan_counts(run._ws, batch.B)[3] == kept, name
        for gname, got, r in zip(("dq", "dk", "dv", "du"), (dq, dk, dv, du), ref):
            assert_close_bf16(to_np(got), r, TOL_BF16, f"{gname} ({name})")
        runs[name] = [to_np(t) for t in (dq, dk, dv, du)]
    for i, gname in enumerate(("dq", "dk", "dv", "du")):  # recorded: both passes already meet the oracle bound
        a, b = runs["store"][i].astype(np.float64), runs["none"][i].astype(np.float64)
        print(f"{gname}: stored vs recomputed dS, max |diff| / RMS = "
              f"{np.abs(a - b).max() / (np.sqrt(np.mean(b ** 2)) + 1e-30):.2e}")
