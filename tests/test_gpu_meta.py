"""Integer metadata on the GPU: bit-exact visible-pair counts and validation."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import mtgr, synth
from hstu_attention_attn_b300.layer import device_batch
from tests.gpu_common import need_gpu, ragged_users

pytestmark = pytest.mark.gpu


def _counts(batch):
    db = device_batch(batch)
    cnt = torch.zeros(max(db.T, 1), dtype=torch.int32, device="cuda")
    tot = torch.zeros(1, dtype=torch.int64, device="cuda")
    mtgr.mtgr_debug_visible_counts(db.offsets, db.gid, db.ts, db.T, cnt, tot)
    torch.cuda.synchronize()
    return cnt[: db.T].cpu().numpy(), int(tot.item())


@pytest.mark.parametrize("case", ["tiny", "tiny_ties", "ragged", "small"])
def test_visible_counts_bit_exact(orc, case):
    need_gpu()
    rng = np.random.default_rng(7)
    if case == "tiny":
        batch = synth.tiny_attn(0).batch
    elif case == "tiny_ties":
        batch = synth.tiny_attn(1, ts_hi=16).batch
    elif case == "ragged":
        batch = synth.make_batch(rng, ragged_users(), ts_hi=300)
    else:
        batch = synth.make_batch(rng, synth.small_users(rng))
    cnt, tot = _counts(batch)
    ref_cnt, ref_tot = orc.visible_counts(batch)
    assert np.array_equal(cnt, ref_cnt)
    assert tot == ref_tot


def test_validate_batch_flags():
    need_gpu()
    rng = np.random.default_rng(3)
    good = synth.make_batch(rng, ragged_users())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(offsets, gid, T):
        o = torch.tensor(offsets, dtype=torch.int32, device="cuda")
        g = torch.tensor(gid, dtype=torch.uint8, device="cuda")
        mtgr.mtgr_validate_batch(o, g, T, st)
        torch.cuda.synchronize()
        return int(st.item())

    assert run(good.offsets, good.gid, good.T) == 0
    bad_order = good.gid.copy()
    s0 = int(good.offsets[1])
    bad_order[s0 + 2], bad_order[s0 + 100] = 3, 1       # a candidate before Seq tokens
    assert run(good.offsets, bad_order, good.T) & mtgr.STATUS_BAD_GROUP_ORDER
    bad_id = good.gid.copy()
    bad_id[5] = 7
    assert run(good.offsets, bad_id, good.T) & mtgr.STATUS_BAD_GROUP_ID
    offs = good.offsets.copy()
    offs[3] = offs[2] - 1                                # decreasing offsets
    assert run(offs, good.gid, good.T) & mtgr.STATUS_BAD_OFFSETS
    offs = good.offsets.copy()
    offs[-1] = good.T - 1                                # offsets[B] != T
    assert run(offs, good.gid, good.T) & mtgr.STATUS_BAD_OFFSETS
