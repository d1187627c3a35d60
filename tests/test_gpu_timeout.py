"""The bounded-wait path on the GPU.  A CTA whose mbarrier never completes
gives up after the library's wait limit (2 s), reports MTGR_STATUS_TIMEOUT in
the status word and frees its tensor memory; the tcgen05 kernels launched next
on the same context run and stay within tolerance.  Nothing faults or hangs:
the wait is bounded by construction."""
import time

import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import mtgr, synth
from hstu_attention_attn_b300.layer import HstuAttention, device_batch
from tests.gpu_common import bf16_round, dev, need_gpu, ragged_users
from tests.util import TOL_BF16, assert_close_bf16, assert_close_f16, to_np

pytestmark = pytest.mark.gpu


def test_wait_timeout_reported_and_context_usable(orc):
    need_gpu()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mtgr.mtgr_debug_wait_timeout(st)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(st.item()) == mtgr.STATUS_TIMEOUT
    assert 1.9 < elapsed < 60.0
    # the same context, next: the bf16 attention forward on ragged users
    rng = np.random.default_rng(5)
    batch = synth.make_batch(rng, ragged_users(), ts_hi=500)
    H, dh = 2, 128
    mats = [rng.standard_normal((batch.T, H * dh)).astype(np.float32) for _ in range(4)]
    q, k, v, u = (dev(m, torch.bfloat16) for m in mats)
    y, saved = HstuAttention(H, dh, torch.bfloat16).forward(q, k, v, u, device_batch(batch))
    torch.cuda.synchronize()
    Y, O, _, _ = orc.attn_fwd(batch, H, dh, *(bf16_round(m) for m in mats))
    assert_close_f16(to_np(saved[0]), O, TOL_BF16, "O")
    assert_close_bf16(to_np(y), Y, TOL_BF16, "Y")
