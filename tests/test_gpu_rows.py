"""Row expansion of a sparse upstream gradient (mtgr_expand_rows): exact
against zeros plus indexed assignment; rows outside [0, T) are skipped."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import mtgr
from tests.gpu_common import need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_expand_rows_exact(dt):
    need_gpu()
    rng = np.random.default_rng(3)
    T, D, n = 1000, 64, 37
    rows = rng.choice(T, n, replace=False).astype(np.int32)
    src = torch.from_numpy(rng.standard_normal((n, D)).astype(np.float32)).to("cuda", dt)
    r = torch.from_numpy(rows).cuda()
    dst = torch.full((T, D), 7.0, device="cuda", dtype=dt)          # stale contents must vanish
    mtgr.mtgr_expand_rows(src, r, dst)
    ref = torch.zeros_like(dst)
    ref[r.long()] = src
    torch.cuda.synchronize()
    assert torch.equal(dst, ref)
    # out-of-range rows are skipped, the valid ones still land
    bad = torch.tensor([-1, 5, T, 9], dtype=torch.int32, device="cuda")
    src4 = torch.ones(4, D, device="cuda", dtype=dt)
    mtgr.mtgr_expand_rows(src4, bad, dst)
    torch.cuda.synchronize()
    assert dst[5].eq(1).all() and dst[9].eq(1).all() and dst.sum().item() == 2 * D
