"""GPU test of mtgr_group_layernorm_bwd_noalloc, the Group LayerNorm backward
for callers that cannot allocate device memory (their allocator owns every
byte, or the step must not allocate), so cannot pass a workspace.

It is called through the C ABI twice in a row, on two different batches, and
each result is compared with the workspace entry point mtgr_group_layernorm_bwd
on the same inputs.  The second batch is smaller than the first, so the second
call runs on a fixed device array that still holds the first call's partial
sums: it must not read them.  The file name sorts after the parity tests so
that a run stopping at the first failure has already run them."""
import numpy as np
import pytest
import torch

from tests.gpu_common import dev, need_gpu
from tests.util import TOL_F32, assert_close, to_np

pytestmark = pytest.mark.gpu


def _inputs(seed, T, D, dtype):
    rng = np.random.default_rng(seed)
    x = dev(rng.standard_normal((T, D)), dtype)
    dy = dev(rng.standard_normal((T, D)), dtype)
    dres = dev(rng.standard_normal((T, D)), dtype)
    gid = torch.from_numpy(rng.integers(0, 4, T).astype(np.uint8)).cuda()
    gamma = dev(1.0 + 0.1 * rng.standard_normal((4, D)), torch.float32)
    beta = dev(0.1 * rng.standard_normal((4, D)), torch.float32)
    return x, dy, dres, gid, gamma, beta


def _forward_stats(x, gid, gamma, beta):
    from hstu_attention_attn_b300 import mtgr
    T = x.shape[0]
    y = torch.empty_like(x)
    mean = torch.empty(T, dtype=torch.float32, device="cuda")
    rstd = torch.empty(T, dtype=torch.float32, device="cuda")
    mtgr.mtgr_group_layernorm_fwd(x, y, mean, rstd, gid, gamma, beta)
    return mean, rstd


def _both(x, dy, dres, gid, gamma, beta):
    from hstu_attention_attn_b300 import mtgr
    T, D = x.shape
    mean, rstd = _forward_stats(x, gid, gamma, beta)
    out = {}
    for name in ("workspace", "noalloc"):
        dx = torch.full_like(x, float("nan"))
        dg = torch.full((4, D), float("nan"), dtype=torch.float32, device="cuda")
        db = torch.full((4, D), float("nan"), dtype=torch.float32, device="cuda")
        if name == "workspace":
            ws = torch.empty(mtgr.mtgr_group_layernorm_bwd_workspace_size(T, D), dtype=torch.uint8, device="cuda")
            mtgr.mtgr_group_layernorm_bwd(dy, x, mean, rstd, gid, gamma, dres, dx, dg, db, ws)
        else:
            mtgr.mtgr_group_layernorm_bwd_noalloc(dy, x, mean, rstd, gid, gamma, dres, dx, dg, db)
        torch.cuda.synchronize()
        out[name] = {"dx": to_np(dx), "dgamma": to_np(dg), "dbeta": to_np(db)}
    return out


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 1024), (torch.float32, 64)])
def test_noalloc_matches_workspace_entry_point_twice(dtype, D):
    need_gpu()
    # first call: many rows (the scratch is filled by as many blocks as fit);
    # second call: few rows and other values (fewer blocks, stale scratch beyond them)
    for seed, T in ((11, 6000), (12, 300)):
        r = _both(*_inputs(seed, T, D, dtype))
        for k in ("dx", "dgamma", "dbeta"):
            assert_close(r["noalloc"][k], r["workspace"][k], TOL_F32, f"noalloc {k} (T={T}, D={D})")


def test_noalloc_rejects_oversized_rows():
    need_gpu()
    from hstu_attention_attn_b300 import mtgr
    L = mtgr.lib()
    r = L.mtgr_group_layernorm_bwd_noalloc(16, 16, 16, 16, 16, 16, None, 16, 16, 16, 10, 8192, mtgr.MTGR_BF16,
                                           None)
    assert r == -4 and "maximum of 4096" in mtgr.mtgr_last_error()
