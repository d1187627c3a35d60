"""GPU test of mtgr_group_layernorm_bwd_noalloc, the Group LayerNorm backward
for callers that cannot allocate device memory (their allocator owns every
byte, or the step must not allocate), so cannot pass a workspace.

It is called through the C ABI twice in a row, on two different batches, and
each result is compared with the workspace entry point mtgr_group_layernorm_bwd
on the same inputs and with the fp64 oracle.  The second batch is smaller than
the first, so the second call runs on a fixed device array that still holds the
first call's partial sums: it must not read them.  D = 4096 runs with fewer
blocks than the workspace entry point (the array's cap), D <= 1024 with the
same grid.  The file name sorts after the parity tests so that a run stopping
at the first failure has already run them."""
import numpy as np
import pytest
import torch

from tests.gpu_common import bf16_round, dev, need_gpu
from tests.util import TOL_BF16, TOL_F32, assert_close, assert_close_bf16, to_np

pytestmark = pytest.mark.gpu


def _inputs(seed, T, D, dtype):
    rng = np.random.default_rng(seed)
    h = {n: rng.standard_normal((T, D)).astype(np.float32) for n in ("x", "dy", "dres")}
    gid = rng.integers(0, 4, T).astype(np.uint8)
    gamma = (1.0 + 0.1 * rng.standard_normal((4, D))).astype(np.float32)
    beta = (0.1 * rng.standard_normal((4, D))).astype(np.float32)
    d = dict(x=dev(h["x"], dtype), dy=dev(h["dy"], dtype), dres=dev(h["dres"], dtype),
             gid=torch.from_numpy(gid).cuda(), gamma=dev(gamma, torch.float32), beta=dev(beta, torch.float32))
    rnd = bf16_round if dtype == torch.bfloat16 else (lambda a: np.asarray(a, np.float64))
    host = dict(x=rnd(h["x"]), dy=rnd(h["dy"]), dres=rnd(h["dres"]), gid=gid, gamma=gamma)
    return d, host


def _run(d, name):
    from hstu_attention_attn_b300 import mtgr
    x = d["x"]
    T, D = x.shape
    y = torch.empty_like(x)
    mean = torch.empty(T, dtype=torch.float32, device="cuda")
    rstd = torch.empty(T, dtype=torch.float32, device="cuda")
    mtgr.mtgr_group_layernorm_fwd(x, y, mean, rstd, d["gid"], d["gamma"], d["beta"])
    dx = torch.full_like(x, float("nan"))
    dg = torch.full((4, D), float("nan"), dtype=torch.float32, device="cuda")
    db = torch.full((4, D), float("nan"), dtype=torch.float32, device="cuda")
    if name == "workspace":
        ws = torch.empty(max(1, mtgr.mtgr_group_layernorm_bwd_workspace_size(T, D)), dtype=torch.uint8,
                         device="cuda")
        mtgr.mtgr_group_layernorm_bwd(d["dy"], x, mean, rstd, d["gid"], d["gamma"], d["dres"], dx, dg, db, ws)
    else:
        mtgr.mtgr_group_layernorm_bwd_noalloc(d["dy"], x, mean, rstd, d["gid"], d["gamma"], d["dres"], dx, dg, db)
    torch.cuda.synchronize()
    return {"dx": to_np(dx), "dgamma": to_np(dg), "dbeta": to_np(db)}


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 1024), (torch.bfloat16, 4096), (torch.float32, 4096),
                                     (torch.float32, 64)])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(orc, dtype, D):
    need_gpu()
    bf = dtype == torch.bfloat16
    tol = TOL_BF16 if bf else TOL_F32
    # first call: many rows (as many blocks as the scratch holds);
    # second call: few rows and other values (fewer blocks, stale scratch beyond them)
    for seed, T in ((11, 6000), (12, 300)):
        d, h = _inputs(seed, T, D, dtype)
        ws, na = _run(d, "workspace"), _run(d, "noalloc")
        for k in ("dx", "dgamma", "dbeta"):
            assert_close(na[k], ws[k], TOL_F32, f"noalloc vs workspace {k} (T={T}, D={D})")
        rdx, rdg, rdb = orc.gln_bwd(h["dy"], h["x"], h["gid"], h["gamma"])
        check_dx = assert_close_bf16 if bf else assert_close
        check_dx(na["dx"], rdx + h["dres"], tol, f"noalloc dx vs oracle (T={T}, D={D})")
        assert_close(na["dgamma"], rdg, tol, f"noalloc dgamma vs oracle (T={T}, D={D})")
        assert_close(na["dbeta"], rdb, tol, f"noalloc dbeta vs oracle (T={T}, D={D})")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_zero_rows_gives_zero_parameter_gradients(dtype):
    """T = 0: still one block, which writes zero partial sums; dγ and dβ come
    back zero, not the NaN they were filled with (also after a call on rows)."""
    need_gpu()
    d, _ = _inputs(13, 500, 256, dtype)
    _run(d, "noalloc")
    e, _ = _inputs(14, 0, 256, dtype)
    r = _run(e, "noalloc")
    assert r["dx"].shape == (0, 256)
    assert np.all(r["dgamma"] == 0.0) and np.all(r["dbeta"] == 0.0)


def test_noalloc_rejects_oversized_d():
    need_gpu()
    from hstu_attention_attn_b300 import mtgr
    T, D = 4, 8192
    d, _ = _inputs(15, T, D, torch.bfloat16)
    mean = torch.zeros(T, dtype=torch.float32, device="cuda")
    rstd = torch.ones(T, dtype=torch.float32, device="cuda")
    dx = torch.empty_like(d["x"])
    dg = torch.empty((4, D), dtype=torch.float32, device="cuda")
    db = torch.empty((4, D), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError, match="maximum of 4096"):
        mtgr.mtgr_group_layernorm_bwd_noalloc(d["dy"], d["x"], mean, rstd, d["gid"], d["gamma"], d["dres"], dx, dg, db)
