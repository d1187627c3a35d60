"""Chunked candidate scoring of one ranking request with the history encoded
once (mtgr_hstu_stack_hist_fwd + mtgr_hstu_stack_cand_fwd) vs the whole request
run at once (the library's stack) and vs the fp64 oracle's layers chained over
the whole request.  Under the dynamic mixed mask the history rows never see a
candidate and a candidate sees only the history and itself, with n_u the whole
request's token count, so a chunk's rows equal the whole request's rows."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import synth
from hstu_attention_attn_b300.layer import HstuLayer, HstuStack, device_batch
from tests.gpu_common import bf16_round, f16_round, need_gpu
from tests.util import TOL_BF16, assert_close, assert_close_bf16, assert_close_f16, to_np

pytestmark = pytest.mark.gpu


def _request(seed, user, D, H, dh, n_layers):
    rng = np.random.default_rng(seed)
    batch = synth.make_batch(rng, [user], ts_hi=3000)
    weights = []
    for _ in range(n_layers):
        w_uqkv = synth.xavier(rng, D, 4 * H * dh)
        w_o = synth.xavier(rng, H * dh, D)
        gamma, beta = synth.gln_params(rng, D)
        weights.append((w_uqkv, w_o, gamma, beta))
    x = synth.normal(rng, (batch.T, D))
    return batch, weights, x


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("user,chunk", [((8, 200, 30, 150), 64), ((4, 90, 0, 40), 16), ((8, 300, 64, 20), 20)])
def test_chunked_candidates_equal_whole_request_and_oracle(orc, dtype, user, chunk):
    need_gpu()
    D, H, dh, n_layers = 256, 2, 128, 3
    batch, weights, x = _request(17 + sum(user), user, D, H, dh, n_layers)
    n_cand = user[3]
    n_hist = batch.T - n_cand
    layers = [HstuLayer(D, H, dh, *(torch.from_numpy(w) for w in ws), dtype=dtype) for ws in weights]
    db = device_batch(batch)
    xd = torch.from_numpy(x).cuda().to(dtype)
    stack = HstuStack(layers)
    whole = stack.forward(xd, db).clone()
    chunked = stack.score_chunked(xd, db.gid, db.ts, n_hist, chunk)
    torch.cuda.synchronize()
    got = to_np(chunked)
    # the same rows as the whole request through the same kernels, up to the
    # order of fp32 sums: the candidate's own key sits in another tile position,
    # and the whole request (more rows) runs its output projection split over K
    # where a chunk does not, so x' is rounded to 16 bits from another fp32 sum;
    # held to 5e-3 beyond one rounding of the stored type, 4x inside the bound
    # against the oracle below
    check_close = assert_close_bf16 if dtype == torch.bfloat16 else assert_close_f16
    check_close(got, to_np(whole)[n_hist:], 5e-3, "chunked vs whole request")
    # the oracle's layers chained over the whole request on the same 16-bit inputs
    rnd = bf16_round if dtype == torch.bfloat16 else (lambda a: np.asarray(f16_round(a), np.float64))
    h = rnd(x)
    for (wu, wo, g, b) in weights:
        h = orc.layer_fwd_blas(batch, D, H, dh, h, rnd(wu), rnd(wo), g, b)["x_out"]
    check = assert_close_bf16 if dtype == torch.bfloat16 else assert_close_f16
    check(got, h[n_hist:], TOL_BF16, "chunked candidates vs oracle")


def test_chunked_rejects_bad_chunk():
    need_gpu()
    from hstu_attention_attn_b300 import mtgr
    D, H, dh = 256, 2, 128
    batch, weights, x = _request(3, (8, 50, 5, 10), D, H, dh, 1)
    layer = HstuLayer(D, H, dh, *(torch.from_numpy(w) for w in weights[0]), dtype=torch.bfloat16)
    db = device_batch(batch)
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    n_hist = batch.T - 10
    ws = torch.empty(mtgr.mtgr_stack_chunk_workspace_size(n_hist, 4, D, H, dh, mtgr.MTGR_BF16), dtype=torch.uint8,
                     device="cuda")
    cache = torch.empty(mtgr.mtgr_stack_cache_size(1, n_hist, 4, D, H, dh), dtype=torch.uint8, device="cuda")
    out = torch.empty(10, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError, match="chunk"):   # 10 candidates in one call of a 4-candidate chunk
        mtgr.mtgr_hstu_stack_cand_fwd([layer.weights], xd[n_hist:], out, out, cache, 4, db.gid, db.ts, n_hist, 10, 0,
                                      ws)
