"""The mask invariants on the tcgen05 attention path (bf16 inputs, f16 O).

The harness of tests/invariants.py, checked on the oracle by
tests/test_invariant_harness.py, is run here on the GPU.  Every comparison
sets a row of an edited batch against the same row of the base batch; both
see the same keys and differ only in n_u, so n_u * O agrees to within two
f16 roundings of O (each at most 2^-11 relative) and a change of fp32
summation order: the bound is 2^-9 relative plus 1e-4 of RMS."""
import pytest
import torch

from hstu_attention_attn_b300.layer import HstuAttention, device_batch
from tests.gpu_common import dev, need_gpu
from tests.invariants import check_invariants
from tests.test_invariant_harness import EDITED, invariant_inputs

pytestmark = pytest.mark.gpu


def test_mask_invariants_on_the_gpu():
    need_gpu()
    H, dh = 2, 64
    rng, batch, q, k, v = invariant_inputs(17, H, dh)
    op = HstuAttention(H, dh, torch.bfloat16)

    def attn(bt, q_, k_, v_):
        qt, kt, vt = (dev(m, torch.bfloat16) for m in (q_, k_, v_))
        _, saved = op.forward(qt, kt, vt, torch.ones_like(qt), device_batch(bt))
        torch.cuda.synchronize()
        return saved[0].double().cpu().numpy()

    fails, control = check_invariants(attn, batch, q, k, v, EDITED, rng, rel=2.0 ** -9, atol_frac=1e-4)
    assert not fails, fails
    assert control > 1e-2      # an earlier RealTime token does reach the last candidate
