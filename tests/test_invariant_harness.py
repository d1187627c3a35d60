"""The mask-invariant harness (tests/invariants.py) run on the fp64 oracle,
where the invariants hold exactly: this checks the harness itself (its edits
and row mappings) before the GPU test runs the same harness on the tcgen05
path."""
import numpy as np

from hstu_attention_attn_b300 import synth
from tests.gpu_common import bf16_round, ragged_users
from tests.invariants import check_invariants

USERS = ragged_users()[:4] + [(8, 300, 40, 20)] + ragged_users()[4:7]
EDITED = 4


def invariant_inputs(seed, H, dh):
    rng = np.random.default_rng(seed)
    batch = synth.make_batch(rng, USERS)
    q, k, v = (bf16_round(rng.standard_normal((batch.T, H * dh)).astype(np.float32)) for _ in range(3))
    return rng, batch, q, k, v


def test_invariant_harness_on_the_oracle(orc):
    H, dh = 2, 64
    rng, batch, q, k, v = invariant_inputs(17, H, dh)
    fails, control = check_invariants(lambda bt, q_, k_, v_: orc.attn_core_fwd(bt, H, dh, q_, k_, v_),
                                      batch, q, k, v, EDITED, rng, rel=1e-12, atol_frac=1e-12)
    assert not fails, fails
    assert control > 1e-3      # an earlier RealTime token does reach the last candidate


def test_invariant_harness_catches_a_leaky_mask(orc):
    """Planted on the CPU: the oracle fed a 'mask' in which candidates see each
    other (every candidate stamp replaced by a RealTime one before the call),
    must fail the candidate invariants."""
    H, dh = 2, 64
    rng, batch, q, k, v = invariant_inputs(17, H, dh)

    def leaky(bt, q_, k_, v_):
        g = bt.gid.copy()
        g[g == 3] = 2          # candidates become RealTime tokens: they see one another by stamp
        return orc.attn_core_fwd(synth.Batch(bt.offsets, g, bt.ts), H, dh, q_, k_, v_)

    fails, _ = check_invariants(leaky, batch, q, k, v, EDITED, rng, rel=1e-12, atol_frac=1e-12)
    assert any(f.startswith("candidates") for f in fails), fails


def test_invariant_bound_admits_f16_rounding_of_o(orc):
    """The GPU test's bound (2^-9 relative + 1e-4 of RMS) admits the f16
    rounding of O that the tcgen05 path stores: the oracle's O rounded to f16
    passes the harness at that bound."""
    from tests.gpu_common import f16_round
    H, dh = 2, 64
    rng, batch, q, k, v = invariant_inputs(17, H, dh)
    f16_oracle = lambda bt, q_, k_, v_: f16_round(orc.attn_core_fwd(bt, H, dh, q_, k_, v_)).astype(np.float64)
    fails, control = check_invariants(f16_oracle, batch, q, k, v, EDITED, rng, rel=2.0 ** -9, atol_frac=1e-4)
    assert not fails, fails
    assert control > 1e-2
