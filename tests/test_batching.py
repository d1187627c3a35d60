"""Host-side batch construction (stochastic length, token-balanced ranks): the
oracle against what the definitions fix, then the library against the oracle
(bit-exact for the selection; for the split the minimax value, which is
unique, plus the validity of the cut, which need not be)."""
import numpy as np
import pytest

from hstu_attention_attn_b300 import synth
from oracle import batching as ob


def _batch(users, seed):
    return synth.make_batch(np.random.default_rng(seed), users)


# ---------------------------------------------------------------------------
# oracle pins
# ---------------------------------------------------------------------------
def pin_stochastic_length(ob):
    """What the definition fixes for the stochastic-length oracle `ob`."""
    b = _batch([(8, 30, 5, 3), (0, 0, 2, 1), (2, 7, 0, 4)], 1)
    keep, off = ob.stochastic_length(b.offsets, b.gid, 1000, [5, 6, 7])
    assert keep == list(range(b.T)) and off == list(b.offsets)
    # hand example: User 0,1; Seq 2..7; RealTime 8; candidate 9 | Seq 10; candidates 11, 12
    gid = [0, 0, 1, 1, 1, 1, 1, 1, 2, 3, 1, 3, 3]
    keep, off = ob.stochastic_length([0, 10, 13], gid, 3, [7, 2])
    assert keep == [0, 1, 5, 6, 7, 8, 9, 10, 11, 12] and off == [0, 7, 10]   # 7 mod (6-3+1) = 3
    # windows at the start and in the middle of the Seq run: 0 mod 4 = 0, 5 mod 4 = 1
    keep, off = ob.stochastic_length([0, 10, 13], gid, 3, [0, 2])
    assert keep == [0, 1, 2, 3, 4, 8, 9, 10, 11, 12] and off == [0, 7, 10]
    keep, off = ob.stochastic_length([0, 10, 13], gid, 3, [5, 2])
    assert keep == [0, 1, 3, 4, 5, 8, 9, 10, 11, 12] and off == [0, 7, 10]
    keep, off = ob.stochastic_length([0, 10, 13], gid, 0, [7, 2])
    assert keep == [0, 1, 8, 9, 11, 12] and off == [0, 4, 6]


def pin_min_max_split(ob):
    """Closed forms and the pages' picture for the token-balanced split oracle `ob`."""
    assert ob.min_max_split([3, 1, 4, 1, 5], 1) == 14
    assert ob.min_max_split([3, 1, 4, 1, 5], 5) == 5
    assert ob.min_max_split([3, 1, 4, 1, 5], 9) == 5       # more ranks than users: the largest user
    assert ob.min_max_split([7] * 9, 3) == 21 and ob.min_max_split([7] * 10, 3) == 28
    assert ob.min_max_split([5, 1, 1, 1, 1, 5, 5, 5], 2) == 14
    # the pages' two-card picture: four users per card at first; the card with the
    # shorter users takes a fifth so that both hold the same tokens
    assert ob.min_max_split([800] * 5 + [1000] * 4, 2) == 4000


def test_oracle_stochastic_length_identity_and_window():
    pin_stochastic_length(ob)


def test_oracle_min_max_split_closed_forms():
    pin_min_max_split(ob)


# ---------------------------------------------------------------------------
# library vs oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed,max_seq", [(0, 64), (1, 300), (2, 0), (3, 10_000)])
def test_stochastic_length_matches_oracle(seed, max_seq):
    from hstu_attention_attn_b300 import mtgr
    rng = np.random.default_rng(seed)
    users = synth.large_users(rng, 40) + [(0, 0, 0, 0), (4, 0, 3, 2), (0, 50, 0, 0), (1, 0, 0, 0)]
    b = _batch(users, seed)
    draws = rng.integers(0, 2**63, size=b.B, dtype=np.uint64) * np.uint64(2) + np.uint64(1)  # full 64-bit range
    keep, off = mtgr.mtgr_stochastic_length(b.offsets, b.gid, max_seq, draws)
    rkeep, roff = ob.stochastic_length(b.offsets, b.gid, max_seq, draws)
    assert keep.tolist() == rkeep and off.tolist() == roff
    # the kept batch is a batch: group order holds and the gathered metadata validates
    g2 = b.gid[keep]
    for u in range(b.B):
        seg = g2[off[u]:off[u + 1]]
        assert np.all(np.diff(seg.astype(int)) >= 0)
        assert (seg == 1).sum() == min((b.gid[b.offsets[u]:b.offsets[u + 1]] == 1).sum(), max_seq)


def test_stochastic_length_empty_batch_and_errors():
    from hstu_attention_attn_b300 import mtgr
    keep, off = mtgr.mtgr_stochastic_length(np.array([0], np.int32), np.zeros(0, np.uint8), 5,
                                            np.zeros(0, np.uint64))
    assert keep.size == 0 and off.tolist() == [0]
    with pytest.raises(mtgr.MtgrError, match="offsets"):
        mtgr.mtgr_stochastic_length(np.array([0, 3, 2], np.int32), np.zeros(2, np.uint8), 5, np.zeros(2, np.uint64))
    with pytest.raises(mtgr.MtgrError, match="group ids"):
        mtgr.mtgr_stochastic_length(np.array([0, 3], np.int32), np.array([1, 0, 3], np.uint8), 5,
                                    np.zeros(1, np.uint64))
    with pytest.raises(mtgr.MtgrError):
        mtgr.mtgr_stochastic_length(np.array([0, 3], np.int32), np.array([0, 1, 3], np.uint8), -1,
                                    np.zeros(1, np.uint64))


def _check_cut(tokens, n_ranks, first, rank_tokens, weight, best):
    B = len(tokens)
    assert first[0] == 0 and first[-1] == B and np.all(np.diff(first) >= 0)
    for r in range(n_ranks):
        assert rank_tokens[r] == sum(tokens[first[r]:first[r + 1]])
        assert weight[r] == pytest.approx((first[r + 1] - first[r]) / B if B else 0.0)
        if B >= n_ranks:
            assert first[r + 1] > first[r], "a rank left without users"
    assert max(rank_tokens) == best


@pytest.mark.parametrize("seed", range(12))
def test_token_balanced_split_small_vs_bruteforce(seed):
    from hstu_attention_attn_b300 import mtgr
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 10))
    n_ranks = int(rng.integers(1, 5))
    tokens = [int(t) for t in rng.integers(0, 50, size=B)]
    first, rt, w = mtgr.mtgr_token_balanced_split(tokens, n_ranks)
    _check_cut(tokens, n_ranks, first, rt, w, ob.min_max_split(tokens, n_ranks))


def _minimax_dp(tokens, n_ranks):
    """Exact smallest largest group sum by dynamic programming over prefixes."""
    B = len(tokens)
    pre = np.concatenate([[0], np.cumsum(tokens)])
    best = [float(pre[i]) for i in range(B + 1)]  # one group: the prefix sums
    for _ in range(n_ranks - 1):
        nxt = [0.0] * (B + 1)
        for i in range(B + 1):
            nxt[i] = min(max(best[j], float(pre[i] - pre[j])) for j in range(i + 1))
        best = nxt
    return int(best[B])


def test_token_balanced_split_training_batch():
    from hstu_attention_attn_b300 import mtgr
    rng = np.random.default_rng(3)
    users = synth.large_users(rng, 200)
    tokens = [sum(u) for u in users]
    for n_ranks in (2, 3, 8):
        first, rt, w = mtgr.mtgr_token_balanced_split(tokens, n_ranks)
        _check_cut(tokens, n_ranks, first, rt, w, _minimax_dp(tokens, n_ranks))
        # balanced to within one user of the even share
        assert max(rt) - sum(tokens) / n_ranks <= max(tokens)
    with pytest.raises(mtgr.MtgrError):
        mtgr.mtgr_token_balanced_split([1, -2], 2)
    with pytest.raises(mtgr.MtgrError):
        mtgr.mtgr_token_balanced_split([1, 2], 0)
