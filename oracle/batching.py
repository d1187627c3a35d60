"""Oracle of the host-side batch construction -- TEST INFRASTRUCTURE ONLY
(imported by ``tests/`` alone; shares no code with the library).

Plain Python loops over the definitions:

* stochastic length (paper-daily "MTGR：美团外卖生成式推荐Scaling Law落地实践",
  "计算量涨了 65 倍…": training shortens long user sequences by sampling a
  piece of them, scoring keeps the whole sequence), in the reading that keeps
  User, RealTime and candidate tokens and a window of ``max_seq`` consecutive
  Seq tokens whose start within the Seq run is ``draw mod (n_S - max_seq + 1)``;
* token-balanced contiguous split of users over ranks (zzxanthony.github.io
  "MTGR：工业级生成式推荐框架", §11.3 "Dynamic batch size 做负载均衡"): the
  smallest possible largest per-rank token count, by enumerating every cut.
"""
from __future__ import annotations

import itertools


def stochastic_length(offsets, gid, max_seq, draws):
    """Returns (keep, new_offsets) as Python lists."""
    keep, new_offsets = [], [0]
    for u in range(len(offsets) - 1):
        s0, s1 = int(offsets[u]), int(offsets[u + 1])
        tokens = list(range(s0, s1))
        user = [t for t in tokens if gid[t] == 0]
        seq = [t for t in tokens if gid[t] == 1]
        rest = [t for t in tokens if gid[t] >= 2]
        if len(seq) > max_seq:
            start = int(draws[u]) % (len(seq) - max_seq + 1)
            seq = seq[start:start + max_seq]
        keep += user + seq + rest
        new_offsets.append(len(keep))
    return keep, new_offsets


def min_max_split(tokens, n_ranks):
    """Smallest possible largest group sum over all cuts of `tokens` (in
    order) into n_ranks contiguous, possibly empty, groups."""
    B = len(tokens)
    best = None
    for cuts in itertools.combinations_with_replacement(range(B + 1), n_ranks - 1):
        bounds = (0,) + cuts + (B,)
        worst = max(sum(tokens[bounds[r]:bounds[r + 1]]) for r in range(n_ranks))
        best = worst if best is None else min(best, worst)
    return best
