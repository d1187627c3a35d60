"""The dynamic mixed mask's invariants as edits of one batch (fun-rec chapter
7.3, §7.3.4; the specification of this build lists the three):

* a candidate's output does not change when other candidates of its user are
  removed, permuted or added;
* User/Seq outputs do not change under any edit of the user's RealTime and
  candidate tokens (values, stamps, or removal);
* a candidate's output does not change when RealTime tokens stamped at or
  after it are added -- and does change for one stamped before it.

Edits change the user's token count n_u, which scales every row of that user
by a common factor (reading c7), so the comparisons are made on the
unnormalised output n_u * O.  `attn(batch, q, k, v)` returns O [T, H*d_h]; it is
the fp64 oracle in the CPU test of this harness and the tcgen05 path in the
GPU test, which share every edit and every row mapping below.
"""
from __future__ import annotations

import numpy as np

from hstu_attention_attn_b300 import synth

G_RT, G_CAND = synth.G_RT, synth.G_CAND


class Case:
    """A batch held as per-user token lists; `ids` maps each token to its row
    in the base batch (-1 for a token an edit added)."""

    def __init__(self, users):
        self.users = users          # list of dicts: gid, ts, q, k, v, ids

    @classmethod
    def base(cls, batch, q, k, v):
        users = []
        for b in range(batch.B):
            s0, s1 = int(batch.offsets[b]), int(batch.offsets[b + 1])
            users.append(dict(gid=batch.gid[s0:s1].copy(), ts=batch.ts[s0:s1].copy(), q=q[s0:s1].copy(),
                              k=k[s0:s1].copy(), v=v[s0:s1].copy(), ids=np.arange(s0, s1)))
        return cls(users)

    def with_user(self, b, **arrays):
        users = [dict(u) for u in self.users]
        users[b] = dict(users[b], **arrays)
        return Case(users)

    def select(self, b, rows):
        """User b keeps its tokens `rows` (indices into the user), in that order."""
        u = self.users[b]
        return self.with_user(b, **{n: u[n][rows] for n in ("gid", "ts", "q", "k", "v", "ids")})

    def insert(self, b, pos, gid, ts, rng):
        """New tokens of groups `gid` and stamps `ts` inserted at `pos` of user b."""
        u = self.users[b]
        n, w = len(gid), u["q"].shape[1]
        new = {n_: np.insert(u[n_], pos, vals, axis=0) for n_, vals in
               (("gid", np.asarray(gid, np.uint8)), ("ts", np.asarray(ts, np.int64)), ("ids", [-1] * n))}
        for m in ("q", "k", "v"):
            new[m] = np.insert(u[m], pos, rng.standard_normal((n, w)).astype(u[m].dtype), axis=0)
        return self.with_user(b, **new)

    def batch(self):
        offs = np.cumsum([0] + [len(u["gid"]) for u in self.users]).astype(np.int32)
        cat = lambda n: np.concatenate([u[n] for u in self.users])
        return synth.Batch(offs, cat("gid").astype(np.uint8), cat("ts").astype(np.int64)), cat("q"), cat("k"), \
            cat("v"), cat("ids")


def o_hat(attn, case):
    """n_u * O for every row of the case, and the rows' base ids."""
    batch, q, k, v, ids = case.batch()
    O = np.asarray(attn(batch, q, k, v), np.float64)
    n = np.repeat(np.diff(batch.offsets), np.diff(batch.offsets)).astype(np.float64)
    return O * n[:, None], ids, batch


def rows_match(got, want, rel, atol_frac):
    """Largest error beyond `rel` * max(|got|, |want|), as a fraction of RMS(want)."""
    if want.size == 0:
        return 0.0
    scale = max(float(np.sqrt(np.mean(want ** 2))), 1e-300)
    err = np.abs(got - want) - rel * np.maximum(np.abs(got), np.abs(want))
    return float(max(err.max(), 0.0)) / scale


def check_invariants(attn, batch, q, k, v, b, rng, rel, atol_frac):
    """Runs every edit on user b of the batch; returns the list of failures
    (empty when all invariants hold) and the positive control's deviation."""
    base_case = Case.base(batch, q, k, v)
    base, _, _ = o_hat(attn, base_case)
    u = base_case.users[b]
    cand = np.where(u["gid"] == G_CAND)[0]
    rt = np.where(u["gid"] == G_RT)[0]
    static = np.where(u["gid"] < G_RT)[0]
    assert len(cand) >= 6 and len(rt) >= 2 and len(static) > 0, "user b needs RealTime tokens and candidates"
    fails = []

    def compare(name, case, rows_of_b):
        got, ids, bt = o_hat(attn, case)
        s0 = int(bt.offsets[b])
        # rows of other users are untouched by the edit
        other = np.array([i for i in range(bt.T) if not (s0 <= i < int(bt.offsets[b + 1]))], np.int64)
        for what, rows in (("edited user", s0 + np.asarray(rows_of_b, np.int64)), ("other users", other)):
            rows = rows[ids[rows] >= 0]
            e = rows_match(got[rows], base[ids[rows]], rel, atol_frac)
            if e > atol_frac:
                fails.append(f"{name}: {what} moved by {e:.3g} of RMS")

    # candidates: two removed, then all permuted, then three added
    keep = np.array([i for i in range(len(u["gid"])) if i not in (cand[1], cand[4])])
    c1 = base_case.select(b, keep)
    compare("candidates removed", c1, np.where(c1.users[b]["gid"] == G_CAND)[0])
    perm = np.concatenate([np.arange(cand[0]), cand[0] + rng.permutation(len(cand))])
    c2 = base_case.select(b, perm)
    compare("candidates permuted", c2, np.where(c2.users[b]["gid"] == G_CAND)[0])
    c3 = base_case.insert(b, len(u["gid"]), [G_CAND] * 3, [5, 40000, 86400], rng)
    compare("candidates added", c3, np.where(c3.users[b]["gid"] == G_CAND)[0])
    # User/Seq rows: every RealTime / candidate value and stamp redrawn, then all of them dropped
    tail = np.arange(len(static), len(u["gid"]))
    new = {m: u[m].copy() for m in ("q", "k", "v", "ts")}
    for m in ("q", "k", "v"):
        new[m][tail] = rng.standard_normal((len(tail), u[m].shape[1])).astype(u[m].dtype)
    new["ts"][tail] = np.sort(rng.integers(0, 86400, len(tail)))
    new["ts"][len(static) + len(rt):] = np.sort(new["ts"][len(static) + len(rt):])
    c4 = base_case.with_user(b, **new)
    compare("RealTime and candidates redrawn", c4, static)
    c5 = base_case.select(b, static)
    compare("RealTime and candidates dropped", c5, static)
    # candidates and RealTime stamped at or after every candidate
    late = int(u["ts"][cand].max())
    c6 = base_case.insert(b, int(rt[-1]) + 1, [G_RT] * 2, [late, late + 100], rng)
    compare("RealTime added after the candidates", c6, np.where(c6.users[b]["gid"] == G_CAND)[0])
    # positive control: a RealTime token stamped before the last candidate moves that candidate
    c7 = base_case.insert(b, int(rt[-1]) + 1, [G_RT], [int(u["ts"][cand[-1]]) - 1], rng)
    got7, ids7, bt7 = o_hat(attn, c7)
    last = int(bt7.offsets[b + 1]) - 1
    control = rows_match(got7[last:last + 1], base[ids7[last:last + 1]], 0.0, 0.0)
    return fails, control
