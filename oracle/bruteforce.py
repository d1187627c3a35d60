"""Brute-force NumPy restatement of the attention core -- TEST INFRASTRUCTURE ONLY.

Independent of ``mtgr_oracle.c``: it builds the explicit n x n mask matrix of
each user from the three rules of the dynamic mixed mask (fun-rec chapter 7.3,
§7.3.4; zzxanthony MTGR post §9) with vectorised comparisons, then evaluates
the block formula of the marovi.ai summary ("Métodos") densely with
``numpy.matmul``:  O = ((silu(Q Kᵀ / sqrt(d_h)) ⊙ M) / n_u) · V.
Used only to pin the C oracle on tiny inputs.
"""
from __future__ import annotations

import numpy as np

USER, SEQ, RT, CAND = 0, 1, 2, 3


def mask_matrix(gid: np.ndarray, ts: np.ndarray) -> np.ndarray:
    """Explicit visibility matrix of one user segment (rows = queries)."""
    gid = np.asarray(gid)
    ts = np.asarray(ts, dtype=np.int64)
    n = len(gid)
    row_g = gid[:, None]
    col_g = gid[None, :]
    row_t = ts[:, None]
    col_t = ts[None, :]
    # rule 1: User and Seq columns are visible to every row
    static_cols = np.isin(col_g, (USER, SEQ)) & np.ones((n, n), bool)
    # rule 2: a RealTime column is visible to RealTime rows at or after it and
    # to candidate rows strictly after it
    rt_cols = (col_g == RT) & (((row_g == RT) & (col_t <= row_t)) | ((row_g == CAND) & (col_t < row_t)))
    # rule 3: candidate columns only on the diagonal
    cand_cols = (col_g == CAND) & np.eye(n, dtype=bool)
    return static_cols | rt_cols | cand_cols


def attn_core(offsets, gid, ts, H, dh, q, k, v, n_override=0.0):
    T = int(offsets[-1])
    O = np.zeros((T, H * dh))
    for b in range(len(offsets) - 1):
        s0, s1 = int(offsets[b]), int(offsets[b + 1])
        if s1 == s0:
            continue
        M = mask_matrix(gid[s0:s1], ts[s0:s1]).astype(np.float64)
        n = n_override if n_override > 0 else float(s1 - s0)
        for h in range(H):
            cols = slice(h * dh, (h + 1) * dh)
            Q = np.asarray(q[s0:s1, cols], np.float64)
            K = np.asarray(k[s0:s1, cols], np.float64)
            V = np.asarray(v[s0:s1, cols], np.float64)
            S = (Q @ K.T) / np.sqrt(dh)
            A = S / (1.0 + np.exp(-S)) * M / n
            O[s0:s1, cols] = A @ V
    return O


def visible_counts(offsets, gid, ts):
    T = int(offsets[-1])
    cnt = np.zeros(T, np.int64)
    for b in range(len(offsets) - 1):
        s0, s1 = int(offsets[b]), int(offsets[b + 1])
        if s1 > s0:
            cnt[s0:s1] = mask_matrix(gid[s0:s1], ts[s0:s1]).sum(axis=1)
    return cnt
