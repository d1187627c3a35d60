"""Tile plan of the attention kernels against the oracle's mask, on the CPU.

The kernels visit (query tile, key tile) pairs from the rules in plan.cuh
(compiled here as host code by tests/plan_lists.cu).  The plan never looks at
timestamps, so it must cover every pair that some choice of stamps can make
visible: the mask with every RealTime key visible to every RealTime and
candidate row (all RealTime stamps 0, candidate stamps 1), built by the
oracle's explicit mask matrix (fun-rec chapter 7.3, §7.3.4).  Each list
below must equal that tile set exactly: nothing visible is skipped and no
fully masked tile is visited.  Users sweep tile-boundary cases of every
group size, including empty groups and an empty user."""
import itertools
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle.bruteforce import mask_matrix

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "hstu_attention_attn_b300", "csrc")
TILE = 128


@pytest.fixture(scope="module")
def plan_lists(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_lists")
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-o", exe, os.path.join(HERE, "plan_lists.cu")], check=True)

    def run(users):
        inp = "".join(f"{n} {eS} {eR}\n" for n, eS, eR in users)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
        res = []
        for line in out.splitlines():
            f = line.split()
            if f[0] == "U":
                res.append({"nt": int(f[4]), "Q": {}, "K": {}, "P": []})
            elif f[0] in ("SR", "SW"):
                res[-1][f[0]] = [int(v) for v in f[1:]]
            elif f[0] == "Q":
                res[-1]["Q"][int(f[1])] = [int(v) for v in f[2:]]
            elif f[0] == "K":
                res[-1]["K"][int(f[1])] = [int(v) for v in f[2:]]
            else:
                mem = [(int(a), b[0] == "1", b[1] == "1") for a, b in (t.split(":") for t in f[4:])]
                res[-1]["P"].append((int(f[1]), int(f[2]), int(f[3]), mem))
        return res
    return run


def _users():
    sizes = itertools.product((0, 1, 8), (0, 1, 119, 120, 127, 128, 247, 248, 300),
                              (0, 1, 7, 8, 64, 128, 136), (0, 1, 20, 128, 129))
    return [s for s in sizes]


def _needed_tiles(nU, nS, nR, K):
    gid = np.array([0] * nU + [1] * nS + [2] * nR + [3] * K, np.uint8)
    ts = np.where(gid == 3, 1, 0).astype(np.int64)
    n = len(gid)
    nt = -(-n // TILE)
    M = np.zeros((nt * TILE, nt * TILE), bool)
    M[:n, :n] = mask_matrix(gid, ts)
    return M.reshape(nt, TILE, nt, TILE).any(axis=(1, 3))


def test_tile_lists_equal_the_visible_tiles(plan_lists):
    users = _users()
    meta = [(nU + nS + nR + K, nU + nS, nU + nS + nR) for nU, nS, nR, K in users]
    lists = plan_lists(meta)
    assert len(lists) == len(users)
    visited = 0
    for (nU, nS, nR, K), L in zip(users, lists):
        need = _needed_tiles(nU, nS, nR, K)
        nt = need.shape[0]
        assert L["nt"] == nt
        for qt in range(nt):    # dQ kernel: key tiles of each query tile, ascending, no repeats
            ks = L["Q"][qt]
            assert ks == sorted(set(ks)), (nU, nS, nR, K, qt)
            assert ks == list(np.nonzero(need[qt])[0]), (nU, nS, nR, K, qt)
            visited += len(ks)
        for kt in range(nt):    # dK/dV kernel: query tiles of each key tile
            qs = L["K"][kt]
            assert len(qs) == len(set(qs)), (nU, nS, nR, K, kt)
            assert sorted(qs) == list(np.nonzero(need[:, kt])[0]), (nU, nS, nR, K, kt)
        # forward items: pairs (qa, qa + 1) or single tiles; each query tile in exactly one item
        for single in (0, 1):
            items = [p for p in L["P"] if p[0] == single]
            covered = sorted([qa for _, qa, _, _ in items] + [qb for _, _, qb, _ in items if qb >= 0])
            assert covered == list(range(nt)), (nU, nS, nR, K, single)
            for _, qa, qb, mem in items:
                assert qb == (qa + 1 if not single and qa + 1 < nt else -1)
                kts = [kt for kt, _, _ in mem]
                assert kts == sorted(set(kts)), (nU, nS, nR, K, qa)
                assert [kt for kt, a, _ in mem if a] == list(np.nonzero(need[qa])[0])
                want_b = list(np.nonzero(need[qb])[0]) if qb >= 0 else []
                assert [kt for kt, _, b in mem if b] == want_b
                assert all(a or b for _, a, b in mem)
    assert visited > 1000


def test_ds_tile_slots_written_and_read_agree(plan_lists):
    """The backward's stored dS tiles: the dK/dV pass writes tile (head, key
    tile, query tile) to the slot the dQ pass reads it from, every visited
    pair of every head has a slot of its own, and all slots lie in the user's
    H * nt^2 range (plan.cuh's ds_slot, compiled as host code)."""
    users = _users()
    lists = plan_lists([(nU + nS + nR + K, nU + nS, nU + nS + nR) for nU, nS, nR, K in users])
    for (nU, nS, nR, K), L in zip(users, lists):
        nt, rd, wr = L["nt"], L["SR"], L["SW"]
        assert len(rd) == len(set(rd)) and len(wr) == len(set(wr)), (nU, nS, nR, K)
        assert sorted(rd) == sorted(wr), (nU, nS, nR, K)
        assert all(0 <= v < 3 * nt * nt for v in rd), (nU, nS, nR, K)
        assert len(rd) == 3 * sum(len(v) for v in L["Q"].values())
