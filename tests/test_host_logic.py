"""Host logic of the GEMM split-K path, on the CPU.

For a request of S slices over K, gemm_splits (gemm.cuh) returns the number
of fp32 slices the tcgen05 GEMM writes and the caller reduces.  The kernel
gives slice s the K blocks [s*per, min((s+1)*per, nk)) of 64 columns, with
nk = ceil(K/64) and per = ceil(nk/slices).  Every slice must hold at least
one block (an empty slice would be written from an accumulator no MMA ever
initialised), the slices must cover all nk blocks, and the count must not
exceed the request."""
import os
import shutil
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "hstu_attention_attn_b300", "csrc")


def test_gemm_splits_partition_k(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "gemm_splits")
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-o", exe, os.path.join(HERE, "gemm_splits.cu")], check=True)
    out = subprocess.run([exe, "1100"], capture_output=True, text=True, check=True).stdout
    rows = np.array([line.split() for line in out.splitlines()], dtype=np.int64)
    assert len(rows) == 1100 * 21
    for K, req, slices in rows:
        nk = -(-K // 64)
        assert 1 <= slices <= max(req, 1) and slices <= nk, (K, req, slices)
        per = -(-nk // slices)
        starts = np.arange(slices) * per
        ends = np.minimum(starts + per, nk)
        assert np.all(ends > starts), (K, req, slices)      # no empty slice
        assert ends[-1] == nk                               # all K blocks covered, once
    # a request well below the block count is honoured exactly (K = 8,800: 138 blocks)
    got = {(int(K), int(r)): int(s) for K, r, s in rows}
    assert got[(8 * 1100, 8)] == 8 and got[(8 * 1100, 16)] == 16
