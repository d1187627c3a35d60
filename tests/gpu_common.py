"""Fixtures shared by the GPU parity tests."""
import numpy as np
import pytest
import torch

from hstu_attention_attn_b300 import synth


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hstu_attention_attn_b300 import build
    build.build()


def dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype)


def bf16_round(a):
    """The bf16 values the GPU sees, widened back (host-side rounding by torch)."""
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def ragged_users(rng=None):
    """Users whose segments span several 128-row tiles with ragged tails, plus
    degenerate ones (no RealTime, one candidate, a lone token, an empty user)."""
    return [(8, 5, 0, 1), (8, 300, 64, 20), (4, 117, 10, 3), (8, 700, 33, 20), (1, 0, 0, 0),
            (0, 0, 0, 0), (8, 128 - 8, 0, 0), (2, 250, 1, 5), (0, 0, 7, 9)]


def sub_batch(batch, users):
    """Rows of the chosen users as a batch of their own (users are independent)."""
    rows, offs = [], [0]
    for b in users:
        s0, s1 = int(batch.offsets[b]), int(batch.offsets[b + 1])
        rows.append(np.arange(s0, s1))
        offs.append(offs[-1] + s1 - s0)
    rows = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    return synth.Batch(np.asarray(offs, np.int32), batch.gid[rows], batch.ts[rows]), rows


def f16_round(a):
    """Round to f16 and back (the values an f16 tensor holds)."""
    return np.asarray(a, np.float32).astype(np.float16).astype(np.float32)
