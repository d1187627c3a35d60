"""Seeded synthetic inputs for the MTGR HSTU layer.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no mask, no SiLU, no normalisation).  Both the CUDA path
(tests, bench) and the fp64 oracle are fed from here.

Sample layout (MTGR, "Métodos", user-sample aggregation into one row
D = [U, S, R, (C, I)_1..K]; paper-daily "训练数据怎么组织", one row per user
with the raw timestamp of every action and exposure kept for the mask):

* tokens of one user are contiguous, in group order User*, Seq*, RealTime*,
  Cand*; ``offsets[b]..offsets[b+1]`` is user ``b``'s segment (int32, B+1);
* ``gid[t]`` in {0: User, 1: Seq, 2: RealTime, 3: Cand} (uint8);
* ``ts[t]`` int64 seconds.  RealTime and candidate stamps are independently
  sorted uniform draws in [0, 86400] (one day), so some candidates precede
  some RealTime tokens; User tokens carry 0 and Seq tokens sorted draws from
  the 30 days before the window (the mask ignores both).

Length distributions (configs of the MTGR-small / MTGR-large workloads):
Seq length is round(median * exp(sigma * N(0,1))) with sigma = 1.0, clamped.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np

G_USER, G_SEQ, G_RT, G_CAND = 0, 1, 2, 3
DAY = 86400


@dataclass
class Batch:
    offsets: np.ndarray          # int32 [B+1]
    gid: np.ndarray              # uint8 [T]
    ts: np.ndarray               # int64 [T]
    counts: list = field(default_factory=list)  # per user (nU, nS, nR, K)

    @property
    def B(self) -> int:
        return len(self.offsets) - 1

    @property
    def T(self) -> int:
        return int(self.offsets[-1])


def _user_tokens(rng, nU, nS, nR, K, ts_hi=DAY):
    gid = np.concatenate([np.full(nU, G_USER), np.full(nS, G_SEQ),
                          np.full(nR, G_RT), np.full(K, G_CAND)]).astype(np.uint8)
    ts_u = np.zeros(nU, np.int64)
    ts_s = np.sort(rng.integers(-30 * DAY, 0, size=nS, endpoint=False)).astype(np.int64)
    ts_r = np.sort(rng.integers(0, ts_hi, size=nR, endpoint=True)).astype(np.int64)
    ts_c = np.sort(rng.integers(0, ts_hi, size=K, endpoint=True)).astype(np.int64)
    return gid, np.concatenate([ts_u, ts_s, ts_r, ts_c])


def make_batch(rng, users, ts_hi=DAY) -> Batch:
    """users: list of (nU, nS, nR, K)."""
    gids, tss = [], []
    offs = [0]
    for (nU, nS, nR, K) in users:
        g, t = _user_tokens(rng, nU, nS, nR, K, ts_hi)
        gids.append(g)
        tss.append(t)
        offs.append(offs[-1] + len(g))
    gid = np.concatenate(gids) if gids else np.zeros(0, np.uint8)
    ts = np.concatenate(tss) if tss else np.zeros(0, np.int64)
    return Batch(np.asarray(offs, np.int32), gid, ts, list(users))


def lognormal_len(rng, median, lo, hi, sigma=1.0):
    return int(np.clip(np.rint(median * np.exp(sigma * rng.standard_normal())), lo, hi))


# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------
@dataclass
class Shape:
    name: str
    D: int
    H: int
    dh: int


TINY = Shape("tiny: 4 users, d_model 64, 2 heads x d_h 32", 64, 2, 32)
SMALL = Shape("MTGR-small-like attention: 64 users, d_model 512, 4 heads x d_h 128", 512, 4, 128)
LARGE = Shape("MTGR-large-like layer: d_model 1024, 8 heads x d_h 128", 1024, 8, 128)


def tiny_users(rng, n_users=4):
    return [(4, int(rng.integers(8, 48, endpoint=True)), int(rng.integers(0, 8, endpoint=True)),
             int(rng.integers(2, 6, endpoint=True))) for _ in range(n_users)]


def small_users(rng, n_users=64):
    return [(8, lognormal_len(rng, 400, 16, 3000), int(rng.integers(0, 64, endpoint=True)), 20)
            for _ in range(n_users)]


def large_users(rng, n_users=128):
    return [(8, lognormal_len(rng, 300, 16, 1000), int(rng.integers(0, 64, endpoint=True)), 20)
            for _ in range(n_users)]


def large_users_token_budget(rng, min_tokens=262144):
    """Users drawn from the MTGR-large length distribution until the batch holds
    at least ``min_tokens`` tokens (token-balanced batch of one training step)."""
    users, T = [], 0
    while T < min_tokens:
        u = (8, lognormal_len(rng, 300, 16, 1000), int(rng.integers(0, 64, endpoint=True)), 20)
        users.append(u)
        T += sum(u)
    return users


def inference_users(K, batch=1):
    return [(8, 1000, 64, K)] * batch


# --------------------------------------------------------------------------
# Tensors
# --------------------------------------------------------------------------
def normal(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def xavier(rng, fan_in, fan_out):
    bound = np.sqrt(6.0 / (fan_in + fan_out))
    return rng.uniform(-bound, bound, size=(fan_in, fan_out)).astype(np.float32)


def gln_params(rng, D, perturb=True):
    """Per-group (User/Seq/RealTime/Cand) scale and shift, [4, D] each.
    Tests perturb them around (1, 0) so every group has its own values."""
    if not perturb:
        return np.ones((4, D), np.float32), np.zeros((4, D), np.float32)
    g = (1.0 + 0.2 * rng.standard_normal((4, D))).astype(np.float32)
    b = (0.2 * rng.standard_normal((4, D))).astype(np.float32)
    return g, b


@dataclass
class AttnInputs:
    batch: Batch
    H: int
    dh: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    u: np.ndarray


def attn_inputs(seed: int, users_fn, H, dh, scale=1.0, ts_hi=DAY) -> AttnInputs:
    rng = np.random.default_rng(seed)
    batch = make_batch(rng, users_fn(rng), ts_hi)
    T, HD = batch.T, H * dh
    q, k, v, u = (normal(rng, (T, HD), scale) for _ in range(4))
    return AttnInputs(batch, H, dh, q, k, v, u)


@dataclass
class LayerInputs:
    batch: Batch
    D: int
    H: int
    dh: int
    x: np.ndarray        # [T, D]
    w_uqkv: np.ndarray   # [D, 4*H*dh], columns [U | Q | K | V], each head-major
    w_o: np.ndarray      # [H*dh, D]
    gamma: np.ndarray    # [4, D]
    beta: np.ndarray     # [4, D]
    dx_out: np.ndarray   # [T, D] upstream gradient


def layer_inputs(seed: int, users_fn, D, H, dh, grad="dense", ts_hi=DAY) -> LayerInputs:
    rng = np.random.default_rng(seed)
    batch = make_batch(rng, users_fn(rng), ts_hi)
    T, HD = batch.T, H * dh
    x = normal(rng, (T, D))
    w_uqkv = xavier(rng, D, 4 * HD)
    w_o = xavier(rng, HD, D)
    gamma, beta = gln_params(rng, D)
    dx = normal(rng, (T, D))
    if grad == "cand":   # loss only at candidate positions
        dx[batch.gid != G_CAND] = 0.0
    return LayerInputs(batch, D, H, dh, x, w_uqkv, w_o, gamma, beta, dx)


# Named workloads -----------------------------------------------------------
def tiny_attn(seed=0, ts_hi=DAY):
    return attn_inputs(seed, tiny_users, TINY.H, TINY.dh, 1.0, ts_hi)


def tiny_layer(seed=0, ts_hi=DAY):
    return layer_inputs(seed, tiny_users, TINY.D, TINY.H, TINY.dh, "dense", ts_hi)


def small_attn(seed=1):
    return attn_inputs(seed, small_users, SMALL.H, SMALL.dh, 0.5)


def large_layer(seed=2):
    return layer_inputs(seed, large_users, LARGE.D, LARGE.H, LARGE.dh, "dense")


def large_train_layer(seed=3, min_tokens=262144):
    return layer_inputs(seed, lambda rng: large_users_token_budget(rng, min_tokens), LARGE.D, LARGE.H, LARGE.dh,
                        "cand")
