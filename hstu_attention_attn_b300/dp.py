"""Data parallelism across the GPUs of one node (one process per GPU).

A training step's users are independent, so a step shards by user: each rank
takes a contiguous, token-balanced share of the users (mtgr_token_balanced_split,
zzxanthony.github.io "MTGR：工业级生成式推荐框架" §11.3 "Dynamic batch size
做负载均衡") and runs the layer on its own rows with no exchange.  The only
exchange is the weight-gradient all-reduce: a rank whose loss is the mean over
its own users weights its gradients by its share of the users, so that the sum
over ranks is the gradient of the mean over the whole step (the pages weight
by each GPU's batch size for the same reason).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import mtgr


def rank_users(tokens_per_user, world):
    """Token-balanced contiguous split: returns (rank_first [world+1],
    rank_tokens [world], grad_weight [world]) as numpy arrays."""
    return mtgr.mtgr_token_balanced_split(np.asarray(tokens_per_user, np.int64), world)


def user_rows(offsets, first_user, end_user):
    """Rows and rebased offsets of users first_user .. end_user-1 of a batch:
    returns (row0, row1, offsets[first_user .. end_user] - row0)."""
    offsets = np.asarray(offsets, np.int64)
    row0, row1 = int(offsets[first_user]), int(offsets[end_user])
    return row0, row1, (offsets[first_user:end_user + 1] - row0).astype(np.int32)


def allreduce_weighted(grads, weight, group=None):
    """grads: dict of tensors holding this rank's gradients of its mean loss.
    In place: grads <- sum over ranks of weight_r * grads_r."""
    for t in grads.values():
        t.mul_(weight)
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return grads
