"""Canary-padded buffers: each tensor handed to the library sits between two
pads of a sentinel byte, checked after the call.  A write outside the tensor's
extent (a ragged tail, a clipped box, a workspace overrun) changes a pad."""
from __future__ import annotations

import math

import torch

SENTINEL = 0xA5
PAD = 4096          # bytes on each side; keeps the allocation's alignment (16 bytes or more)


class Canaries:
    def __init__(self, device):
        self.device = device
        self.bufs = []

    def tensor(self, shape, dtype):
        nbytes = math.prod(shape) * torch.empty(0, dtype=dtype).element_size()
        raw = torch.full((PAD + nbytes + PAD,), SENTINEL, dtype=torch.uint8, device=self.device)
        self.bufs.append((raw, nbytes))
        return raw[PAD:PAD + nbytes].view(dtype).view(*shape)

    def like(self, t):
        return self.tensor(tuple(t.shape), t.dtype)

    def broken(self):
        """Indices of the buffers whose pads changed."""
        bad = []
        for i, (raw, nbytes) in enumerate(self.bufs):
            pads = torch.cat([raw[:PAD], raw[PAD + nbytes:]])
            if not bool((pads == SENTINEL).all()):
                bad.append(i)
        return bad
