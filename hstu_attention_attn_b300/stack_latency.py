"""Forward latency of an HSTU layer stack for ranking requests.

A request is one user of 8 User, 1000 Seq and 64 RealTime tokens followed by
K candidates (the long-history inference shape of MTGR-large: 22 layers at
d_model 1024, 8 heads x 128 — paper-daily deep reading §2), or a batch of such
users.  The stack runs eagerly (one library call per layer, or one call for the
whole stack) and replayed from one captured CUDA Graph; all are timed with CUDA events on the launching stream
after warm-up, and the two outputs are checked to be identical.  Weights are
random (Xavier), inputs N(0, 1), timestamps drawn as in the training batches.

    python -m hstu_attention_attn_b300.stack_latency [--layers 22] [--k 20,50,100,200,500] [--batch 1,64]

Prints one JSON line per (batch, K).
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import synth
from .layer import HstuLayer, HstuStack, device_batch


def _time(fn, iters):
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for _ in range(iters):
        fn()
    stop.record()
    stop.synchronize()
    return start.elapsed_time(stop) / iters


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=22)
    ap.add_argument("--k", default="20,50,100,200,500")
    ap.add_argument("--batch", default="1,64")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--seed", type=int, default=4)
    args = ap.parse_args()
    shape = synth.LARGE
    rng = np.random.default_rng(args.seed)
    layers = []
    for _ in range(args.layers):
        w_uqkv = synth.xavier(rng, shape.D, 4 * shape.H * shape.dh)
        w_o = synth.xavier(rng, shape.H * shape.dh, shape.D)
        gamma, beta = synth.gln_params(rng, shape.D)
        layers.append(HstuLayer(shape.D, shape.H, shape.dh, torch.from_numpy(w_uqkv), torch.from_numpy(w_o),
                                torch.from_numpy(gamma), torch.from_numpy(beta), dtype=torch.bfloat16))
    for nb in (int(v) for v in args.batch.split(",")):
        for K in (int(v) for v in args.k.split(",")):
            batch = synth.make_batch(rng, synth.inference_users(K, nb))
            db = device_batch(batch)
            x = torch.from_numpy(synth.normal(rng, (batch.T, shape.D))).to("cuda", torch.bfloat16)
            stack = HstuStack(layers)
            for _ in range(2):
                y_eager = stack.forward(x, db, native=False)
            y_eager = y_eager.clone()
            layers_ms = _time(lambda: stack.forward(x, db, native=False), args.iters)
            stack.forward(x, db)
            stack_ms = _time(lambda: stack.forward(x, db), args.iters)
            y = stack.capture(x, db)
            for _ in range(2):
                stack.replay()
            graph_ms = _time(stack.replay, args.iters)
            same = bool(torch.equal(y, y_eager))
            print(json.dumps({"metric": "layer stack forward latency", "layers": args.layers, "users": nb,
                              "candidates_per_user": K, "tokens": int(batch.T), "eager_layer_calls_ms": layers_ms,
                              "eager_stack_call_ms": stack_ms, "graph_ms": graph_ms,
                              "graph_speedup_vs_layer_calls": layers_ms / graph_ms, "graph_equals_eager": same,
                              "d_model": shape.D, "n_heads": shape.H, "d_h": shape.dh, "dtype": "bf16"}))


if __name__ == "__main__":
    main()
