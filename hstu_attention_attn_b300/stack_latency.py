"""Forward latency and precision of an HSTU layer stack for ranking requests.

A request is one user of 8 User, 1000 Seq and 64 RealTime tokens followed by
K candidates (the long-history inference shape of MTGR-large: 22 layers at
d_model 1024, 8 heads x 128 — paper-daily deep reading §2), or a batch of such
users.  For each 16-bit dtype (bf16; f16, the pages' serving precision) the
stack runs eagerly (one library call per layer, or one call for the whole
stack) and replayed from one captured CUDA Graph; all are timed with CUDA
events on the launching stream after warm-up, and the outputs are checked to
be identical.  For one-user requests the same stack also runs in fp32 (the
library's CUDA-core path), and every candidate is scored by a fixed random
linear head with a sigmoid on its last-layer row: the report gives how far the
16-bit scores lie from the fp32 ones (the pages quote FP16 vs FP32 score
deviations within 0.006, paper-daily deep reading §3).  Weights are random
(Xavier), inputs N(0, 1), timestamps drawn as in the training batches.

    python -m hstu_attention_attn_b300.stack_latency [--layers 22] [--k 20,500] [--batch 1,64] [--dtypes bf16,f16]

Prints one JSON line per measurement.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import synth
from .layer import HstuLayer, HstuStack, device_batch

DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _time(fn, iters):
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for _ in range(iters):
        fn()
    stop.record()
    stop.synchronize()
    return start.elapsed_time(stop) / iters


def _layers(weights, dtype):
    return [HstuLayer(synth.LARGE.D, synth.LARGE.H, synth.LARGE.dh, *(torch.from_numpy(w) for w in ws), dtype=dtype)
            for ws in weights]


def _scores(y, rows, head):
    return torch.sigmoid(y[rows].double() @ head)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=22)
    ap.add_argument("--k", default="20,500")
    ap.add_argument("--batch", default="1,64")
    ap.add_argument("--dtypes", default="bf16,f16")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--seed", type=int, default=4)
    args = ap.parse_args()
    shape = synth.LARGE
    rng = np.random.default_rng(args.seed)
    weights = []
    for _ in range(args.layers):
        w_uqkv = synth.xavier(rng, shape.D, 4 * shape.H * shape.dh)
        w_o = synth.xavier(rng, shape.H * shape.dh, shape.D)
        gamma, beta = synth.gln_params(rng, shape.D)
        weights.append((w_uqkv, w_o, gamma, beta))
    head = torch.from_numpy(rng.standard_normal(shape.D) / np.sqrt(shape.D)).cuda()
    stacks = {name: _layers(weights, DTYPES[name]) for name in args.dtypes.split(",")}
    for nb in (int(v) for v in args.batch.split(",")):
        for K in (int(v) for v in args.k.split(",")):
            batch = synth.make_batch(rng, synth.inference_users(K, nb))
            db = device_batch(batch)
            x32 = torch.from_numpy(synth.normal(rng, (batch.T, shape.D))).cuda()
            rows = torch.from_numpy(np.nonzero(batch.gid == 3)[0]).cuda()
            ref = None
            if nb == 1:  # fp32 scores of the same request
                y32 = HstuStack(_layers(weights, torch.float32)).forward(x32, db)
                ref = _scores(y32, rows, head)
            for name, layers in stacks.items():
                x = x32.to(DTYPES[name])
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
                line = {"metric": "layer stack forward latency", "dtype": name, "layers": args.layers, "users": nb,
                        "candidates_per_user": K, "tokens": int(batch.T), "eager_layer_calls_ms": layers_ms,
                        "eager_stack_call_ms": stack_ms, "graph_ms": graph_ms,
                        "graph_speedup_vs_layer_calls": layers_ms / graph_ms,
                        "graph_equals_eager": bool(torch.equal(y, y_eager)), "d_model": shape.D,
                        "n_heads": shape.H, "d_h": shape.dh}
                if ref is not None:
                    dev = (_scores(y, rows, head) - ref).abs()
                    line.update(score_dev_vs_f32_max=float(dev.max()), score_dev_vs_f32_mean=float(dev.mean()))
                print(json.dumps(line))


if __name__ == "__main__":
    main()
