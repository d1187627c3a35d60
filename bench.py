#!/usr/bin/env python
"""Benchmark of the MTGR HSTU hot path on B300.

Default workload (the MTGR-large-like training step): users drawn from the
MTGR-large length distribution (8 User tokens, Seq ~ lognormal median 300
clamped to [16, 1000], RealTime ~ U[0, 64], 20 candidates) until the batch
holds >= 262,144 tokens; one HSTU layer at d_model 1024, 8 heads x d_h 128;
a step is the layer forward + backward (Group LayerNorm, UQKV projection +
SiLU, masked jagged attention, LayerNorm(O)*U, output projection + residual,
and all their gradients), with the upstream gradient non-zero only on
candidate rows.  Inputs are synthetic and seeded; weights are Xavier.

Printed metric (one JSON line): useful masked HSTU attention fwd+bwd TFLOP/s
(visible (i, j, head) pairs x 12*d_h FLOP: 4*d_h forward, 8*d_h backward),
timed as the device time of the attention op's kernels inside the timed layer
steps (CUDA events on the launching stream), plus tokens/s/layer of the whole
step.  --impl reference times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "masked HSTU attn fwd+bwd useful TFLOP/s, % BF16 tensor peak; tokens/s/layer"
# DRAM bytes of the dominant kernel per unit of its work, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum, --clock-control none; the
# command is in profiles/).  Each entry names the source file the capture was
# taken on and its SHA-256: a kernel whose source has changed since reports no
# traffic until it is captured again.
TRAFFIC = {
    "attn_bwd": dict(file="hstu_attention_attn_b300/csrc/attn_bwd_sm103.cu",
                     sha256="88dc13bd18d7a5d17d0769befba18209b7c9a7b1f327718687990206bd21ce33",
                     bytes_per_pair=(1942.95e6 + 2135.91e6) / 82381761,
                     note="ncu capture of the 131,297-token training batch (82,381,761 visible pairs, inputs "
                          "larger than L2), scaled by visible pairs; the kernel also writes the dS tiles "
                          "(32 KB per tile pair) that the dQ kernel reads"),
}


def traffic_per_launch(kernel, npairs):
    """(bytes, note) for one launch of `kernel`, or (None, reason)."""
    import hashlib
    t = TRAFFIC.get(kernel)
    if t is None:
        return None, "no ncu capture of this kernel"
    with open(os.path.join(ROOT, t["file"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != t["sha256"]:
            return None, "kernel source changed since its ncu capture"
    return t["bytes_per_pair"] * npairs, t["note"]


ATTN_KERNELS = ("plan_users", "plan_items", "attn_fwd", "gate_fwd", "gate_bwd", "attn_bwd", "attn_bwd_dq")


def rank_totals(sums, maxes, device=None):
    """Whole-job figures from this rank's own: the sum over the ranks of each
    entry of `sums` (work processed) and the maximum over the ranks of each
    entry of `maxes` (times), one all-reduce per non-empty list.  Without a
    process group of more than one rank the values pass through unchanged."""
    import torch
    import torch.distributed as dist
    sums, maxes = [float(v) for v in sums], [float(v) for v in maxes]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return sums, maxes
    out = []
    for vals, op in ((sums, dist.ReduceOp.SUM), (maxes, dist.ReduceOp.MAX)):
        if vals:
            t = torch.tensor(vals, dtype=torch.float64, device=device)
            dist.all_reduce(t, op=op)
            vals = t.tolist()
        out.append(vals)
    return out[0], out[1]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--workload", choices=["large_train", "small_attn"], default="large_train")
    ap.add_argument("--seed", type=int, default=3)
    ap.add_argument("--tokens", type=int, default=262144,
                    help="training-step batch: users are drawn until it holds at least this many tokens")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads (MTGR-small attention, 22-layer stacks, inference sweep)")
    ap.add_argument("--no-ds-store", dest="ds_store", action="store_false",
                    help="lend the attention backward no store for its dS tiles (dQ recomputes S and dP)")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p["bf16_tflops_sustained"], src="measured")
    except Exception:
        return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for nm, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
def attention_useful_flops(npairs, H, dh):
    return dict(fwd=4.0 * dh * npairs * H, bwd=8.0 * dh * npairs * H)


def cpu_baseline(batch, H, dh, budget_s=12.0):
    """fp64 oracle (as it stands) timed on whole users of the same batch: the
    attention op forward + backward; returns useful TFLOP/s and the sample."""
    cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    import oracle
    from hstu_attention_attn_b300 import synth
    rng = np.random.default_rng(0)
    lens = np.diff(batch.offsets)
    order = rng.permutation(len(lens))
    chosen, t_used, flops, pairs_tot = [], 0.0, 0.0, 0
    t_start = time.perf_counter()
    # grow the sample one group of users at a time until the budget is used
    i = 0
    group = max(1, cores)
    while i < len(order) and t_used < budget_s:
        users = [int(b) for b in order[i:i + group]]
        i += group
        rows, offs = [], [0]
        for b in users:
            s0, s1 = int(batch.offsets[b]), int(batch.offsets[b + 1])
            rows.append(np.arange(s0, s1))
            offs.append(offs[-1] + s1 - s0)
        rows = np.concatenate(rows)
        sb = synth.Batch(np.asarray(offs, np.int32), batch.gid[rows], batch.ts[rows])
        T = sb.T
        q, k, v, u, dY = (rng.standard_normal((T, H * dh)) for _ in range(5))
        _, pairs = oracle.visible_counts(sb)
        t0 = time.perf_counter()
        oracle.attn_fwd(sb, H, dh, q, k, v, u)
        oracle.attn_bwd(sb, H, dh, q, k, v, u, dY)
        dt = time.perf_counter() - t0
        t_used += dt
        f = attention_useful_flops(pairs, H, dh)
        flops += f["fwd"] + f["bwd"]
        pairs_tot += pairs
        chosen += users
    return {"value": flops / t_used / 1e12, "unit": "TFLOP/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
            "kind": "oracle",
            "sample": f"{len(chosen)} whole users ({pairs_tot} visible pairs x {H} heads) of the same batch, "
                      f"attention op forward+backward in fp64, {t_used:.1f} s of CPU time",
            "wall_s": time.perf_counter() - t_start}


# ---------------------------------------------------------------------------
def run_reference(args):
    """The fp64 CPU oracle timed on the host cores (bounded sample per step)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from hstu_attention_attn_b300 import synth
    L = synth.large_train_layer(args.seed, args.tokens) if args.workload == "large_train" else None
    if L is None:
        a = synth.small_attn(1)
        batch, H, dh = a.batch, a.H, a.dh
    else:
        batch, H, dh = L.batch, L.H, L.dh
    per_step = 3.0
    vals = []
    for _ in range(args.warmup):
        cpu_baseline(batch, H, dh, budget_s=1.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(batch, H, dh, budget_s=per_step))
    wall = time.perf_counter() - t0
    value = float(np.mean([v["value"] for v in vals]))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args, batch, H, dh),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "kind": "oracle", "cores": vals[0]["cores"],
                             "sample": vals[0]["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def workload_config(args, batch, H, dh, D=None):
    if args.workload == "large_train":
        return {"workload": f"MTGR-large-like HSTU layer training step (fwd+bwd): {batch.B} users, "
                            f"{batch.T} tokens, d_model 1024, {H} heads x d_h {dh}, Seq lognormal median 300 "
                            f"in [16,1000], RealTime U[0,64], 20 candidates, grad on candidates only",
                "tokens": int(batch.T), "users": int(batch.B), "d_model": 1024, "n_heads": H, "d_h": dh,
                "l2": (f"inputs larger than L2 (x and dx_out are {batch.T * 2048 / 2**20:.0f} MiB each)"
                       if batch.T * 2048 > 126 * 2**20 else
                       f"working set larger than L2 (uqkv and silu'(z) are {batch.T * 2 * 4096 * 2 / 2**20:.0f} MiB)"),
                "parallelism": "replicas only",
                "attn_bwd_dq": ("dQ = dS K from the dS tiles the dK/dV kernel stores" if args.ds_store
                                else "dQ kernel recomputes S and dP"),
                "e2e_upstream_gradient": "only the candidate rows of dx' are copied in (the loss is on the "
                                         "candidates; dx' is zero elsewhere and is expanded on the device)"}
    return {"workload": f"MTGR-small-like attention fwd+bwd: {batch.B} users, {batch.T} tokens, {H} heads x d_h {dh}",
            "tokens": int(batch.T), "users": int(batch.B), "n_heads": H, "d_h": dh,
            "l2": "inputs larger than L2", "parallelism": "replicas only"}



# ---------------------------------------------------------------------------
# The other workloads, measured after the headline timed region
# ---------------------------------------------------------------------------
def _event_ms(fn, iters, warmup=3):
    import torch
    for _ in range(warmup):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / iters


def _stack_weights(rng, n_layers, shape):
    from hstu_attention_attn_b300 import synth
    out = []
    for _ in range(n_layers):
        w_uqkv = synth.xavier(rng, shape.D, 4 * shape.H * shape.dh)
        w_o = synth.xavier(rng, shape.H * shape.dh, shape.D)
        gamma, beta = synth.gln_params(rng, shape.D)
        out.append((w_uqkv, w_o, gamma, beta))
    return out


def _stack_graph_ms(weights, dtype, batch, x32, iters, dev):
    """22-layer stack forward replayed from one CUDA Graph: (ms per replay, ms of one eager layer call)."""
    import torch
    from hstu_attention_attn_b300 import synth
    from hstu_attention_attn_b300.layer import HstuLayer, HstuStack, device_batch
    sh = synth.LARGE
    layers = [HstuLayer(sh.D, sh.H, sh.dh, *(torch.from_numpy(w) for w in ws), dtype=dtype, device=dev)
              for ws in weights]
    db = device_batch(batch, dev)
    x = x32.to(dtype)
    stack = HstuStack(layers)
    stack.forward(x, db)
    stack.capture(x, db)
    graph_ms = _event_ms(stack.replay, iters)
    out = torch.empty_like(x)
    layer_ms = _event_ms(lambda: layers[0].forward(x, db, stack._saved, out), iters)
    return graph_ms, layer_ms


def run_extras(dev, pk):
    """MTGR-small-like attention fwd+bwd; the MTGR-large-like 22-layer stack
    forward (128 users); the inference sweep over K candidates at batch 1 and 64
    (22 layers, one user = 8 User + 1000 Seq + 64 RealTime + K candidates).
    Device time by CUDA events on the launching stream, after warm-up."""
    import torch
    from hstu_attention_attn_b300 import mtgr, synth
    from hstu_attention_attn_b300.layer import HstuAttention, device_batch
    out = {}
    # MTGR-small-like attention (64 users, 4 heads x 128), forward + backward
    A = synth.small_attn(1)
    db = device_batch(A.batch, dev)
    cnt = torch.empty(A.batch.T, dtype=torch.int32, device=dev)
    tot = torch.zeros(1, dtype=torch.int64, device=dev)
    mtgr.mtgr_debug_visible_counts(db.offsets, db.gid, db.ts, A.batch.T, cnt, tot)
    pairs = int(tot.item())
    op = HstuAttention(A.H, A.dh, torch.bfloat16, device=dev)
    q, k, v, u = (torch.from_numpy(m).to(dev).to(torch.bfloat16) for m in (A.q, A.k, A.v, A.u))
    dy = torch.randn(A.batch.T, A.H * A.dh, device=dev, dtype=torch.bfloat16,
                     generator=torch.Generator(dev).manual_seed(5))

    def attn_step():
        y, sv = op.forward(q, k, v, u, db)
        op.backward(dy, q, k, v, u, sv, db)
    ms = _event_ms(attn_step, 10)
    fl = attention_useful_flops(pairs, A.H, A.dh)
    out["small_attn"] = {"workload": f"MTGR-small-like attention fwd+bwd: {A.batch.B} users, {A.batch.T} tokens, "
                                     f"{A.H} heads x d_h {A.dh}, bf16",
                         "visible_pairs": pairs, "ms_per_step": ms,
                         "useful_tflops": (fl["fwd"] + fl["bwd"]) / (ms * 1e-3) / 1e12,
                         "frac_of_bf16_peak": (fl["fwd"] + fl["bwd"]) / (ms * 1e-3) / 1e12 / pk["bf16"]}
    del op, q, k, v, u, dy
    # MTGR-large-like 22-layer stack forward, 128 users
    rng = np.random.default_rng(4)
    sh = synth.LARGE
    weights = _stack_weights(rng, 22, sh)
    Lg = synth.large_layer(2)
    x32 = torch.from_numpy(Lg.x).to(dev)
    res = {}
    for name, dt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        g_ms, l_ms = _stack_graph_ms(weights, dt, Lg.batch, x32, 10, dev)
        res[name] = {"stack_ms": g_ms, "stack_tokens_per_s": Lg.batch.T / (g_ms * 1e-3), "layer_ms": l_ms,
                     "tokens_per_s_per_layer": Lg.batch.T / (l_ms * 1e-3)}
    out["large_stack_fwd"] = {"workload": f"MTGR-large-like 22-layer HSTU stack forward (CUDA Graph replay): "
                                          f"{Lg.batch.B} users, {Lg.batch.T} tokens, d_model 1024, 8 heads x 128",
                              **res}
    del x32
    # inference sweep: K candidates, batch 1 and 64 requests, 22 layers
    sweep = []
    for nb in (1, 64):
        for K in (20, 50, 100, 200, 500):
            batch = synth.make_batch(rng, synth.inference_users(K, nb))
            x32 = torch.from_numpy(synth.normal(rng, (batch.T, sh.D))).to(dev)
            row = {"requests": nb, "candidates_per_request": K, "tokens": int(batch.T)}
            for name, dt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
                g_ms, _ = _stack_graph_ms(weights, dt, batch, x32, 10 if nb == 64 else 30, dev)
                row[name] = {"latency_ms": g_ms, "candidates_per_s": nb * K / (g_ms * 1e-3)}
            sweep.append(row)
            del x32
    out["inference_sweep"] = {"workload": "22-layer stack forward per request of 8 User + 1000 Seq + 64 RealTime "
                                          "tokens + K candidates (CUDA Graph replay), d_model 1024, 8 heads x 128",
                              "points": sweep}
    # one request of K = 500 candidates scored in chunks of 100 against its history,
    # encoded once (history pass + 5 chunk passes, one CUDA Graph), against one pass
    from hstu_attention_attn_b300.layer import HstuLayer, HstuStack
    K, chunk = 500, 100
    batch = synth.make_batch(rng, synth.inference_users(K, 1))
    n_hist = batch.T - K
    x = torch.from_numpy(synth.normal(rng, (batch.T, sh.D))).to(dev).to(torch.bfloat16)
    db = device_batch(batch, dev)
    layers = [HstuLayer(sh.D, sh.H, sh.dh, *(torch.from_numpy(w) for w in ws), dtype=torch.bfloat16, device=dev)
              for ws in weights]
    stack = HstuStack(layers)
    stack.score_chunked(x, db.gid, db.ts, n_hist, chunk)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        stack.score_chunked(x, db.gid, db.ts, n_hist, chunk)
    torch.cuda.current_stream(dev).wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        stack.score_chunked(x, db.gid, db.ts, n_hist, chunk)
    chunked_ms = _event_ms(g.replay, 20)
    whole_ms, _ = _stack_graph_ms(weights, torch.bfloat16, batch, x.float(), 20, dev)
    # chunks without the cache: the whole stack on history + one chunk, once per chunk
    b1 = synth.make_batch(rng, synth.inference_users(chunk, 1))
    x1 = torch.from_numpy(synth.normal(rng, (b1.T, sh.D))).to(dev)
    per_chunk_ms, _ = _stack_graph_ms(weights, torch.bfloat16, b1, x1, 20, dev)
    out["chunked_scoring"] = {"workload": f"one request (8 User + 1000 Seq + 64 RealTime + {K} candidates), 22 layers, "
                                          f"d_model 1024, bf16: history encoded once, candidates in chunks of {chunk}",
                              "chunk": chunk, "chunked_ms": chunked_ms, "one_pass_ms": whole_ms,
                              "chunks_recomputing_history_ms": per_chunk_ms * ((K + chunk - 1) // chunk),
                              "candidates_per_s_chunked": K / (chunked_ms * 1e-3)}
    return out

# ---------------------------------------------------------------------------
def run_mine(args):
    import torch
    import torch.distributed as dist

    from hstu_attention_attn_b300 import mtgr, synth
    from hstu_attention_attn_b300.layer import HstuAttention, HstuLayer, device_batch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    mtgr.lib()
    pk = peaks()

    # ---- inputs (seeded, synthetic; each replica draws its own batch) ----
    if args.workload == "large_train":
        L = synth.large_train_layer(args.seed + rank, args.tokens)
        batch, H, dh, D = L.batch, L.H, L.dh, L.D
    else:
        A = synth.small_attn(1 + rank)
        batch, H, dh, D = A.batch, A.H, A.dh, None
    T = batch.T
    db = device_batch(batch, dev)
    cnt = torch.empty(T, dtype=torch.int32, device=dev)
    tot = torch.zeros(1, dtype=torch.int64, device=dev)
    mtgr.mtgr_debug_visible_counts(db.offsets, db.gid, db.ts, T, cnt, tot)
    npairs = int(tot.item())
    uf = attention_useful_flops(npairs, H, dh)

    bf = torch.bfloat16
    if args.workload == "large_train":
        layer = HstuLayer(D, H, dh, torch.from_numpy(L.w_uqkv), torch.from_numpy(L.w_o), torch.from_numpy(L.gamma),
                          torch.from_numpy(L.beta), dtype=bf, device=dev, ds_store=args.ds_store)
        x_h = torch.from_numpy(L.x).to(bf).pin_memory()
        dxo_h = torch.from_numpy(L.dx_out).to(bf).pin_memory()
        x = x_h.to(dev)
        dxo = dxo_h.to(dev)
        saved = layer.alloc_saved(T)
        x_out = torch.empty_like(x)
        dx = torch.empty_like(x)
        f = lambda *s: torch.empty(*s, dtype=torch.float32, device=dev)
        grads = dict(dw_uqkv=f(D, 4 * H * dh), dw_o=f(H * dh, D), dgamma=f(4, D), dbeta=f(4, D))

        def step():
            layer.forward(x, db, saved, x_out)
            layer.backward(x, saved, dxo, db, dx, grads)
    else:
        op = HstuAttention(H, dh, bf, device=dev, ds_store=args.ds_store)
        q, k, v, u = (torch.from_numpy(m).to(dev).to(bf) for m in (A.q, A.k, A.v, A.u))
        dy = torch.randn(T, H * dh, device=dev, dtype=bf, generator=torch.Generator(dev).manual_seed(5))

        def step():
            y, sv = op.forward(q, k, v, u, db)
            op.backward(dy, q, k, v, u, sv, db)

    # ---- warm-up, then the timed region ----
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    mtgr.mtgr_trace_reset()
    mtgr.mtgr_trace_enable(True)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    mtgr.mtgr_trace_enable(False)
    ms_total = e0.elapsed_time(e1)
    cl = clocks.stop()
    trace = mtgr.mtgr_trace_report()
    K = args.steps
    attn_ms = sum(trace.get(k, (0.0, 0))[0] for k in ATTN_KERNELS) / K
    attn_core_ms = sum(trace.get(k, (0, 0))[0] for k in ("attn_fwd", "attn_bwd", "attn_bwd_dq")) / K
    launches = sum(c for name, (_, c) in trace.items())
    # whole job: work and launches summed over the ranks (each drew its own batch), times of the slowest rank
    (total_flops, flash_flops, total_tokens, total_pairs, launches), (ms_total, attn_ms, attn_core_ms) = rank_totals(
        [uf["fwd"] + uf["bwd"], uf["fwd"] + uf["bwd"] * 10.0 / 8.0, T, npairs, launches],
        [ms_total, attn_ms, attn_core_ms], dev)
    ms_step = ms_total / K
    value = total_flops / (attn_ms * 1e-3) / 1e12

    # ---- roofline of the dominant kernel ----
    dom = max(trace.items(), key=lambda kv: kv[1][0])
    dname, (dms, dcnt) = dom
    per_launch_ms = dms / dcnt
    algo = None
    if dname == "attn_bwd":    # dK/dV kernel: dV, dA = dO·Vᵀ and dK (6·d_h of the 8·d_h per pair)
        algo = dict(bound="tensor", flops=uf["bwd"] * 0.75)
    elif dname == "attn_bwd_dq":  # dQ kernel: dQ = dS·K (2·d_h per pair)
        algo = dict(bound="tensor", flops=uf["bwd"] * 0.25)
    elif dname == "attn_fwd":
        algo = dict(bound="tensor", flops=uf["fwd"])
    elif dname.startswith("gemm") and args.workload == "large_train":
        HD, N4 = H * dh, 4 * H * dh
        shapes = {"gemm_uqkv": (T, N4, D), "gemm_out": (T, D, HD), "gemm_dY": (T, HD, D), "gemm_dWo": (HD, D, T),
                  "gemm_dWuqkv": (D, N4, T), "gemm_dxn": (T, D, N4)}
        M, N, Kd = shapes[dname]
        algo = dict(bound="tensor", flops=2.0 * M * N * Kd)
    roof = None
    if algo:
        ach = algo["flops"] / (per_launch_ms * 1e-3) / 1e12
        traffic, tnote = traffic_per_launch(dname, npairs)
        roof = {"kernel": dname, "bound": "tensor", "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16"], "frac_sustained": ach / pk["bf16_sus"],
                "traffic": traffic, "traffic_note": tnote,
                "peak_note": f"{pk['src']} dense bf16 burst (the bench runs at the maximum SM clock; the sustained "
                             f"figure, {pk['bf16_sus']} TF/s, was measured at a lower clock under the power cap); "
                             "f16 operands run at the same tensor rate"}

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e and args.workload == "large_train":
        from hstu_attention_attn_b300.layer import DeviceBatch
        # The step's inputs as a training loader ships them: x, and one packed
        # block (one copy, as the pages do for serving features) with the
        # metadata, the rows that carry a loss (the candidates) and their
        # upstream gradient; the library expands that gradient to [T, D] on the
        # device (dx' is zero on every other row).
        rows_np = np.nonzero(np.any(L.dx_out != 0, axis=1))[0].astype(np.int32)
        n_rows = len(rows_np)
        dxc = dxo_h[torch.from_numpy(rows_np).long()].contiguous()
        pieces = [np.ascontiguousarray(batch.offsets, np.int32).view(np.uint8),
                  np.ascontiguousarray(batch.gid, np.uint8),
                  np.ascontiguousarray(batch.ts, np.int64).view(np.uint8),
                  rows_np.view(np.uint8), dxc.view(torch.int16).numpy().reshape(-1).view(np.uint8)]
        starts, nbytes = [], 0
        for pc in pieces:
            starts.append(nbytes)
            nbytes += (pc.size + 15) // 16 * 16
        blk_h = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
        blk_np = blk_h.numpy()
        for st, pc in zip(starts, pieces):
            blk_np[st:st + pc.size] = pc
        g_h = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in grads.items()}
        h2d = x_h.numel() * 2 + nbytes
        d2h = sum(t.numel() * t.element_size() for t in g_h.values())

        def unpack(blk):
            o = starts
            db_ = DeviceBatch(blk[o[0]:o[0] + 4 * (batch.B + 1)].view(torch.int32), blk[o[1]:o[1] + T],
                              blk[o[2]:o[2] + 8 * T].view(torch.int64), batch.B, T,
                              np.ascontiguousarray(batch.offsets, dtype=np.int32))
            rows_ = blk[o[3]:o[3] + 4 * n_rows].view(torch.int32)
            dxc_ = blk[o[4]:o[4] + 2 * n_rows * D].view(torch.bfloat16).view(n_rows, D)
            return db_, rows_, dxc_

        # Input prefetch as a training loop does it: two device sets of inputs
        # and weight gradients; a copy stream brings step k+1's inputs in while
        # step k computes, then reads step k's weight gradients out.  Every
        # step's copies are inside the timed region (the first input copy is
        # issued in it, and nothing is copied for a step after the last).
        comp_s = torch.cuda.current_stream(dev)
        copy_s = torch.cuda.Stream(dev)
        xs, dxos = [x, torch.empty_like(x)], [dxo, torch.empty_like(dxo)]
        blks = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        packed = [unpack(bk) for bk in blks]
        gs = [grads, {n: torch.empty_like(t) for n, t in grads.items()}]
        ghs = [g_h, {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in grads.items()}]
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in_ready", "in_free", "out_ready", "out_free")}
        for k in ("in_free", "out_free"):
            for e in ev[k]:
                e.record(comp_s)

        def copy_in(b):
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(ev["in_free"][b])
                xs[b].copy_(x_h, non_blocking=True)
                blks[b].copy_(blk_h, non_blocking=True)
                ev["in_ready"][b].record(copy_s)

        def compute_and_d2h(b):
            comp_s.wait_event(ev["in_ready"][b])
            comp_s.wait_event(ev["out_free"][b])
            db_b, rows_b, dxc_b = packed[b]
            mtgr.mtgr_expand_rows(dxc_b, rows_b, dxos[b])
            layer.forward(xs[b], db_b, saved, x_out)
            layer.backward(xs[b], saved, dxos[b], db_b, dx, gs[b])
            ev["in_free"][b].record(comp_s)
            ev["out_ready"][b].record(comp_s)
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(ev["out_ready"][b])
                for n, t in gs[b].items():
                    ghs[b][n].copy_(t, non_blocking=True)
                ev["out_free"][b].record(copy_s)

        def run(steps):
            copy_in(0)
            for k in range(steps):
                if k + 1 < steps:
                    copy_in((k + 1) & 1)
                compute_and_d2h(k & 1)
        run(2)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        run(K)
        torch.cuda.synchronize()
        e2e_ms = rank_totals([], [(time.perf_counter() - t0) * 1e3 / K], dev)[1][0]
        e2e = {"value": total_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
               "note": "whole layer step through the public API incl. pinned-host copies in (x, and one packed block "
                       "of metadata and the candidate rows' upstream gradient, expanded on the device) and of the "
                       "weight gradients out; the next step's inputs are copied in on a second stream while the "
                       "current step computes"}

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 (f16 attention operands, fp32 accumulate)", "data": "synthetic",
            "config": workload_config(args, batch, H, dh, D),
            "pct_bf16_peak": value / pk["bf16"] * 100.0,
            "tokens_per_s_per_layer": total_tokens / (ms_step * 1e-3),
            "attention": {"visible_pairs": int(total_pairs), "useful_gflop_per_step": total_flops / 1e9,
                          "op_ms_per_step": attn_ms, "core_kernels_ms_per_step": attn_core_ms,
                          "core_tflops": total_flops / (attn_core_ms * 1e-3) / 1e12,
                          # FlashAttention-style count: the backward's recomputed S counted too (10 d_h per pair)
                          "flash_count_tflops": flash_flops / (attn_ms * 1e-3) / 1e12},
            "kernels_ms_per_step": {k: round(v[0] / K, 4) for k, v in sorted(trace.items(), key=lambda kv: -kv[1][0])},
            "gpu_launches": int(launches), "roofline": roof, "clocks": cl, "e2e": e2e}
    if rank == 0 and not args.no_extras and args.workload == "large_train":
        del layer, saved, x_out, dx, grads
        torch.cuda.empty_cache()
        line["other_workloads"] = run_extras(dev, pk)
    if rank == 0 and not args.no_cpu:
        try:
            line["cpu_baseline"] = {k: v for k, v in cpu_baseline(batch, H, dh).items() if k != "wall_s"}
        except Exception as ex:  # the CPU leg must not hide the GPU result
            line["cpu_baseline"] = {"error": str(ex)}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_mine(args)


if __name__ == "__main__":
    main()
