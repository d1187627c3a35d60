"""User-facing helpers around the C ABI: device batches, the attention op and
one HSTU layer, with buffers allocated through torch (device memory only).

Every computation runs in libmtgr.so; this module allocates outputs and
workspace and forwards pointers (see ``mtgr.py``).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import mtgr


@dataclass
class DeviceBatch:
    offsets: torch.Tensor   # int32 [B+1]
    gid: torch.Tensor       # uint8 [T]
    ts: torch.Tensor        # int64 [T]
    B: int
    T: int
    offsets_host: np.ndarray | None = None  # the same offsets in host memory (sizes the dS tile store)


def device_batch(batch, device="cuda", pin=False) -> DeviceBatch:
    """Copy a host batch (offsets / gid / ts numpy arrays) to the device."""
    def mk(a, dt):
        t = torch.from_numpy(np.ascontiguousarray(a)).to(dt)
        if pin:
            t = t.pin_memory()
        return t.to(device, non_blocking=pin)
    return DeviceBatch(mk(batch.offsets, torch.int32), mk(batch.gid, torch.uint8), mk(batch.ts, torch.int64),
                       len(batch.offsets) - 1, int(batch.offsets[-1]),
                       np.ascontiguousarray(batch.offsets, dtype=np.int32))


def ds_store_bytes(db: DeviceBatch, n_heads, d_h, dtype) -> int:
    """Workspace bytes beyond the required size with which the bf16 backward
    keeps its dS tiles and forms dQ from them (0 without host offsets)."""
    if db.offsets_host is None or dtype != torch.bfloat16:
        return 0
    return mtgr.mtgr_attn_ds_store_size(db.offsets_host, n_heads, d_h, mtgr.MTGR_BF16)


def _dt(dtype):
    return {torch.bfloat16: mtgr.MTGR_BF16, torch.float16: mtgr.MTGR_F16}.get(dtype, mtgr.MTGR_F32)


def workspace(nbytes, device="cuda"):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class HstuAttention:
    """Y = LayerNorm(A·V) ⊙ U with A = M ⊙ silu(QKᵀ/sqrt(d_h)) / n_u (jagged, per head)."""

    def __init__(self, n_heads, d_h, dtype=torch.bfloat16, eps=1e-5, device="cuda", ds_store=True):
        self.H, self.dh, self.dtype, self.eps, self.device = n_heads, d_h, dtype, eps, device
        # lend the backward a store for its dS tiles (ds_store_bytes more workspace):
        # dQ then needs one product per tile pair instead of three
        self.ds_store = ds_store
        self._ws = None

    def _workspace(self, db):
        n = mtgr.mtgr_attn_workspace_size(db.B, db.T, self.H, self.dh, _dt(self.dtype))
        if self.ds_store:
            n += ds_store_bytes(db, self.H, self.dh, self.dtype)
        if self._ws is None or self._ws.numel() < n:
            self._ws = workspace(n, self.device)
        return self._ws

    def device_status(self):
        """MTGR_STATUS_* bits the last forward or backward left in its status
        word (0: every bounded wait completed).  Waits for the device."""
        return 0 if self._ws is None else int(self._ws[:4].view(torch.int32).item())

    def forward(self, q, k, v, u, db: DeviceBatch, ld=None):
        T, HD = db.T, self.H * self.dh
        ld = ld if ld is not None else q.stride(0)
        y = torch.empty(T, HD, dtype=self.dtype, device=self.device)
        # O before the gate: f16 in the bf16 path, fp32 in the fp32 path
        o = torch.empty(T, HD, dtype=torch.float16 if self.dtype == torch.bfloat16 else torch.float32,
                        device=self.device)
        mean = torch.empty(T, dtype=torch.float32, device=self.device)
        rstd = torch.empty(T, dtype=torch.float32, device=self.device)
        mtgr.mtgr_hstu_attn_fwd(q, k, v, u, ld, db.offsets, db.gid, db.ts, T, self.H, self.dh, self.eps, y, o,
                                mean, rstd, self._workspace(db))
        return y, (o, mean, rstd)

    def backward(self, dy, q, k, v, u, saved, db: DeviceBatch, ld=None, dsilu_uqkv=None, grads=None):
        T, HD = db.T, self.H * self.dh
        ld = ld if ld is not None else q.stride(0)
        o, mean, rstd = saved
        if grads is None:
            g = torch.empty(T, 4 * HD, dtype=self.dtype, device=self.device)
            du, dq, dk, dv = g[:, :HD], g[:, HD:2 * HD], g[:, 2 * HD:3 * HD], g[:, 3 * HD:]
        else:
            dq, dk, dv, du = grads
        mtgr.mtgr_hstu_attn_bwd(dy, q, k, v, u, ld, o, mean, rstd, db.offsets, db.gid, db.ts, T, self.H, self.dh,
                                dq, dk, dv, du, dq.stride(0), dsilu_uqkv, self._workspace(db))
        return dq, dk, dv, du


class HstuLayer:
    """One HSTU layer: x' = x + (LN(attn(silu(GLN(x) W_uqkv))) ⊙ U) W_o, forward and backward."""

    def __init__(self, d_model, n_heads, d_h, w_uqkv, w_o, gamma, beta, dtype=torch.bfloat16, eps_gln=1e-5,
                 eps_ln=1e-5, device="cuda", ds_store=True):
        self.D, self.H, self.dh, self.dtype, self.device = d_model, n_heads, d_h, dtype, device
        self.ds_store = ds_store  # as HstuAttention.ds_store
        to = dict(device=device)
        self.w_uqkv = torch.as_tensor(w_uqkv).to(dtype=dtype, **to).contiguous()
        self.w_o = torch.as_tensor(w_o).to(dtype=dtype, **to).contiguous()
        self.gamma = torch.as_tensor(gamma).to(dtype=torch.float32, **to).contiguous()
        self.beta = torch.as_tensor(beta).to(dtype=torch.float32, **to).contiguous()
        self.weights = mtgr.make_weights(d_model, n_heads, d_h, self.w_uqkv, self.w_o, self.gamma, self.beta,
                                         eps_gln, eps_ln)
        self._ws = None
        self._w16 = None

    def keep_f16_weights(self):
        """bf16 layer with fixed weights (inference): make f16 copies of W_uqkv
        and W_o once, which every later call reads instead of converting them
        again.  Call again after changing the weights (the copies are
        rewritten in place, so a captured CUDA Graph reads the new ones);
        drop_f16_weights() returns to converting on every call."""
        if self.dtype != torch.bfloat16:
            return
        if self._w16 is None:  # refreshed in place afterwards, so captured graphs stay valid
            self._w16 = (torch.empty_like(self.w_uqkv, dtype=torch.float16),
                         torch.empty_like(self.w_o, dtype=torch.float16))
        self.weights.w_uqkv_f16 = self.weights.w_o_f16 = None
        mtgr.mtgr_layer_weights_to_f16(self.weights, *self._w16)
        self.weights.w_uqkv_f16, self.weights.w_o_f16 = (t.data_ptr() for t in self._w16)

    def drop_f16_weights(self):
        self.weights.w_uqkv_f16 = self.weights.w_o_f16 = None
        self._w16 = None

    def _workspace(self, db, bwd=True):
        n = mtgr.mtgr_layer_workspace_size(db.B, db.T, self.D, self.H, self.dh, _dt(self.dtype))
        if bwd and self.ds_store:
            n += ds_store_bytes(db, self.H, self.dh, self.dtype)
        if self._ws is None or self._ws.numel() < n:
            self._ws = workspace(n, self.device)
        return self._ws

    def alloc_saved(self, T):
        """Buffers the forward saves for the backward.  The bf16 layer keeps its
        activations between steps in f16 (xn, silu'(z), [U|Q|K|V], O, y);
        the fp32 layer in fp32."""
        HD = self.H * self.dh
        a16 = torch.float16 if self.dtype == torch.bfloat16 else self.dtype
        e = lambda *s: torch.empty(*s, dtype=a16, device=self.device)
        f = lambda *s: torch.empty(*s, dtype=torch.float32, device=self.device)
        return dict(xn=e(T, self.D), dsilu=e(T, 4 * HD), uqkv=e(T, 4 * HD), o=e(T, HD), y=e(T, HD),
                    gln_mean=f(T), gln_rstd=f(T), ln_mean=f(T), ln_rstd=f(T))

    def forward(self, x, db: DeviceBatch, saved=None, x_out=None):
        saved = saved if saved is not None else self.alloc_saved(db.T)
        x_out = x_out if x_out is not None else torch.empty_like(x)
        mtgr.mtgr_hstu_layer_fwd(self.weights, x, x_out, mtgr.make_saved(saved), db.offsets, db.gid, db.ts, db.T,
                                 self._workspace(db))
        return x_out, saved

    def backward(self, x, saved, dx_out, db: DeviceBatch, dx=None, grads=None):
        HD = self.H * self.dh
        dx = dx if dx is not None else torch.empty_like(x)
        if grads is None:
            f = lambda *s: torch.empty(*s, dtype=torch.float32, device=self.device)
            grads = dict(dw_uqkv=f(self.D, 4 * HD), dw_o=f(HD, self.D), dgamma=f(4, self.D), dbeta=f(4, self.D))
        mtgr.mtgr_hstu_layer_bwd(self.weights, x, mtgr.make_saved(saved), dx_out, dx, mtgr.make_grads(grads),
                                 db.offsets, db.gid, db.ts, db.T, self._workspace(db))
        return dx, grads


class HstuStack:
    """A stack of HSTU layers run forward for ranking (22 layers at d_model 1024
    in paper-daily deep reading §2), eagerly or replayed from one captured CUDA
    Graph (the pages' inference path uses CUDA Graphs, paper-daily
    "计算量涨了 65 倍…").

    All layers share two activation buffers (layer l reads one and writes the
    other), one set of saved-state buffers (inference keeps nothing between
    layers) and one workspace, so after the first run nothing is allocated and
    the whole stack can be captured."""

    def __init__(self, layers, keep_f16_weights=True):
        """keep_f16_weights: bf16 layers keep f16 copies of their weights
        (HstuLayer.keep_f16_weights), so a forward pass converts nothing."""
        self.layers = list(layers)
        self._key = None
        self._graph = None
        if keep_f16_weights:
            for layer in self.layers:
                layer.keep_f16_weights()

    def _prepare(self, x, db):
        key = (db.B, db.T, x.dtype, x.device)
        if self._key == key:
            return
        l0 = self.layers[0]
        self._act = [torch.empty_like(x), torch.empty_like(x)]
        self._saved = l0.alloc_saved(db.T)
        ws = l0._workspace(db, bwd=False)
        for layer in self.layers:
            layer._ws = ws
        self._key, self._graph = key, None

    def forward(self, x, db: DeviceBatch, outs=None, native=True):
        """Run every layer on x; returns the last output (one of the stack's own
        buffers).  By default the whole stack is one library call
        (mtgr_hstu_stack_fwd: the attention work lists are built once); with
        native=False, or when `outs` is a list (each layer's output is then
        appended to it as a copy), the layers are called one by one."""
        self._prepare(x, db)
        if native and outs is None:
            mtgr.mtgr_hstu_stack_fwd([l.weights for l in self.layers], x, self._act[0], self._act[1],
                                     mtgr.make_saved(self._saved), db.offsets, db.gid, db.ts, db.T,
                                     self.layers[0]._ws)
            return self._act[0]
        h = x
        for i, layer in enumerate(self.layers):
            o = self._act[i & 1]
            layer.forward(h, db, saved=self._saved, x_out=o)
            if outs is not None:
                outs.append(o.clone())
            h = o
        return h

    def score_chunked(self, x, gid, ts, n_hist, chunk):
        """One ranking request scored in chunks of candidates with its history
        encoded once: x [n_hist + n_cand, D] holds the request's rows (history
        first), gid / ts its device metadata.  The history rows run through the
        stack once (each layer's [U|Q|K|V] of the history kept in a cache); then
        every chunk of `chunk` candidates runs through the stack against that
        cache.  Returns the candidates' last-layer rows [n_cand, D], equal to
        those of the whole request run at once."""
        l0 = self.layers[0]
        T, D = x.shape
        n_cand = T - n_hist
        H, dh = l0.H, l0.dh
        dev = x.device
        cache = torch.empty(max(mtgr.mtgr_stack_cache_size(len(self.layers), n_hist, chunk, D, H, dh), 256),
                            dtype=torch.uint8, device=dev)
        ws = workspace(mtgr.mtgr_stack_chunk_workspace_size(n_hist, chunk, D, H, dh, _dt(x.dtype)), dev)
        half = (n_hist * D * x.element_size() + 255) // 256 * 256
        act = torch.empty(2 * half // x.element_size() + 8, dtype=x.dtype, device=dev)
        weights = [l.weights for l in self.layers]
        mtgr.mtgr_hstu_stack_hist_fwd(weights, x[:n_hist], act, cache, chunk, gid, ts, n_hist, n_cand, ws)
        out = torch.empty(n_cand, D, dtype=x.dtype, device=dev)
        tmp = torch.empty(chunk, D, dtype=x.dtype, device=dev)
        for c0 in range(0, n_cand, chunk):
            c = min(chunk, n_cand - c0)
            mtgr.mtgr_hstu_stack_cand_fwd(weights, x[n_hist + c0:n_hist + c0 + c], out[c0:c0 + c], tmp[:c], cache,
                                          chunk, gid, ts, n_hist, n_cand, c0, ws)
        return out

    def capture(self, x, db: DeviceBatch):
        """Capture the stack's forward on x (a static buffer the caller refills
        between replays) and db; returns the static output buffer."""
        self._prepare(x, db)
        side = torch.cuda.Stream(device=x.device)
        side.wait_stream(torch.cuda.current_stream(x.device))
        with torch.cuda.stream(side):  # warm-up outside the capture
            self.forward(x, db)
        torch.cuda.current_stream(x.device).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            y = self.forward(x, db)
        self._graph, self._y = g, y
        return y

    def replay(self):
        """Replay the captured forward; returns the static output buffer."""
        if self._graph is None:
            raise RuntimeError("HstuStack.replay before capture")
        self._graph.replay()
        return self._y
