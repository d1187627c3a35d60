"""Thin Python binding of libmtgr.so (the C ABI declared in include/mtgr.h).

Argument marshalling only: every function has the same name as its C entry
point, takes torch tensors (device memory owned by the caller) and passes their
data pointers and the current CUDA stream through.  All compute runs in the
library's CUDA kernels.  There is no fallback: if libmtgr.so cannot be loaded,
``lib()`` raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmtgr.so")

MTGR_F32, MTGR_BF16, MTGR_F16 = 0, 1, 2
MTGR_OK, MTGR_ERR_INVALID_ARG, MTGR_ERR_UNSUPPORTED = 0, -1, -4
STATUS_BAD_OFFSETS, STATUS_BAD_GROUP_ORDER, STATUS_BAD_GROUP_ID, STATUS_TIMEOUT = 1, 2, 4, 8

_lib = None


class MtgrError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


class LayerWeights(C.Structure):
    _fields_ = [("d_model", C.c_int32), ("n_heads", C.c_int32), ("d_h", C.c_int32),
                ("w_uqkv", C.c_void_p), ("w_o", C.c_void_p), ("gamma", C.c_void_p), ("beta", C.c_void_p),
                ("eps_gln", C.c_float), ("eps_ln", C.c_float), ("w_uqkv_f16", C.c_void_p), ("w_o_f16", C.c_void_p)]


class LayerSaved(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("xn", "dsilu", "uqkv", "o", "y", "gln_mean", "gln_rstd",
                                          "ln_mean", "ln_rstd")]


class LayerGrads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("dw_uqkv", "dw_o", "dgamma", "dbeta")]


EXPORTS = {
    # name: (restype, argtypes)
    "mtgr_last_error": (C.c_char_p, []),
    "mtgr_version": (C.c_int, []),
    "mtgr_trace_enable": (None, [C.c_int]),
    "mtgr_trace_reset": (None, []),
    "mtgr_trace_report": (C.c_int, [C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]),
    "mtgr_validate_batch": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p]),
    "mtgr_debug_visible_counts": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int64,
                                            C.c_void_p, C.c_void_p, C.c_void_p]),
    "mtgr_group_layernorm_fwd": (C.c_int, [C.c_void_p] * 7 + [C.c_int64, C.c_int32, C.c_float, C.c_int,
                                                               C.c_void_p]),
    "mtgr_group_layernorm_bwd_workspace_size": (C.c_size_t, [C.c_int64, C.c_int32]),
    "mtgr_group_layernorm_bwd": (C.c_int, [C.c_void_p] * 10 + [C.c_int64, C.c_int32, C.c_int, C.c_void_p,
                                                                C.c_size_t, C.c_void_p]),
    "mtgr_group_layernorm_bwd_noalloc": (C.c_int, [C.c_void_p] * 10 + [C.c_int64, C.c_int32, C.c_int, C.c_void_p]),
    "mtgr_debug_wait_timeout": (C.c_int, [C.c_void_p, C.c_void_p]),
    "mtgr_debug_plan_counts": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "mtgr_expand_rows": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int32, C.c_int,
                                   C.c_void_p]),
    "mtgr_stochastic_length": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_int32] + [C.c_void_p] * 4),
    "mtgr_token_balanced_split": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32] + [C.c_void_p] * 3),
    "mtgr_attn_workspace_size": (C.c_size_t, [C.c_int32, C.c_int64, C.c_int32, C.c_int32, C.c_int]),
    "mtgr_attn_ds_store_size": (C.c_size_t, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int]),
    "mtgr_hstu_attn_fwd": (C.c_int, [C.c_void_p] * 4 + [C.c_int64, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p,
                                                         C.c_int64, C.c_int32, C.c_int32, C.c_float]
                           + [C.c_void_p] * 4 + [C.c_int, C.c_void_p, C.c_size_t, C.c_void_p]),
    "mtgr_hstu_attn_bwd": (C.c_int, [C.c_void_p] * 5 + [C.c_int64] + [C.c_void_p] * 3
                           + [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int64, C.c_int32, C.c_int32]
                           + [C.c_void_p] * 4 + [C.c_int64, C.c_void_p, C.c_int, C.c_void_p, C.c_size_t,
                                                 C.c_void_p]),
    "mtgr_layer_workspace_size": (C.c_size_t, [C.c_int32, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int]),
    "mtgr_layer_weights_to_f16": (C.c_int, [C.POINTER(LayerWeights), C.c_void_p, C.c_void_p, C.c_void_p]),
    "mtgr_hstu_layer_fwd": (C.c_int, [C.POINTER(LayerWeights), C.c_void_p, C.c_void_p, C.POINTER(LayerSaved),
                                      C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int64, C.c_int,
                                      C.c_void_p, C.c_size_t, C.c_void_p]),
    "mtgr_hstu_stack_fwd": (C.c_int, [C.POINTER(LayerWeights), C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.POINTER(LayerSaved), C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p,
                                      C.c_int64, C.c_int, C.c_void_p, C.c_size_t, C.c_void_p]),
    "mtgr_stack_cache_size": (C.c_size_t, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "mtgr_stack_chunk_workspace_size": (C.c_size_t, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int]),
    "mtgr_hstu_stack_hist_fwd": (C.c_int, [C.POINTER(LayerWeights), C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                           C.c_int32, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int,
                                           C.c_void_p, C.c_size_t, C.c_void_p]),
    "mtgr_hstu_stack_cand_fwd": (C.c_int, [C.POINTER(LayerWeights), C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                           C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                           C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_size_t, C.c_void_p]),
    "mtgr_hstu_layer_bwd": (C.c_int, [C.POINTER(LayerWeights), C.c_void_p, C.POINTER(LayerSaved), C.c_void_p,
                                      C.c_void_p, C.POINTER(LayerGrads), C.c_void_p, C.c_int32, C.c_void_p,
                                      C.c_void_p, C.c_int64, C.c_int, C.c_void_p, C.c_size_t, C.c_void_p]),
}


def lib():
    """Load libmtgr.so (built in-tree by hstu_attention_attn_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m hstu_attention_attn_b300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
def _p(t):
    """Address of a tensor argument: None is NULL and an int passes as a raw
    address.  Tensor arguments of the C ABI are device memory, so a tensor in
    host memory is refused here, before a kernel could dereference it."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return MTGR_BF16
    if t.dtype == torch.float32:
        return MTGR_F32
    if t.dtype == torch.float16:
        return MTGR_F16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(fn, code):
    if code != 0:
        raise MtgrError(fn, code, lib().mtgr_last_error().decode())


def mtgr_last_error() -> str:
    return lib().mtgr_last_error().decode()


def mtgr_version() -> int:
    return lib().mtgr_version()


def mtgr_trace_enable(on: bool = True):
    lib().mtgr_trace_enable(1 if on else 0)


def mtgr_trace_reset():
    lib().mtgr_trace_reset()


def mtgr_trace_report(max_entries: int = 64) -> dict:
    """{kernel name: (total device ms, launches)} since the last reset."""
    name_len = 48
    names = C.create_string_buffer(max_entries * name_len)
    ms = (C.c_double * max_entries)()
    cnt = (C.c_int32 * max_entries)()
    n = lib().mtgr_trace_report(max_entries, C.cast(names, C.c_void_p), name_len, C.cast(ms, C.c_void_p),
                                C.cast(cnt, C.c_void_p))
    if n < 0:
        raise MtgrError("mtgr_trace_report", n, "CUDA error while reading trace events")
    out = {}
    for k in range(min(n, max_entries)):
        nm = names.raw[k * name_len:(k + 1) * name_len].split(b"\0", 1)[0].decode()
        out[nm] = (float(ms[k]), int(cnt[k]))
    return out


def mtgr_validate_batch(offsets, gid, T, status_word, stream=None):
    _check("mtgr_validate_batch", lib().mtgr_validate_batch(_p(offsets), offsets.numel() - 1, _p(gid), T,
                                                            _p(status_word), _stream(stream)))


def mtgr_debug_visible_counts(offsets, gid, ts, T, cnt, total_pairs, stream=None):
    _check("mtgr_debug_visible_counts",
           lib().mtgr_debug_visible_counts(_p(offsets), offsets.numel() - 1, _p(gid), _p(ts), T, _p(cnt),
                                           _p(total_pairs), _stream(stream)))


def mtgr_debug_wait_timeout(status_word, stream=None):
    _check("mtgr_debug_wait_timeout", lib().mtgr_debug_wait_timeout(_p(status_word), _stream(stream)))


def mtgr_group_layernorm_fwd(x, y, mean, rstd, gid, gamma, beta, eps=1e-5, stream=None):
    T, D = x.shape
    _check("mtgr_group_layernorm_fwd",
           lib().mtgr_group_layernorm_fwd(_p(x), _p(y), _p(mean), _p(rstd), _p(gid), _p(gamma), _p(beta), T, D,
                                          eps, _dtype(x), _stream(stream)))


def mtgr_group_layernorm_bwd_workspace_size(T, D) -> int:
    return lib().mtgr_group_layernorm_bwd_workspace_size(T, D)


def mtgr_group_layernorm_bwd(dy, x, mean, rstd, gid, gamma, dx_residual, dx, dgamma, dbeta, workspace, stream=None):
    T, D = x.shape
    _check("mtgr_group_layernorm_bwd",
           lib().mtgr_group_layernorm_bwd(_p(dy), _p(x), _p(mean), _p(rstd), _p(gid), _p(gamma), _p(dx_residual),
                                          _p(dx), _p(dgamma), _p(dbeta), T, D, _dtype(x), _p(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))


def mtgr_group_layernorm_bwd_noalloc(dy, x, mean, rstd, gid, gamma, dx_residual, dx, dgamma, dbeta, stream=None):
    """Group LayerNorm backward without a workspace argument, for callers that
    cannot allocate device memory; the library keeps its partial sums in a fixed
    device array, so calls must not overlap on the GPU."""
    T, D = x.shape
    _check("mtgr_group_layernorm_bwd_noalloc",
           lib().mtgr_group_layernorm_bwd_noalloc(_p(dy), _p(x), _p(mean), _p(rstd), _p(gid), _p(gamma),
                                                  _p(dx_residual), _p(dx), _p(dgamma), _p(dbeta), T, D, _dtype(x),
                                                  _stream(stream)))


def mtgr_attn_workspace_size(B, T, n_heads, d_h, dtype) -> int:
    return lib().mtgr_attn_workspace_size(B, T, n_heads, d_h, dtype)


def mtgr_debug_plan_counts(workspace, B, stream=None):
    """[forward items, dK/dV items, dQ items, 1 if the backward kept its dS tiles]
    of the last attention or layer call on `workspace` (synchronises)."""
    out = np.zeros(4, dtype=np.int32)
    _check("mtgr_debug_plan_counts", lib().mtgr_debug_plan_counts(_p(workspace), B, out.ctypes.data, _stream(stream)))
    return [int(v) for v in out]


def mtgr_attn_ds_store_size(offsets_host, n_heads, d_h, dtype) -> int:
    """Extra workspace bytes with which the backward keeps its dS tiles;
    offsets_host: the batch's B+1 offsets in host memory (array-like)."""
    o = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int32))
    return lib().mtgr_attn_ds_store_size(o.ctypes.data, len(o) - 1, n_heads, d_h, dtype)


def mtgr_hstu_attn_fwd(q, k, v, u, ld_in, offsets, gid, ts, T, n_heads, d_h, eps, y, o_saved, ln_mean, ln_rstd,
                       workspace, stream=None):
    _check("mtgr_hstu_attn_fwd",
           lib().mtgr_hstu_attn_fwd(_p(q), _p(k), _p(v), _p(u), ld_in, _p(offsets), offsets.numel() - 1, _p(gid),
                                    _p(ts), T, n_heads, d_h, eps, _p(y), _p(o_saved), _p(ln_mean), _p(ln_rstd),
                                    _dtype(y), _p(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)))


def mtgr_hstu_attn_bwd(dy, q, k, v, u, ld_in, o_saved, ln_mean, ln_rstd, offsets, gid, ts, T, n_heads, d_h,
                       dq, dk, dv, du, ld_grad, dsilu_uqkv, workspace, stream=None):
    _check("mtgr_hstu_attn_bwd",
           lib().mtgr_hstu_attn_bwd(_p(dy), _p(q), _p(k), _p(v), _p(u), ld_in, _p(o_saved), _p(ln_mean),
                                    _p(ln_rstd), _p(offsets), offsets.numel() - 1, _p(gid), _p(ts), T, n_heads,
                                    d_h, _p(dq), _p(dk), _p(dv), _p(du), ld_grad, _p(dsilu_uqkv), _dtype(dy),
                                    _p(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)))


def mtgr_layer_workspace_size(B, T, d_model, n_heads, d_h, dtype) -> int:
    return lib().mtgr_layer_workspace_size(B, T, d_model, n_heads, d_h, dtype)


def make_weights(d_model, n_heads, d_h, w_uqkv, w_o, gamma, beta, eps_gln=1e-5, eps_ln=1e-5) -> LayerWeights:
    return LayerWeights(d_model, n_heads, d_h, _p(w_uqkv), _p(w_o), _p(gamma), _p(beta), eps_gln, eps_ln)


def make_saved(d) -> LayerSaved:
    return LayerSaved(*[_p(d[n]) for n, _ in LayerSaved._fields_])


def make_grads(d) -> LayerGrads:
    return LayerGrads(*[_p(d[n]) for n, _ in LayerGrads._fields_])


def mtgr_layer_weights_to_f16(weights: LayerWeights, w_uqkv_f16, w_o_f16, stream=None):
    _check("mtgr_layer_weights_to_f16",
           lib().mtgr_layer_weights_to_f16(C.byref(weights), _p(w_uqkv_f16), _p(w_o_f16), _stream(stream)))


def mtgr_hstu_layer_fwd(weights: LayerWeights, x, x_out, saved: LayerSaved, offsets, gid, ts, T, workspace,
                        stream=None):
    _check("mtgr_hstu_layer_fwd",
           lib().mtgr_hstu_layer_fwd(C.byref(weights), _p(x), _p(x_out), C.byref(saved), _p(offsets),
                                     offsets.numel() - 1, _p(gid), _p(ts), T, _dtype(x), _p(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def mtgr_stack_cache_size(n_layers, n_hist, chunk, d_model, n_heads, d_h) -> int:
    return int(lib().mtgr_stack_cache_size(n_layers, n_hist, chunk, d_model, n_heads, d_h))


def mtgr_stack_chunk_workspace_size(n_hist, chunk, d_model, n_heads, d_h, dtype) -> int:
    return int(lib().mtgr_stack_chunk_workspace_size(n_hist, chunk, d_model, n_heads, d_h, dtype))


def mtgr_hstu_stack_hist_fwd(weights, x_hist, act, cache, chunk, gid, ts, n_hist, n_cand, workspace, stream=None):
    """History rows of one request through every layer (cache filled); weights: LayerWeights per layer."""
    arr = (LayerWeights * len(weights))(*weights)
    _check("mtgr_hstu_stack_hist_fwd",
           lib().mtgr_hstu_stack_hist_fwd(arr, len(weights), _p(x_hist), _p(act), _p(cache), chunk, _p(gid), _p(ts),
                                          n_hist, n_cand, _dtype(x_hist), _p(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))


def mtgr_hstu_stack_cand_fwd(weights, x_cand, x_out, act, cache, chunk, gid, ts, n_hist, n_cand, c0, workspace,
                             stream=None):
    """One chunk of candidates (rows of x_cand) of the request through every layer against the cached history."""
    arr = (LayerWeights * len(weights))(*weights)
    _check("mtgr_hstu_stack_cand_fwd",
           lib().mtgr_hstu_stack_cand_fwd(arr, len(weights), _p(x_cand), _p(x_out), _p(act), _p(cache), chunk,
                                          _p(gid), _p(ts), n_hist, n_cand, c0, x_cand.shape[0], _dtype(x_cand),
                                          _p(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream)))


def mtgr_hstu_stack_fwd(weights, x, x_out, act, saved: LayerSaved, offsets, gid, ts, T, workspace, stream=None):
    """weights: a sequence of LayerWeights (one per layer)."""
    arr = (LayerWeights * len(weights))(*weights)
    _check("mtgr_hstu_stack_fwd",
           lib().mtgr_hstu_stack_fwd(arr, len(weights), _p(x), _p(x_out), _p(act), C.byref(saved), _p(offsets),
                                     offsets.numel() - 1, _p(gid), _p(ts), T, _dtype(x), _p(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def mtgr_hstu_layer_bwd(weights: LayerWeights, x, saved: LayerSaved, dx_out, dx, grads: LayerGrads, offsets, gid,
                        ts, T, workspace, stream=None):
    _check("mtgr_hstu_layer_bwd",
           lib().mtgr_hstu_layer_bwd(C.byref(weights), _p(x), C.byref(saved), _p(dx_out), _p(dx), C.byref(grads),
                                     _p(offsets), offsets.numel() - 1, _p(gid), _p(ts), T, _dtype(x),
                                     _p(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


# ---------------------------------------------------------------------------
# Training batches (host arrays in, host arrays out; no device work)
# ---------------------------------------------------------------------------
def mtgr_stochastic_length(offsets, gid, max_seq, draws):
    """Stochastic-length selection of one batch: returns (keep, new_offsets),
    the kept token indices (int32, ascending) and the new offsets (int32 [B+1]).
    offsets int32 [B+1], gid uint8 [T], draws uint64 [B] (host arrays)."""
    offsets = np.ascontiguousarray(offsets, np.int32)
    gid = np.ascontiguousarray(gid, np.uint8)
    draws = np.ascontiguousarray(draws, np.uint64)
    B, T = len(offsets) - 1, len(gid)
    keep = np.empty(max(T, 1), np.int32)
    new_offsets = np.empty(B + 1, np.int32)
    new_T = C.c_int64(0)
    _check("mtgr_stochastic_length",
           lib().mtgr_stochastic_length(offsets.ctypes.data, B, gid.ctypes.data, T, int(max_seq), draws.ctypes.data,
                                        keep.ctypes.data, new_offsets.ctypes.data, C.addressof(new_T)))
    return keep[:new_T.value].copy(), new_offsets


def mtgr_token_balanced_split(tokens, n_ranks):
    """Token-balanced contiguous split of users over n_ranks: returns
    (rank_first int32 [n_ranks+1], rank_tokens int64 [n_ranks], grad_weight float64 [n_ranks])."""
    tokens = np.ascontiguousarray(tokens, np.int64)
    first = np.empty(n_ranks + 1, np.int32)
    rank_tokens = np.empty(n_ranks, np.int64)
    weight = np.empty(n_ranks, np.float64)
    _check("mtgr_token_balanced_split",
           lib().mtgr_token_balanced_split(tokens.ctypes.data, len(tokens), int(n_ranks), first.ctypes.data,
                                           rank_tokens.ctypes.data, weight.ctypes.data))
    return first, rank_tokens, weight


def mtgr_expand_rows(src, rows, dst, stream=None):
    """dst [T, D] <- zeros, then dst[rows[k]] = src[k] (device tensors; rows int32)."""
    _check("mtgr_expand_rows",
           lib().mtgr_expand_rows(_p(src), _p(rows), rows.numel(), _p(dst), dst.shape[0], dst.shape[1], _dtype(dst),
                                  _stream(stream)))
