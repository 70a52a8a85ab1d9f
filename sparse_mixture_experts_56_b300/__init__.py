"""B300-native sparse mixture-of-experts feed-forward layer (Mixtral 8x7B style).

    G(x) = Softmax(TopK(x · W_g)),   y = sum_i G(x)_i · w2_i (SiLU(w1_i x) ⊙ (w3_i x))

Thin Python binding of libmoe.so.  Each function marshals torch CUDA tensors (device
memory and the current stream) into the C call of the same name declared in
include/moe.h; every step of the layer runs in the library's CUDA kernels.  When a result
tensor is not passed in, it is allocated with torch on the input's device.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import _native
from ._native import (MOE_BF16, MOE_F32, MOE_TC_FORM_AUTO, MOE_TC_FORM_PAIR, MOE_TC_FORM_SINGLE,
                      MOE_TC_FORM_SWAP, MoEError, check)

__all__ = [
    "MOE_F32", "MOE_BF16", "MoEError", "dtype_code", "moe_workspace_size", "workspace",
    "moe_router_topk", "moe_permute", "moe_permute_noalloc", "moe_grouped_swiglu", "moe_expert_up", "moe_expert_down",
    "moe_combine", "moe_rmsnorm", "moe_routing_stats", "moe_backward_workspace_size",
    "backward_workspace", "moe_layer_backward", "moe_train_saved_size", "train_saved",
    "moe_layer_forward_train", "moe_layer_backward_saved", "moe_attention_gqa",
    "moe_layer_forward", "moe_check_device_error", "moe_set_wait_limit_ns", "moe_set_tc_form",
    "MOE_TC_FORM_AUTO", "MOE_TC_FORM_SINGLE", "MOE_TC_FORM_PAIR", "MOE_TC_FORM_SWAP", "moe_version",
    "library_path", "moe_ep_regroup", "moe_gather_rows", "moe_decoder_workspace_size",
    "decoder_workspace", "moe_decoder_layer_forward",
]


def library_path() -> str:
    return _native.LIB_PATH


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return MOE_F32
    if dt == torch.bfloat16:
        return MOE_BF16
    raise ValueError(f"unsupported dtype {dt}: float32 or bfloat16")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def moe_version() -> int:
    return _native.lib().moe_version()


def moe_workspace_size(T: int, d: int, f: int, n: int, k: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return int(_native.lib().moe_workspace_size(T, d, f, n, k, code))


def workspace(T: int, d: int, f: int, n: int, k: int, dtype, device="cuda") -> torch.Tensor:
    """A zeroed workspace buffer of moe_workspace_size bytes."""
    size = moe_workspace_size(T, d, f, n, k, dtype)
    if size == 0:
        raise ValueError("invalid sizes")
    return torch.zeros(size, dtype=torch.uint8, device=device)


def moe_set_wait_limit_ns(ns: int) -> None:
    _native.lib().moe_set_wait_limit_ns(int(ns))


def moe_set_tc_form(form: int) -> None:
    """Selects the tensor-core GEMM form: MOE_TC_FORM_AUTO, _SINGLE, _PAIR or _SWAP."""
    check("moe_set_tc_form", _native.lib().moe_set_tc_form(int(form)))


def moe_check_device_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the workspace's device status."""
    return int(_native.lib().moe_check_device_error(_ptr(ws), ws.numel(), _stream(stream)))


def moe_router_topk(x: torch.Tensor, w_gate: torch.Tensor, k: int,
                    logit_bias: Optional[torch.Tensor] = None, *, want_logits: bool = False,
                    topk_idx: Optional[torch.Tensor] = None, topk_w: Optional[torch.Tensor] = None,
                    logits: Optional[torch.Tensor] = None, stream=None):
    T, d = x.shape
    n = w_gate.shape[1]
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if want_logits and logits is None:
        logits = torch.empty((T, n), dtype=torch.float32, device=dev)
    st = _native.lib().moe_router_topk(_ptr(x), _ptr(w_gate), _ptr(logit_bias), T, d, n, k,
                                       dtype_code(x.dtype), _ptr(topk_idx), _ptr(topk_w),
                                       _ptr(logits), _stream(stream))
    check("moe_router_topk", st)
    return topk_idx, topk_w, logits


def moe_permute(topk_idx: torch.Tensor, n: int, ws: torch.Tensor, *,
                expert_offsets: Optional[torch.Tensor] = None, perm: Optional[torch.Tensor] = None,
                inv_perm: Optional[torch.Tensor] = None, stream=None):
    T, k = topk_idx.shape
    dev = topk_idx.device
    if expert_offsets is None:
        expert_offsets = torch.empty(n + 1, dtype=torch.int32, device=dev)
    if perm is None:
        perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    if inv_perm is None:
        inv_perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    st = _native.lib().moe_permute(_ptr(topk_idx), T, k, n, _ptr(expert_offsets), _ptr(perm),
                                   _ptr(inv_perm), _ptr(ws), ws.numel(), _stream(stream))
    check("moe_permute", st)
    return expert_offsets, perm, inv_perm


def moe_permute_noalloc(topk_idx: torch.Tensor, n: int, *, expert_offsets: torch.Tensor,
                        perm: torch.Tensor, inv_perm: torch.Tensor, stream=None):
    """moe_permute for callers that cannot allocate: no workspace, and every result buffer
    must be passed in (this wrapper allocates nothing either)."""
    T, k = topk_idx.shape
    st = _native.lib().moe_permute_noalloc(_ptr(topk_idx), T, k, n, _ptr(expert_offsets),
                                           _ptr(perm), _ptr(inv_perm), _stream(stream))
    check("moe_permute_noalloc", st)
    return expert_offsets, perm, inv_perm


def moe_grouped_swiglu(x: torch.Tensor, perm: torch.Tensor, expert_offsets: torch.Tensor,
                       w1: torch.Tensor, w3: torch.Tensor, w2: torch.Tensor, k: int,
                       ws: torch.Tensor, *, y_perm: Optional[torch.Tensor] = None, stream=None):
    T, d = x.shape
    n, f, _ = w1.shape
    if y_perm is None:
        y_perm = torch.empty((T * k, d), dtype=x.dtype, device=x.device)
    st = _native.lib().moe_grouped_swiglu(_ptr(x), _ptr(perm), _ptr(expert_offsets), _ptr(w1),
                                          _ptr(w3), _ptr(w2), T, d, f, n, k, dtype_code(x.dtype),
                                          _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream))
    check("moe_grouped_swiglu", st)
    return y_perm


def moe_expert_up(x: torch.Tensor, perm: torch.Tensor, expert_offsets: torch.Tensor,
                  w1: torch.Tensor, w3: torch.Tensor, k: int, ws: torch.Tensor, *,
                  h: Optional[torch.Tensor] = None, stream=None):
    T, d = x.shape
    n, f, _ = w1.shape
    if h is None:
        h = torch.empty((T * k, f), dtype=x.dtype, device=x.device)
    st = _native.lib().moe_expert_up(_ptr(x), _ptr(perm), _ptr(expert_offsets), _ptr(w1), _ptr(w3),
                                     T, d, f, n, k, dtype_code(x.dtype), _ptr(h), _ptr(ws),
                                     ws.numel(), _stream(stream))
    check("moe_expert_up", st)
    return h


def moe_expert_down(h: torch.Tensor, expert_offsets: torch.Tensor, w2: torch.Tensor, k: int,
                    ws: torch.Tensor, *, y_perm: Optional[torch.Tensor] = None, stream=None):
    A, f = h.shape
    n, d, _ = w2.shape
    T = A // k
    if y_perm is None:
        y_perm = torch.empty((A, d), dtype=h.dtype, device=h.device)
    st = _native.lib().moe_expert_down(_ptr(h), _ptr(expert_offsets), _ptr(w2), T, d, f, n, k,
                                       dtype_code(h.dtype), _ptr(y_perm), _ptr(ws), ws.numel(),
                                       _stream(stream))
    check("moe_expert_down", st)
    return y_perm


def moe_combine(y_perm: torch.Tensor, inv_perm: torch.Tensor, topk_w: torch.Tensor,
                residual: Optional[torch.Tensor] = None, *, y: Optional[torch.Tensor] = None,
                stream=None):
    T, k = topk_w.shape
    d = y_perm.shape[1]
    if y is None:
        y = torch.empty((T, d), dtype=y_perm.dtype, device=y_perm.device)
    st = _native.lib().moe_combine(_ptr(y_perm), _ptr(inv_perm), _ptr(topk_w), _ptr(residual), T, d,
                                   k, dtype_code(y_perm.dtype), _ptr(y), _stream(stream))
    check("moe_combine", st)
    return y


def moe_rmsnorm(h: torch.Tensor, eps: float = 1e-5, *, x: Optional[torch.Tensor] = None,
                stream=None):
    T, d = h.shape
    if x is None:
        x = torch.empty_like(h)
    st = _native.lib().moe_rmsnorm(_ptr(h), T, d, float(eps), dtype_code(h.dtype), _ptr(x),
                                   _stream(stream))
    check("moe_rmsnorm", st)
    return x


def moe_layer_forward(x: torch.Tensor, w_gate: torch.Tensor, w1: torch.Tensor, w3: torch.Tensor,
                      w2: torch.Tensor, k: int, ws: torch.Tensor, *,
                      logit_bias: Optional[torch.Tensor] = None,
                      residual: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                      topk_idx_out: Optional[torch.Tensor] = None,
                      expert_offsets_out: Optional[torch.Tensor] = None, stream=None):
    T, d = x.shape
    n, f, _ = w1.shape
    if y is None:
        y = torch.empty_like(x)
    st = _native.lib().moe_layer_forward(_ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(w1), _ptr(w3),
                                         _ptr(w2), _ptr(residual), T, d, f, n, k, dtype_code(x.dtype),
                                         _ptr(y), _ptr(topk_idx_out), _ptr(expert_offsets_out),
                                         _ptr(ws), ws.numel(), _stream(stream))
    check("moe_layer_forward", st)
    return y


def moe_routing_stats(topk_idx: torch.Tensor, n: int, seq_len: int = 0, *,
                      expert_counts: Optional[torch.Tensor] = None,
                      pair_counts: Optional[torch.Tensor] = None, stream=None):
    """Expert load and consecutive-token repetition of one layer's TopK selections.

    Returns (expert_counts int64 [n], pair_counts int64 [3] = pairs, same first choice,
    shared expert)."""
    T, k = topk_idx.shape
    dev = topk_idx.device
    if expert_counts is None:
        expert_counts = torch.empty(n, dtype=torch.int64, device=dev)
    if pair_counts is None:
        pair_counts = torch.empty(3, dtype=torch.int64, device=dev)
    st = _native.lib().moe_routing_stats(_ptr(topk_idx), T, k, n, int(seq_len), _ptr(expert_counts),
                                         _ptr(pair_counts), _stream(stream))
    check("moe_routing_stats", st)
    return expert_counts, pair_counts


def moe_backward_workspace_size(T: int, d: int, f: int, n: int, k: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return int(_native.lib().moe_backward_workspace_size(T, d, f, n, k, code))


def backward_workspace(T: int, d: int, f: int, n: int, k: int, dtype=torch.bfloat16,
                       device="cuda") -> torch.Tensor:
    """A zeroed workspace of moe_backward_workspace_size bytes."""
    size = moe_backward_workspace_size(T, d, f, n, k, dtype)
    if size == 0:
        raise ValueError("invalid or unsupported sizes")
    return torch.zeros(size, dtype=torch.uint8, device=device)


def moe_layer_backward(x: torch.Tensor, w_gate: torch.Tensor, w1: torch.Tensor, w3: torch.Tensor,
                       w2: torch.Tensor, k: int, dy: torch.Tensor, ws: torch.Tensor, *,
                       logit_bias: Optional[torch.Tensor] = None, want_dbias: bool = False,
                       dx: Optional[torch.Tensor] = None, dw_gate: Optional[torch.Tensor] = None,
                       dw1: Optional[torch.Tensor] = None, dw3: Optional[torch.Tensor] = None,
                       dw2: Optional[torch.Tensor] = None,
                       dlogit_bias: Optional[torch.Tensor] = None, stream=None):
    """Gradients of <dy, MoE(x)>: returns dict dx, dw_gate, dw1, dw3, dw2 (and dlogit_bias)."""
    T, d = x.shape
    n, f, _ = w1.shape
    dev = x.device
    dx = torch.empty_like(x) if dx is None else dx
    dw_gate = torch.empty((d, n), dtype=torch.float32, device=dev) if dw_gate is None else dw_gate
    dw1 = torch.empty_like(w1) if dw1 is None else dw1
    dw3 = torch.empty_like(w3) if dw3 is None else dw3
    dw2 = torch.empty_like(w2) if dw2 is None else dw2
    if want_dbias and dlogit_bias is None:
        dlogit_bias = torch.empty(n, dtype=torch.float32, device=dev)
    st = _native.lib().moe_layer_backward(
        _ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(dy), T, d, f,
        n, k, dtype_code(x.dtype), _ptr(dx), _ptr(dw_gate), _ptr(dlogit_bias), _ptr(dw1),
        _ptr(dw3), _ptr(dw2), _ptr(ws), ws.numel(), _stream(stream))
    check("moe_layer_backward", st)
    out = {"dx": dx, "dw_gate": dw_gate, "dw1": dw1, "dw3": dw3, "dw2": dw2}
    if dlogit_bias is not None:
        out["dlogit_bias"] = dlogit_bias
    return out


def moe_train_saved_size(T: int, d: int, f: int, n: int, k: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return int(_native.lib().moe_train_saved_size(T, d, f, n, k, code))


def train_saved(T: int, d: int, f: int, n: int, k: int, dtype=torch.bfloat16,
                device="cuda") -> torch.Tensor:
    """An uninitialised buffer of moe_train_saved_size bytes."""
    size = moe_train_saved_size(T, d, f, n, k, dtype)
    if size == 0:
        raise ValueError("invalid or unsupported sizes")
    return torch.empty(size, dtype=torch.uint8, device=device)


def moe_layer_forward_train(x: torch.Tensor, w_gate: torch.Tensor, w1: torch.Tensor,
                            w3: torch.Tensor, w2: torch.Tensor, k: int, ws: torch.Tensor,
                            saved: torch.Tensor, *, logit_bias: Optional[torch.Tensor] = None,
                            residual: Optional[torch.Tensor] = None,
                            y: Optional[torch.Tensor] = None, stream=None):
    """moe_layer_forward that also fills `saved` for moe_layer_backward_saved."""
    T, d = x.shape
    n, f, _ = w1.shape
    if y is None:
        y = torch.empty_like(x)
    st = _native.lib().moe_layer_forward_train(
        _ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(residual), T,
        d, f, n, k, dtype_code(x.dtype), _ptr(y), _ptr(saved), saved.numel(), _ptr(ws), ws.numel(),
        _stream(stream))
    check("moe_layer_forward_train", st)
    return y


def moe_layer_backward_saved(x: torch.Tensor, w_gate: torch.Tensor, w1: torch.Tensor,
                             w3: torch.Tensor, w2: torch.Tensor, k: int, dy: torch.Tensor,
                             saved: torch.Tensor, ws: torch.Tensor, *, want_dbias: bool = False,
                             stream=None):
    """moe_layer_backward from the buffer filled by moe_layer_forward_train."""
    T, d = x.shape
    n, f, _ = w1.shape
    dev = x.device
    out = {"dx": torch.empty_like(x), "dw_gate": torch.empty((d, n), dtype=torch.float32, device=dev),
           "dw1": torch.empty_like(w1), "dw3": torch.empty_like(w3), "dw2": torch.empty_like(w2)}
    if want_dbias:
        out["dlogit_bias"] = torch.empty(n, dtype=torch.float32, device=dev)
    st = _native.lib().moe_layer_backward_saved(
        _ptr(x), _ptr(w_gate), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(dy), T, d, f, n, k,
        dtype_code(x.dtype), _ptr(saved), saved.numel(), _ptr(out["dx"]), _ptr(out["dw_gate"]),
        _ptr(out.get("dlogit_bias")), _ptr(out["dw1"]), _ptr(out["dw3"]), _ptr(out["dw2"]),
        _ptr(ws), ws.numel(), _stream(stream))
    check("moe_layer_backward_saved", st)
    return out


def moe_attention_gqa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ws: torch.Tensor,
                      seq_len: int = 0, *, out: Optional[torch.Tensor] = None, stream=None):
    """Causal grouped-query attention: q [T, hq, dh], k and v [T, hkv, dh] -> [T, hq, dh]."""
    T, hq, dh = q.shape
    hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    st = _native.lib().moe_attention_gqa(_ptr(q), _ptr(k), _ptr(v), T, int(seq_len), hq, hkv, dh,
                                         dtype_code(q.dtype), _ptr(out), _ptr(ws), ws.numel(),
                                         _stream(stream))
    check("moe_attention_gqa", st)
    return out


def moe_ep_regroup(recv_counts: torch.Tensor, R: int, *, local_offsets: Optional[torch.Tensor] = None,
                   row_map: Optional[torch.Tensor] = None, inv_row_map: Optional[torch.Tensor] = None,
                   stream=None):
    """recv_counts [G, E] int32 (device) -> (local_offsets [E+1], row_map [R], inv_row_map [R])."""
    G, E = recv_counts.shape
    dev = recv_counts.device
    if recv_counts.dtype != torch.int32:
        raise ValueError("recv_counts must be int32")
    if local_offsets is None:
        local_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if row_map is None:
        row_map = torch.empty(R, dtype=torch.int32, device=dev)
    if inv_row_map is None:
        inv_row_map = torch.empty(R, dtype=torch.int32, device=dev)
    for t, size in ((local_offsets, E + 1), (row_map, R), (inv_row_map, R)):
        if t.dtype != torch.int32 or t.numel() < size:
            raise ValueError("local_offsets, row_map and inv_row_map: int32 of E + 1, R and R")
    st = _native.lib().moe_ep_regroup(_ptr(recv_counts), G, E, R, _ptr(local_offsets),
                                      _ptr(row_map), _ptr(inv_row_map), _stream(stream))
    check("moe_ep_regroup", st)
    return local_offsets, row_map, inv_row_map


def moe_gather_rows(src: torch.Tensor, index: torch.Tensor, k: int = 1, *,
                    dst: Optional[torch.Tensor] = None, stream=None):
    """dst[p] = src[index[p] // k] (zero rows for indices outside [0, rows(src) * k))."""
    rows = index.shape[0]
    if index.dtype != torch.int32:
        raise ValueError("index must be int32")
    if dst is None:
        dst = torch.empty((rows,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    if rows == 0:
        return dst
    row_bytes = (dst.numel() // rows) * dst.element_size()
    if dst.shape[0] != rows or (src.shape[0] and src[0].numel() * src.element_size() != row_bytes):
        raise ValueError("src and dst rows must have the same size; dst one row per index")
    st = _native.lib().moe_gather_rows(_ptr(src), src.shape[0], _ptr(index), rows, k, row_bytes,
                                       _ptr(dst), _stream(stream))
    check("moe_gather_rows", st)
    return dst


def moe_decoder_workspace_size(T: int, d: int, f: int, n: int, k: int, hq: int, hkv: int) -> int:
    return int(_native.lib().moe_decoder_workspace_size(T, d, f, n, k, hq, hkv))


def decoder_workspace(T: int, d: int, f: int, n: int, k: int, hq: int, hkv: int,
                      device="cuda") -> torch.Tensor:
    """A workspace for moe_decoder_layer_forward with its status header zeroed."""
    size = moe_decoder_workspace_size(T, d, f, n, k, hq, hkv)
    if size == 0:
        raise ValueError("invalid sizes")
    ws = torch.empty(size, dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def moe_decoder_layer_forward(h: torch.Tensor, wq: torch.Tensor, wk: torch.Tensor, wv: torch.Tensor,
                              wo: torch.Tensor, w_gate: torch.Tensor, w1: torch.Tensor,
                              w3: torch.Tensor, w2: torch.Tensor, k: int, hq: int, hkv: int,
                              ws: torch.Tensor, *, seq_len: int = 0, eps: float = 1e-5,
                              logit_bias: Optional[torch.Tensor] = None,
                              y: Optional[torch.Tensor] = None,
                              topk_idx_out: Optional[torch.Tensor] = None, stream=None):
    """One decoder layer (attention sub-block + MoE sub-block, each with its residual)."""
    T, d = h.shape
    n, f, _ = w1.shape
    if y is None:
        y = torch.empty_like(h)
    st = _native.lib().moe_decoder_layer_forward(
        _ptr(h), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _ptr(w_gate), _ptr(logit_bias), _ptr(w1),
        _ptr(w3), _ptr(w2), T, d, f, n, k, hq, hkv, seq_len, eps, dtype_code(h.dtype), _ptr(y),
        _ptr(topk_idx_out), _ptr(ws), ws.numel(), _stream(stream))
    check("moe_decoder_layer_forward", st)
    return y

