"""Shared test helpers: moving seeded inputs to the GPU and comparing with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
import workloads

# Tolerances (max |y - y_ref| <= rel * max |y_ref|)
TOL = {"bf16": 2e-2, "f32": 1e-4}
NEAR_TIE = 1e-4


def to_device(a, w: workloads.Workload, dev):
    import torch
    if a is None:
        return None
    if w.dtype == "bf16" and a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def to_numpy_f32(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy()


def f32_inputs(inp, w):
    return {k: workloads.as_f32(inp[k], w) for k in ("x", "wg", "w1", "w3", "w2") if k in inp}


def check_selection(gpu_idx: np.ndarray, logits_ref: np.ndarray, k: int, eps: float = NEAR_TIE):
    """Bit-exact expert indices except near-tie tokens; near-tie tokens must still hold a valid
    selection (every chosen logit within eps of the K-th largest).  Returns (n_set_ties,
    n_order_ties)."""
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    ref = oracle.topk_select(logits_ref, k)
    set_tie, order_tie = oracle.near_tie_tokens(logits_ref, k, eps)
    same_set = np.all(np.sort(gpu_idx, 1) == np.sort(ref, 1), axis=1)
    bad = ~same_set & ~set_tie
    assert not bad.any(), f"{bad.sum()} tokens chose different experts (first {np.flatnonzero(bad)[:5]})"
    same_order = np.all(gpu_idx == ref, axis=1)
    bad_order = same_set & ~same_order & ~order_tie & ~set_tie
    assert not bad_order.any(), f"{bad_order.sum()} tokens have the slots out of order"
    # validity for the tokens excluded above
    kth = np.sort(logits_ref, axis=1)[:, ::-1][:, k - 1]
    chosen = np.take_along_axis(logits_ref, gpu_idx, axis=1)
    assert np.all(chosen >= kth[:, None] - eps), "a near-tie token holds an invalid selection"
    assert np.all([len(set(r)) == k for r in gpu_idx.tolist()]), "duplicate expert in a selection"
    return int(set_tie.sum()), int(order_tie.sum())


def gate_weights_for(idx: np.ndarray, logits_ref: np.ndarray) -> np.ndarray:
    """Softmax of the oracle's logits at the given selection (fp64)."""
    sel = np.take_along_axis(np.asarray(logits_ref, dtype=np.float64), np.asarray(idx, dtype=np.int64), 1)
    e = np.exp(sel - sel.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def assert_close_rel(got: np.ndarray, ref: np.ndarray, rel: float, what: str = "y"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= rel * scale + 1e-30, f"{what}: max|err| {err:.4e} > {rel} * {scale:.4e}"
    return err / scale if scale > 0 else 0.0
