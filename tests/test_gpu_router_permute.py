"""GPU parity of the router/top-K/softmax kernel and the grouping kernel against the oracle."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from tests.helpers import (TOL, assert_close_rel, check_selection, f32_inputs, gate_weights_for,
                           to_device, to_numpy_f32)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_56_b300 as m
    m._native.lib()
    return m


DEV = "cuda"


ROUTER_CASES = [
    # (T, d, n, k, dtype, skew)
    (64, 128, 8, 2, "f32", False),          # the tiny fp32 workload's shape
    (513, 4096, 8, 2, "bf16", False),       # fast path (n = 8, d % 256 == 0), ragged T
    (300, 4096, 8, 2, "bf16", True),        # with the per-expert logit bias
    (97, 200, 8, 2, "bf16", False),         # generic path (d not a multiple of 256)
    (50, 64, 32, 4, "f32", False),          # n = 32
    (40, 96, 5, 5, "bf16", False),          # K = n
    (33, 48, 1, 1, "f32", False),           # one expert
    (70, 256, 8, 1, "bf16", False),         # K = 1
    (1, 4096, 8, 2, "bf16", False),         # one token
    (2000, 4096, 8, 2, "bf16", True),       # large batch: W_g staged in shared memory
    (1025, 1280, 8, 2, "bf16", False),      # first large-batch size, d not a power of two
]


@pytest.mark.parametrize("case", ROUTER_CASES, ids=lambda c: "T{}-d{}-n{}-k{}-{}{}".format(*c[:5], "-bias" if c[5] else ""))
def test_router_topk_matches_oracle(moe, case):
    T, d, n, k, dt, skew = case
    w = workloads.custom(T, d, 8, n, k, dt, wid=200, skew_bias=skew)
    inp = workloads.make_inputs(w, tensors=("x", "wg"))
    x, wg = to_device(inp["x"], w, DEV), to_device(inp["wg"], w, DEV)
    bias = torch.from_numpy(inp["bias"]).to(DEV) if skew else None
    idx, gw, logits = moe.moe_router_topk(x, wg, k, bias, want_logits=True)
    torch.cuda.synchronize()
    xf, wgf = workloads.as_f32(inp["x"], w), workloads.as_f32(inp["wg"], w)
    lref = oracle.router_logits(xf, wgf, inp["bias"])
    lg = logits.cpu().numpy().astype(np.float64)
    scale = np.abs(xf).astype(np.float64) @ np.abs(wgf).astype(np.float64)
    assert np.all(np.abs(lg - lref) <= 1e-6 * scale + 1e-6), "fp32 logits off by more than rounding"
    gi = idx.cpu().numpy()
    check_selection(gi, lref, k)
    np.testing.assert_allclose(gw.cpu().numpy(), gate_weights_for(gi, lref), rtol=0, atol=2e-6)
    np.testing.assert_allclose(gw.cpu().numpy().sum(1), 1.0, atol=1e-6)


def test_router_worked_example(moe):
    """The page's example: experts 3 and 5 kept, G_3 = 3/4, G_5 = 1/4 (fixture values)."""
    path = os.path.join(os.path.dirname(__file__), "golden", "gate_worked_example.json")
    fx = json.load(open(path))

    def ev(s):
        return math.log(float(Fraction(s[4:-1]))) if s.startswith("log(") else float(Fraction(s))

    l = np.array([ev(v) for v in fx["logits"]], dtype=np.float32)
    x = torch.ones((1, 1), dtype=torch.float32, device=DEV)
    wg = torch.from_numpy(l[None, :].copy()).to(DEV)
    idx, gw, _ = moe.moe_router_topk(x, wg, fx["k"])
    assert idx.cpu().numpy().tolist() == [fx["expected_idx"]]
    g = [ev(v) for v in fx["expected_G"]]
    np.testing.assert_allclose(gw.cpu().numpy()[0], [g[i] for i in fx["expected_idx"]], atol=1e-6)


def test_router_ties_go_to_lower_index(moe):
    wg = torch.tensor([[1.0, 2.0, 2.0, 0.5, 2.0]], device=DEV)
    x = torch.ones((2, 1), device=DEV)
    idx, gw, _ = moe.moe_router_topk(x, wg, 2)
    assert idx.cpu().tolist() == [[1, 2], [1, 2]]
    np.testing.assert_allclose(gw.cpu().numpy(), 0.5, atol=1e-7)


def _permute_check(moe, idx_np, n):
    T, k = idx_np.shape
    ws = moe.workspace(max(T, 1), 64, 64, n, k, torch.bfloat16, DEV)
    ti = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    off, perm, inv = moe.moe_permute(ti, n, ws)
    assert moe.moe_check_device_error(ws) == 0
    roff, rperm, rinv = oracle.group_by_expert(idx_np, n)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert np.array_equal(perm.cpu().numpy(), rperm)
    assert np.array_equal(inv.cpu().numpy(), rinv)


PERMUTE_CASES = {
    "random-t64": (np.random.default_rng(1).integers(0, 8, (64, 2)), 8),
    "all-to-one": (np.full((1000, 2), 3), 8),
    "empty-experts": (np.array([[7, 0]] * 45), 8),
    "ragged-k3": (np.random.default_rng(2).integers(0, 5, (17, 3)), 8),
    "n32": (np.random.default_rng(3).integers(0, 32, (777, 2)), 32),
    "one-token": (np.array([[5, 2]]), 8),
    "chunk-edge": (np.random.default_rng(4).integers(0, 8, (16384, 2)), 8),
    "multi-block": (np.random.default_rng(5).integers(0, 8, (150001, 2)), 8),
    "multi-block-skew": (np.minimum(np.random.default_rng(6).geometric(0.4, (70000, 2)) - 1, 7), 8),
}


@pytest.mark.parametrize("name", sorted(PERMUTE_CASES))
def test_permute_bit_exact(moe, name):
    idx, n = PERMUTE_CASES[name]
    _permute_check(moe, np.asarray(idx), n)


def test_permute_empty(moe):
    ws = moe.workspace(1, 64, 64, 8, 2, torch.bfloat16, DEV)
    off = torch.full((9,), -1, dtype=torch.int32, device=DEV)
    ti = torch.empty((0, 2), dtype=torch.int32, device=DEV)
    moe.moe_permute(ti, 8, ws, expert_offsets=off,
                    perm=torch.empty(0, dtype=torch.int32, device=DEV),
                    inv_perm=torch.empty(0, dtype=torch.int32, device=DEV))
    assert off.cpu().tolist() == [0] * 9


def test_permute_reports_bad_index(moe):
    ws = moe.workspace(4, 64, 64, 8, 2, torch.bfloat16, DEV)
    ti = torch.tensor([[0, 1], [2, 9], [3, 4], [-1, 5]], dtype=torch.int32, device=DEV)
    moe.moe_permute(ti, 8, ws)
    assert moe.moe_check_device_error(ws) == 6   # MOE_ERR_DEVICE_INDEX
    assert moe.moe_check_device_error(ws) == 0   # cleared


def _with_bad(rng, T, k, n, frac):
    idx = rng.integers(0, n, (T, k))
    bad = rng.random((T, k)) < frac
    idx[bad] = rng.choice([-1, n, n + 5, -100], size=int(bad.sum()))
    return idx, bad


@pytest.mark.parametrize("T,k,n", [(45, 2, 8), (40000, 2, 8), (700, 2, 32), (20000, 2, 32)])
def test_permute_bad_indices_go_to_a_trailing_bucket(moe, T, k, n):
    """Assignments with an expert index outside [0, n) land after every expert, in ascending
    order: expert_offsets[n] counts only the valid ones, perm / inv_perm stay a permutation of
    [0, T*k).  Expected: the oracle's grouping of the same indices with every bad index
    relabelled n, over n + 1 buckets.  Single- and multi-block launches; n = 32 puts the
    trailing bucket in the 33rd counter."""
    rng = np.random.default_rng(T + n)
    idx, bad = _with_bad(rng, T, k, n, 0.05)
    ws = moe.workspace(T, 64, 64, n, k, torch.bfloat16, DEV)
    off, perm, inv = moe.moe_permute(torch.from_numpy(idx.astype(np.int32)).to(DEV), n, ws)
    assert moe.moe_check_device_error(ws) == 6
    relabel = np.where(bad, n, idx)
    roff, rperm, rinv = oracle.group_by_expert(relabel, n + 1)
    assert off.cpu().numpy().tolist() == roff[:n + 1].tolist()
    assert off.cpu().numpy()[n] == T * k - bad.sum()
    assert np.array_equal(perm.cpu().numpy(), rperm)
    assert np.array_equal(inv.cpu().numpy(), rinv)


def test_layer_steps_after_bad_indices_stay_in_bounds(moe):
    """The grouping of a selection with bad indices drives the experts and the combine without
    any out-of-bounds access; tokens whose slots are all valid still match the oracle (the
    checks skip the tokens with a bad slot, whose output is unspecified)."""
    w = workloads.custom(200, 128, 192, 8, 2, "bf16", wid=470)
    inp = workloads.make_inputs(w)
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "w1", "w3", "w2")}
    rng = np.random.default_rng(47)
    idx, bad = _with_bad(rng, w.T, w.k, w.n, 0.1)
    gate = rng.random((w.T, w.k)).astype(np.float32)
    gate /= gate.sum(1, keepdims=True)
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    off, perm, inv = moe.moe_permute(torch.from_numpy(idx.astype(np.int32)).to(DEV), w.n, ws)
    yp = moe.moe_grouped_swiglu(g["x"], perm, off, g["w1"], g["w3"], g["w2"], w.k, ws)
    y = moe.moe_combine(yp, inv, torch.from_numpy(gate).to(DEV))
    assert moe.moe_check_device_error(ws) == 6
    ok = ~bad.any(1)
    f = f32_inputs(inp, w)
    xs = f["x"]
    ref = np.zeros((int(ok.sum()), w.d))
    for r, t in enumerate(np.flatnonzero(ok)):
        for s in range(w.k):
            e = idx[t, s]
            ref[r] += gate[t, s] * oracle.expert_swiglu(xs[t:t + 1], f["w1"][e], f["w3"][e], f["w2"][e])[0]
    assert_close_rel(to_numpy_f32(y)[ok], ref, TOL["bf16"])
