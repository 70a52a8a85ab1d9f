"""GPU parity of the layer's backward (moe_layer_backward) against the fp64 oracle's
gradients, on shapes that span several tiles of every backward GEMM (128-row padded expert
segments, 256-column n-tiles, 64-deep reduction blocks) with ragged tails, empty experts,
K = 1, K = n, one expert and 32 experts.

The oracle is evaluated on the GPU router's own selection (a near-tie token may select either
expert; the gates of that selection come from the oracle's fp64 logits).  Every gradient must
satisfy max|g - g_ref| <= 2e-2 * max|g_ref| (the bf16 rule of the forward)."""
import numpy as np
import pytest

import oracle
import workloads
from tests.helpers import TOL, assert_close_rel, check_selection, to_device, to_numpy_f32

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_56_b300 as m
    m._native.lib()
    return m


CASES = {
    # name: (T, d, f, n, k, skew)
    "t300-d256-f384-skew": (300, 256, 384, 8, 2, True),
    "t77-d128-f192": (77, 128, 192, 8, 2, False),          # partial n-tiles, partial M tiles
    "t640-d384-f320-skew": (640, 384, 320, 8, 2, True),    # d, f not multiples of 128 / 256
    "t5-empty-experts": (5, 128, 128, 8, 2, False),        # most experts get no rows
    "n1-k1-t130": (130, 256, 256, 1, 1, False),            # a plain SwiGLU FFN, no router grad
    "k-equals-n-t90": (90, 128, 128, 4, 4, False),
    "n32-k2-t500": (500, 128, 128, 32, 2, False),
    "t1": (1, 256, 256, 8, 2, False),
    "t1100-d512-f768": (1100, 512, 768, 8, 2, False),      # several 128-row tiles per expert
    # CUDA-core path: fp32 storage (tolerance 1e-4), or bf16 shapes off the 64-multiple grid
    "fp32-tiny-t64": (64, 128, 256, 8, 2, False, "f32"),   # the tiny fp32 workload's shape
    "fp32-n4-t45-skew": (45, 96, 80, 4, 2, True, "f32"),
    "fp32-k-equals-n-t20": (20, 40, 24, 3, 3, False, "f32"),
    "simt-bf16-d200-f136": (64, 200, 136, 8, 2, False),
}


def _run(moe, name, wid):
    T, d, f, n, k, skew, *dt = CASES[name]
    dt = dt[0] if dt else "bf16"
    w = workloads.custom(T, d, f, n, k, dt, wid=wid, skew_bias=skew)
    inp = workloads.make_inputs(w, tensors=("x", "wg", "w1", "w3", "w2", "dy"))
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2", "dy")}
    bias = torch.from_numpy(inp["bias"]).to(DEV) if inp["bias"] is not None else None
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    ws = moe.backward_workspace(T, d, f, n, k, tdt, DEV)
    out = moe.moe_layer_backward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], k, g["dy"], ws,
                                 logit_bias=bias, want_dbias=True)
    assert moe.moe_check_device_error(ws) == 0
    idx, _, _ = moe.moe_router_topk(g["x"], g["wg"], k, bias)
    torch.cuda.synchronize()
    return w, inp, out, idx.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(moe, name):
    w, inp, out, gi = _run(moe, name, 600 + sorted(CASES).index(name))
    f = {t: workloads.as_f32(inp[t], w).astype(np.float64) for t in ("x", "wg", "w1", "w3", "w2", "dy")}
    lref = oracle.router_logits(f["x"], f["wg"], inp["bias"])
    check_selection(gi, lref, w.k)
    ref = oracle.moe_layer_backward(f["x"], f["wg"], f["w1"], f["w3"], f["w2"], w.k, f["dy"],
                                    inp["bias"], idx=gi)
    tol = TOL[w.dtype]
    assert_close_rel(to_numpy_f32(out["dx"]), ref["dx"], tol, "dx")
    assert_close_rel(to_numpy_f32(out["dw1"]), ref["dw1"], tol, "dw1")
    assert_close_rel(to_numpy_f32(out["dw3"]), ref["dw3"], tol, "dw3")
    assert_close_rel(to_numpy_f32(out["dw2"]), ref["dw2"], tol, "dw2")
    if w.k == 1:
        # the gate is identically 1: no router gradient at all
        assert torch.count_nonzero(out["dw_gate"]).item() == 0
        assert torch.count_nonzero(out["dlogit_bias"]).item() == 0
    else:
        assert_close_rel(out["dw_gate"].cpu().numpy(), ref["dwg"], tol, "dw_gate")
        assert_close_rel(out["dlogit_bias"].cpu().numpy(), ref["dbias"], tol, "dlogit_bias")
    # experts without rows get exactly zero weight gradients
    counts = np.bincount(gi.reshape(-1), minlength=w.n)
    for e in np.flatnonzero(counts == 0):
        for key in ("dw1", "dw3", "dw2"):
            assert torch.count_nonzero(out[key][e]).item() == 0, (key, e)


def test_backward_is_deterministic(moe):
    """Two calls give bit-identical gradients (no atomics decide any sum)."""
    _, _, a, _ = _run(moe, "t300-d256-f384-skew", 650)
    _, _, b, _ = _run(moe, "t300-d256-f384-skew", 650)
    for key in a:
        assert torch.equal(a[key].view(torch.uint8) if a[key].dtype != torch.float32 else a[key],
                           b[key].view(torch.uint8) if b[key].dtype != torch.float32 else b[key]), key


@pytest.mark.parametrize("name", ["t300-d256-f384-skew", "t640-d384-f320-skew", "t5-empty-experts",
                                  "n32-k2-t500", "t1100-d512-f768", "t1"])
def test_weight_gradient_forms_agree(moe, name):
    """The weight gradients from the CTA-pair form (256-row tiles of dW over two SMs, the
    default) and from the single-CTA form are bit-identical: both reduce every dW element over
    the expert's rows in the same 64-row blocks and 16-row MMA steps.  The shapes include
    dW row counts (f = 384, 320, 768; d = 384) that end inside a 256-row tile, and experts
    without rows (their dW is zero in both forms)."""
    got = {}
    for form in (moe.MOE_TC_FORM_SINGLE, moe.MOE_TC_FORM_AUTO):
        moe.moe_set_tc_form(form)
        try:
            _, _, out, _ = _run(moe, name, 660 + sorted(CASES).index(name))
        finally:
            moe.moe_set_tc_form(moe.MOE_TC_FORM_AUTO)
        got[form] = out
    a, b = got[moe.MOE_TC_FORM_SINGLE], got[moe.MOE_TC_FORM_AUTO]
    for key in a:
        x1, x2 = a[key], b[key]
        same = torch.equal(x1, x2) if x1.dtype == torch.float32 else \
            torch.equal(x1.view(torch.int16), x2.view(torch.int16))
        assert same, key


def _f64(a, w):
    return workloads.as_f32(a, w).astype(np.float64)


@pytest.mark.slow
@pytest.mark.parametrize("wid", [2, 3])
def test_full_size_backward(moe, wid):
    """The Mixtral-shaped decode (T=32) and prefill (T=4096) workloads at full size, in the
    launch configuration the benchmark times.  The oracle's steps run one expert at a time in
    fp64: dG for every assignment (so dW_g and the bias gradient are compared whole), dx on a
    token sample, and every expert's dW1, dW3, dW2 at decode / the largest and the smallest
    expert's at prefill."""
    w = workloads.workload(wid)
    T, d, f, n, k = w.T, w.d, w.f, w.n, w.k
    inp = workloads.make_inputs(w, tensors=("x", "wg", "w1", "w3", "w2", "dy"))
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2", "dy")}
    ws = moe.backward_workspace(T, d, f, n, k, torch.bfloat16, DEV)
    out = moe.moe_layer_backward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], k, g["dy"], ws,
                                 want_dbias=True)
    assert moe.moe_check_device_error(ws) == 0
    idx, _, _ = moe.moe_router_topk(g["x"], g["wg"], k)
    gi = idx.cpu().numpy().astype(np.int64)
    del g
    x, dy, wg = _f64(inp["x"], w), _f64(inp["dy"], w), _f64(inp["wg"], w)
    lref = oracle.router_logits(x, wg)
    check_selection(gi, lref, k)
    gw = oracle.masked_softmax(np.take_along_axis(lref, gi, axis=1))
    offsets, perm, _ = oracle.group_by_expert(gi, n)
    counts = np.diff(offsets)
    rng = np.random.default_rng(wid)
    sample = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=min(T, 48), replace=False)]))
    in_sample = np.zeros(T, dtype=bool)
    in_sample[sample] = True
    check_w = set(range(n)) if T <= 64 else {int(np.argmax(counts)), int(np.argmin(counts))}
    dgate = np.zeros((T, k))
    dx_ref = np.zeros((T, d))
    tol = TOL["bf16"]
    for e in range(n):
        sel = perm[offsets[e]:offsets[e + 1]]
        if sel.size == 0:
            continue
        t, slot = sel // k, sel % k
        w1e, w3e, w2e = (_f64(inp[m][e], w) for m in ("w1", "w3", "w2"))
        xs, ge = x[t], dy[t]
        dgate[t, slot] = np.sum(ge * oracle.expert_swiglu(xs, w1e, w3e, w2e), axis=1)
        do = gw[t, slot][:, None] * ge
        if e in check_w:
            dxs, dw1, dw3, dw2 = oracle.expert_swiglu_backward(xs, do, w1e, w3e, w2e)
            assert_close_rel(to_numpy_f32(out["dw1"][e]), dw1, tol, f"dw1[{e}]")
            assert_close_rel(to_numpy_f32(out["dw3"][e]), dw3, tol, f"dw3[{e}]")
            assert_close_rel(to_numpy_f32(out["dw2"][e]), dw2, tol, f"dw2[{e}]")
            np.add.at(dx_ref, t, dxs)
        else:
            m = in_sample[t]
            if m.any():
                dxs, _, _, _ = oracle.expert_swiglu_backward(xs[m], do[m], w1e, w3e, w2e)
                np.add.at(dx_ref, t[m], dxs)
        del w1e, w3e, w2e
    dl = np.zeros((T, n))
    np.put_along_axis(dl, gi, oracle.softmax_backward(gw, dgate), axis=1)
    dx_ref += dl @ wg.T
    assert_close_rel(to_numpy_f32(out["dx"])[sample], dx_ref[sample], tol, "dx (token sample)")
    assert_close_rel(out["dw_gate"].cpu().numpy(), x.T @ dl, tol, "dw_gate")
    assert_close_rel(out["dlogit_bias"].cpu().numpy(), dl.sum(axis=0), tol, "dlogit_bias")


@pytest.mark.parametrize("name,form", [("t300-d256-f384-skew", 0), ("t640-d384-f320-skew", 0),
                                       ("t5-empty-experts", 0), ("n32-k2-t500", 0),
                                       ("t1100-d512-f768", 0), ("t1100-d512-f768", 2),
                                       ("t300-d256-f384-skew", 2)])
def test_training_pair_matches_the_separate_calls(moe, name, form):
    """moe_layer_forward_train gives moe_layer_forward's y bit for bit, and
    moe_layer_backward_saved the gradients of moe_layer_backward (which recomputes a | b with
    the same tile shapes and reduction order), bit for bit; both match the oracle."""
    T, d, f, n, k, skew = CASES[name][:6]
    w = workloads.custom(T, d, f, n, k, "bf16", wid=700 + sorted(CASES).index(name), skew_bias=skew)
    inp = workloads.make_inputs(w, tensors=("x", "wg", "w1", "w3", "w2", "dy"))
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2", "dy")}
    bias = torch.from_numpy(inp["bias"]).to(DEV) if inp["bias"] is not None else None
    ws = moe.workspace(T, d, f, n, k, torch.bfloat16, DEV)
    bws = moe.backward_workspace(T, d, f, n, k, torch.bfloat16, DEV)
    saved = moe.train_saved(T, d, f, n, k, torch.bfloat16, DEV)
    y_ref = moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], k, ws, logit_bias=bias)
    moe.moe_set_tc_form(form)   # 2: the up-projection saves a | b from the CTA-pair form too
    try:
        y = moe.moe_layer_forward_train(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], k, ws, saved,
                                        logit_bias=bias)
    finally:
        moe.moe_set_tc_form(moe.MOE_TC_FORM_AUTO)
    assert moe.moe_check_device_error(ws) == 0
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    a = moe.moe_layer_backward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], k, g["dy"], bws,
                               logit_bias=bias, want_dbias=True)
    b = moe.moe_layer_backward_saved(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], k, g["dy"], saved,
                                     bws, want_dbias=True)
    assert moe.moe_check_device_error(bws) == 0
    for key in a:
        x1, x2 = a[key], b[key]
        same = torch.equal(x1, x2) if x1.dtype == torch.float32 else \
            torch.equal(x1.view(torch.int16), x2.view(torch.int16))
        assert same, key
