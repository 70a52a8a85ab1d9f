"""GPU parity of the experts (grouped SwiGLU), the combine and the whole layer against the
oracle, on sizes the oracle finishes in seconds that still span several tiles (128-row
m-tiles, 128/256-column n-tiles, 64-wide k-steps) and ragged tails."""
import numpy as np
import pytest

import oracle
import workloads
from tests.helpers import (TOL, assert_close_rel, check_selection, f32_inputs, gate_weights_for,
                           to_device, to_numpy_f32)

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


def _dev_inputs(inp, w):
    return {k: to_device(inp[k], w, DEV) for k in ("x", "wg", "w1", "w3", "w2")}


LAYER_CASES = {
    # name: (T, d, f, n, k, dtype, skew)
    "tiny-fp32-t64": None,                                     # workload 1 itself
    "tc-t300-d256-f384-skew": (300, 256, 384, 8, 2, "bf16", True),
    "tc-t1000-d512-f1024": (1000, 512, 1024, 8, 2, "bf16", False),
    "tc-t77-d128-f192": (77, 128, 192, 8, 2, "bf16", False),   # partial n-tiles in both GEMMs
    "tc-t640-d384-f320-skew": (640, 384, 320, 8, 2, "bf16", True),
    "tc-n1-k1": (130, 256, 256, 1, 1, "bf16", False),          # a plain SwiGLU FFN
    "tc-k-equals-n": (90, 128, 128, 4, 4, "bf16", False),       # dense softmax mixture
    "tc-n32-k2": (500, 128, 128, 32, 2, "bf16", False),
    "tc-t1": (1, 256, 256, 8, 2, "bf16", False),
    "simt-bf16-d200": (64, 200, 136, 8, 2, "bf16", False),     # not a multiple of 64
    # CTA-pair tensor-core form (the down-projection takes it when the experts average >= 256
    # rows, the up-projection at >= 512; pair-t2048 and pair-n1-k1 run both GEMMs as pairs):
    # 256-row tiles split over two CTAs, ragged last tiles in both CTAs of a pair
    "pair-t2048-d256-f384": (2048, 256, 384, 8, 2, "bf16", False),
    "pair-t1500-d384-f320-skew": (1500, 384, 320, 8, 2, "bf16", True),   # partial n-tiles
    "pair-n1-k1-t700": (700, 256, 256, 1, 1, "bf16", False),            # 3 tiles, 188-row tail
    "pair-n2-k1-t600": (600, 128, 192, 2, 1, "bf16", False),
    "pair-n32-k2-t4200": (4200, 128, 128, 32, 2, "bf16", False),
    "simt-fp32-n4": (45, 96, 80, 4, 2, "f32", True),
}


def _workload(name):
    spec = LAYER_CASES[name]
    if spec is None:
        return workloads.workload(1)
    T, d, f, n, k, dt, skew = spec
    return workloads.custom(T, d, f, n, k, dt, wid=300 + sorted(LAYER_CASES).index(name), skew_bias=skew)


@pytest.mark.parametrize("name", sorted(LAYER_CASES))
def test_layer_forward_matches_oracle(moe, name):
    w = _workload(name)
    inp = workloads.make_inputs(w)
    g = _dev_inputs(inp, w)
    bias = torch.from_numpy(inp["bias"]).to(DEV) if inp["bias"] is not None else None
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, dt, DEV)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    off = torch.empty(w.n + 1, dtype=torch.int32, device=DEV)
    y = moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws, logit_bias=bias,
                              topk_idx_out=idx, expert_offsets_out=off)
    assert moe.moe_check_device_error(ws) == 0
    f = f32_inputs(inp, w)
    lref = oracle.router_logits(f["x"], f["wg"], inp["bias"])
    gi = idx.cpu().numpy().astype(np.int64)
    check_selection(gi, lref, w.k)
    # offsets: the grouping of the GPU's own selection (bit-exact)
    roff, _, _ = oracle.group_by_expert(gi, w.n)
    assert np.array_equal(off.cpu().numpy(), roff)
    # y: the oracle evaluated on the GPU's selection where the selection is a near tie,
    # otherwise on its own selection (they coincide there)
    yref = oracle.moe_layer(f["x"], f["wg"], f["w1"], f["w3"], f["w2"], w.k, inp["bias"],
                            idx=gi, w=gate_weights_for(gi, lref))
    assert_close_rel(to_numpy_f32(y), yref, TOL[w.dtype])


@pytest.mark.parametrize("name", ["tc-t300-d256-f384-skew", "tiny-fp32-t64", "simt-bf16-d200",
                                  "pair-t1500-d384-f320-skew", "pair-n1-k1-t700"])
def test_grouped_swiglu_rows(moe, name):
    """y_perm rows are the unweighted expert outputs E_e(x_t), grouped as the oracle groups."""
    w = _workload(name)
    inp = workloads.make_inputs(w)
    g = _dev_inputs(inp, w)
    f = f32_inputs(inp, w)
    ridx, _, _, _ = oracle.gate(f["x"], f["wg"], w.k, inp["bias"])
    roff, rperm, _ = oracle.group_by_expert(ridx, w.n)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, dt, DEV)
    perm = torch.from_numpy(rperm.astype(np.int32)).to(DEV)
    off = torch.from_numpy(roff.astype(np.int32)).to(DEV)
    yp = moe.moe_grouped_swiglu(g["x"], perm, off, g["w1"], g["w3"], g["w2"], w.k, ws)
    assert moe.moe_check_device_error(ws) == 0
    ypn = to_numpy_f32(yp)
    ref = np.zeros_like(ypn, dtype=np.float64)
    for e in range(w.n):
        rows = rperm[roff[e]:roff[e + 1]]
        if rows.size:
            ref[roff[e]:roff[e + 1]] = oracle.expert_swiglu(f["x"][rows // w.k], f["w1"][e], f["w3"][e], f["w2"][e])
    assert_close_rel(ypn, ref, TOL[w.dtype], "y_perm")


def test_combine_with_residual_and_alias(moe):
    T, d, k = 37, 256, 2
    rng = np.random.default_rng(7)
    yp = rng.standard_normal((T * k, d)).astype(np.float32)
    inv = rng.permutation(T * k).astype(np.int32)
    wts = rng.random((T, k)).astype(np.float32)
    res = rng.standard_normal((T, d)).astype(np.float32)
    for dt in (torch.float32, torch.bfloat16):
        ypt = torch.from_numpy(yp).to(DEV).to(dt)
        rt = torch.from_numpy(res).to(DEV).to(dt)
        y = moe.moe_combine(ypt, torch.from_numpy(inv).to(DEV), torch.from_numpy(wts).to(DEV), rt, y=rt)
        ypf = ypt.float().cpu().numpy().astype(np.float64)
        rf = torch.from_numpy(res).to(dt).float().numpy().astype(np.float64)
        ref = rf + sum(wts[:, s:s + 1].astype(np.float64) * ypf[inv.reshape(T, k)[:, s]] for s in range(k))
        assert_close_rel(to_numpy_f32(y), ref, 1e-6 if dt == torch.float32 else 8e-3, "combine")


def test_stacked_layers_small(moe):
    """h <- h + MoE_l(RMSNorm(h)) for 3 layers, oracle chained in fp64 from the same h_0."""
    w = workloads.custom(200, 256, 256, 8, 2, "bf16", wid=450)
    h0 = workloads.make_inputs(w, tensors=("x",))["x"]
    h = to_device(h0, w, DEV)
    href = workloads.as_f32(h0, w).astype(np.float64)
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    xn = torch.empty_like(h)
    excluded = np.zeros(w.T, dtype=bool)
    for layer in range(3):
        inp = workloads.make_inputs(w, layer=layer, tensors=("wg", "w1", "w3", "w2"))
        g = {k: to_device(inp[k], w, DEV) for k in ("wg", "w1", "w3", "w2")}
        f = f32_inputs(inp, w)
        moe.moe_rmsnorm(h, 1e-5, x=xn)
        idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
        h = moe.moe_layer_forward(xn, g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws, residual=h,
                                  y=torch.empty_like(h), topk_idx_out=idx)
        assert moe.moe_check_device_error(ws) == 0
        xr = oracle.rmsnorm(href)
        lref = oracle.router_logits(xr, f["wg"])
        # The GPU stores the normalised rows and h in bf16 (relative rounding error uniform
        # in +-2^-9, std 2^-9/sqrt(3)), which moves logit e by a random amount of std
        # sigma_e = 2^-9/sqrt(3) * sqrt(sum_i (x_i W_ie)^2), compounding over layers.  Tokens
        # whose 2nd/3rd gap is within ~5 sigma of a tie may legitimately route differently;
        # they are excluded from the comparison (and counted by the assert below).
        sigma = 2.0 ** -9 / np.sqrt(3) * np.sqrt(((xr[:, :, None] * f["wg"][None]) ** 2).sum(1)).max(1)
        band = 5 * sigma * (layer + 1)
        srt = np.sort(lref, 1)[:, ::-1]
        excluded |= (srt[:, 1] - srt[:, 2]) < band
        href = oracle.stacked_layer(href, f["wg"], f["w1"], f["w3"], f["w2"], w.k)
        keep = ~excluded
        assert keep.sum() >= 0.85 * w.T, f"{(~keep).sum()} of {w.T} tokens excluded"
        assert_close_rel(to_numpy_f32(h)[keep], href[keep], TOL["bf16"], f"h after layer {layer}")


def test_timeout_path_reports_and_recovers(moe):
    """A wait limit of 1 ns makes the tensor-core kernels give up at their first wait; they
    must stop cleanly (status MOE_ERR_TIMEOUT) and leave the context usable."""
    w = workloads.custom(300, 256, 384, 8, 2, "bf16", wid=460)
    inp = workloads.make_inputs(w)
    g = _dev_inputs(inp, w)
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    try:
        moe.moe_set_wait_limit_ns(1)
        moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws)
        st = moe.moe_check_device_error(ws)
    finally:
        moe.moe_set_wait_limit_ns(0)
    # 600 assignments over 8 experts give several tiles per GEMM: the MMA issuer's first wait
    # is on a TMA copy that cannot land within 1 ns, so the limit must fire
    assert st == 5, f"status {st}, expected MOE_ERR_TIMEOUT (5)"
    y = moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws)
    assert moe.moe_check_device_error(ws) == 0
    f = f32_inputs(inp, w)
    yref = oracle.moe_layer(f["x"], f["wg"], f["w1"], f["w3"], f["w2"], w.k)
    lref = oracle.router_logits(f["x"], f["wg"])
    keep = ~oracle.near_tie_tokens(lref, w.k)[0]
    assert_close_rel(to_numpy_f32(y)[keep], yref[keep], TOL["bf16"])


@pytest.mark.parametrize("name", ["tc-t77-d128-f192", "tc-t640-d384-f320-skew", "pair-t1500-d384-f320-skew",
                                  "pair-n1-k1-t700", "tc-t1"])
def test_tc_forms_agree(moe, name):
    """The single-CTA and CTA-pair forms of the expert GEMMs, each forced on the same inputs,
    give identical outputs (both accumulate K in the same order), and match the oracle."""
    w = _workload(name)
    inp = workloads.make_inputs(w)
    g = _dev_inputs(inp, w)
    bias = torch.from_numpy(inp["bias"]).to(DEV) if inp["bias"] is not None else None
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    ys = {}
    try:
        for form in (moe.MOE_TC_FORM_SINGLE, moe.MOE_TC_FORM_PAIR):
            moe.moe_set_tc_form(form)
            ys[form] = moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws,
                                             logit_bias=bias, topk_idx_out=idx)
            assert moe.moe_check_device_error(ws) == 0
    finally:
        moe.moe_set_tc_form(moe.MOE_TC_FORM_AUTO)
    a, b = ys[moe.MOE_TC_FORM_SINGLE], ys[moe.MOE_TC_FORM_PAIR]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), \
        f"forms differ in {(a != b).sum().item()} elements"
    f = f32_inputs(inp, w)
    lref = oracle.router_logits(f["x"], f["wg"], inp["bias"])
    gi = idx.cpu().numpy().astype(np.int64)
    yref = oracle.moe_layer(f["x"], f["wg"], f["w1"], f["w3"], f["w2"], w.k, inp["bias"],
                            idx=gi, w=gate_weights_for(gi, lref))
    assert_close_rel(to_numpy_f32(b), yref, TOL[w.dtype])


def test_timeout_path_of_the_pair_form(moe):
    """The CTA-pair form under a 1 ns wait limit: both CTAs of every pair give up, meet at
    their final cluster barrier, report MOE_ERR_TIMEOUT, and the next call is correct."""
    name = "pair-t2048-d256-f384"
    w = _workload(name)
    inp = workloads.make_inputs(w)
    g = _dev_inputs(inp, w)
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    moe.moe_set_tc_form(moe.MOE_TC_FORM_PAIR)
    try:
        try:
            moe.moe_set_wait_limit_ns(1)
            moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws)
            st = moe.moe_check_device_error(ws)
        finally:
            moe.moe_set_wait_limit_ns(0)
        assert st == 5, f"status {st}, expected MOE_ERR_TIMEOUT (5)"
        y = moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws)
        assert moe.moe_check_device_error(ws) == 0
    finally:
        moe.moe_set_tc_form(moe.MOE_TC_FORM_AUTO)
    f = f32_inputs(inp, w)
    yref = oracle.moe_layer(f["x"], f["wg"], f["w1"], f["w3"], f["w2"], w.k)
    lref = oracle.router_logits(f["x"], f["wg"])
    keep = ~oracle.near_tie_tokens(lref, w.k)[0]
    assert_close_rel(to_numpy_f32(y)[keep], yref[keep], TOL["bf16"])
