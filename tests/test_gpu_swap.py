"""GPU parity of the swapped form of the expert GEMMs, the form the bf16 layer takes for
batches of at most 64 tokens (decode): the weights are the 128-row side of every MMA and an
expert's token rows, in blocks of 16-64, the other side.  Checked against the oracle, against
the single-CTA form on the same inputs (bit for bit: both sum the same products in the same
16-deep K steps), with several token blocks per expert (the form forced on larger batches),
ragged weight tiles (f = 320: the last up-projection tile holds 64 rows; d = 384: the second
128-row half of the last down-projection tile lies past the expert), experts without rows,
and under a 1 ns wait limit."""
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


CASES = {
    # name: (T, d, f, n, k, skew)           token block (MMA N) under the default rule
    "t1": (1, 256, 256, 8, 2, False),        # 16
    "t20-n32": (20, 256, 384, 32, 2, False),  # 32; most of the 32 experts get 0-2 rows
    "t32-d512-f1024": (32, 512, 1024, 8, 2, False),   # 32: the decode batch, smaller dims
    "t48-n1-k1": (48, 256, 256, 1, 1, False),          # 48: one expert, three token boxes
    "t64-d384-f320-skew": (64, 384, 320, 8, 2, True),  # 64: ragged weight tiles in both GEMMs
}


def _workload(name, wid_base=1200):
    T, d, f, n, k, skew = CASES[name]
    return workloads.custom(T, d, f, n, k, "bf16", wid=wid_base + sorted(CASES).index(name),
                            skew_bias=skew)


def _dev(inp, w):
    return {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2")}


def _forward(moe, g, w, bias, ws, form):
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    off = torch.empty(w.n + 1, dtype=torch.int32, device=DEV)
    moe.moe_set_tc_form(form)
    try:
        y = moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws,
                                  logit_bias=bias, topk_idx_out=idx, expert_offsets_out=off)
        assert moe.moe_check_device_error(ws) == 0
    finally:
        moe.moe_set_tc_form(moe.MOE_TC_FORM_AUTO)
    return y, idx, off


def _oracle_on(inp, w, idx):
    f = f32_inputs(inp, w)
    lref = oracle.router_logits(f["x"], f["wg"], inp["bias"])
    gi = idx.cpu().numpy().astype(np.int64)
    check_selection(gi, lref, w.k)
    return oracle.moe_layer(f["x"], f["wg"], f["w1"], f["w3"], f["w2"], w.k, inp["bias"],
                            idx=gi, w=gate_weights_for(gi, lref)), gi


@pytest.mark.parametrize("name", sorted(CASES))
def test_swap_form_matches_oracle_and_single_form(moe, name):
    w = _workload(name)
    inp = workloads.make_inputs(w)
    g = _dev(inp, w)
    bias = torch.from_numpy(inp["bias"]).to(DEV) if inp["bias"] is not None else None
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    y_auto, idx, off = _forward(moe, g, w, bias, ws, moe.MOE_TC_FORM_AUTO)   # swapped (T <= 64)
    y_single, idx2, _ = _forward(moe, g, w, bias, ws, moe.MOE_TC_FORM_SINGLE)
    assert torch.equal(idx, idx2)
    yref, gi = _oracle_on(inp, w, idx)
    roff, _, _ = oracle.group_by_expert(gi, w.n)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert_close_rel(to_numpy_f32(y_auto), yref, TOL["bf16"])
    assert torch.equal(y_auto.view(torch.int16), y_single.view(torch.int16)), \
        f"swapped and single-CTA forms differ in {(y_auto != y_single).sum().item()} elements"


@pytest.mark.parametrize("T,d,f,n,skew", [(300, 256, 384, 8, True), (200, 128, 192, 2, False)])
def test_swap_form_with_several_token_blocks(moe, T, d, f, n, skew):
    """Forced on batches above 64 tokens, the swapped form splits each expert's rows into
    64-row blocks (the skewed expert 0 holds about 90 rows at T = 300; with n = 2 each
    expert holds about 200 rows: four blocks, the last one partial) and still agrees with the
    oracle and, bit for bit, with the single-CTA form."""
    w = workloads.custom(T, d, f, n, 2, "bf16", wid=1250 + n, skew_bias=skew)
    inp = workloads.make_inputs(w)
    g = _dev(inp, w)
    bias = torch.from_numpy(inp["bias"]).to(DEV) if inp["bias"] is not None else None
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    y_swap, idx, off = _forward(moe, g, w, bias, ws, moe.MOE_TC_FORM_SWAP)
    counts = np.diff(off.cpu().numpy())
    assert counts.max() > 64, counts   # at least one expert spans several blocks
    y_single, _, _ = _forward(moe, g, w, bias, ws, moe.MOE_TC_FORM_SINGLE)
    yref, _ = _oracle_on(inp, w, idx)
    assert_close_rel(to_numpy_f32(y_swap), yref, TOL["bf16"])
    assert torch.equal(y_swap.view(torch.int16), y_single.view(torch.int16))


def test_swap_expert_rows_through_the_split_calls(moe):
    """moe_expert_up and moe_expert_down (the EP building blocks) in the swapped form: h and
    y_perm rows against the oracle's expert outputs, including experts without rows."""
    w = _workload("t20-n32")
    inp = workloads.make_inputs(w)
    g = _dev(inp, w)
    f = f32_inputs(inp, w)
    ridx, _, _, _ = oracle.gate(f["x"], f["wg"], w.k, inp["bias"])
    roff, rperm, _ = oracle.group_by_expert(ridx, w.n)
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    perm = torch.from_numpy(rperm.astype(np.int32)).to(DEV)
    off = torch.from_numpy(roff.astype(np.int32)).to(DEV)
    h = moe.moe_expert_up(g["x"], perm, off, g["w1"], g["w3"], w.k, ws)
    yp = moe.moe_expert_down(h, off, g["w2"], w.k, ws)
    assert moe.moe_check_device_error(ws) == 0
    href = np.zeros((w.T * w.k, w.f))
    yref = np.zeros((w.T * w.k, w.d))
    for e in range(w.n):
        rows = rperm[roff[e]:roff[e + 1]]
        if rows.size:
            xe = f["x"][rows // w.k]
            a, b = xe @ f["w1"][e].T, xe @ f["w3"][e].T
            href[roff[e]:roff[e + 1]] = oracle.silu(a) * b
            yref[roff[e]:roff[e + 1]] = oracle.expert_swiglu(xe, f["w1"][e], f["w3"][e], f["w2"][e])
    assert_close_rel(to_numpy_f32(h), href, TOL["bf16"], "h")
    assert_close_rel(to_numpy_f32(yp), yref, TOL["bf16"], "y_perm")


def test_swap_timeout_path_reports_and_recovers(moe):
    """Under a 1 ns wait limit the swapped kernels stop at their first wait (the MMA issuer
    waits for a weight copy that cannot land in 1 ns), report MOE_ERR_TIMEOUT, and the next
    call on the same context is correct."""
    w = _workload("t32-d512-f1024")
    inp = workloads.make_inputs(w)
    g = _dev(inp, w)
    ws = moe.workspace(w.T, w.d, w.f, w.n, w.k, torch.bfloat16, DEV)
    try:
        moe.moe_set_wait_limit_ns(1)
        moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws)
        st = moe.moe_check_device_error(ws)
    finally:
        moe.moe_set_wait_limit_ns(0)
    assert st == 5, f"status {st}, expected MOE_ERR_TIMEOUT (5)"
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    y = moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], w.k, ws, topk_idx_out=idx)
    assert moe.moe_check_device_error(ws) == 0
    yref, _ = _oracle_on(inp, w, idx)
    assert_close_rel(to_numpy_f32(y), yref, TOL["bf16"])
