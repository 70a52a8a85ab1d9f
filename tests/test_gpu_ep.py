"""Expert parallelism on the GPU: the regrouping kernel bit-exact against the oracle's
receive-side plan, the row gather, and the whole EP layer pass through libmoe.so's kernels
-- with G = 1, 2, 4, 8 ranks emulated on one GPU (exchanges as device copies, no kernel
waiting for another rank's), and with one real NCCL rank -- against the single-GPU oracle
on each rank's tokens."""
import numpy as np
import pytest

import oracle
import workloads
from tests.helpers import TOL, assert_close_rel, check_selection, f32_inputs, gate_weights_for, to_device, to_numpy_f32

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


REGROUP_CASES = {
    "g2-e4": np.array([[3, 0, 5, 1], [2, 2, 0, 7]]),
    "g8-e1": np.random.default_rng(1).integers(0, 50, (8, 1)),
    "g4-e2-empty": np.zeros((4, 2), dtype=np.int64),
    "g1-e8": np.random.default_rng(2).integers(0, 3000, (1, 8)),
    "g16-e2-large": np.random.default_rng(3).integers(0, 9000, (16, 2)),
    "g4-e8-sparse": np.random.default_rng(4).integers(0, 3, (4, 8)) * np.random.default_rng(5).integers(0, 2, (4, 8)),
}


@pytest.mark.parametrize("name", sorted(REGROUP_CASES))
def test_ep_regroup_bit_exact(moe, name):
    c = REGROUP_CASES[name]
    R = int(c.sum())
    lo, rm, inv = moe.moe_ep_regroup(torch.from_numpy(c.astype(np.int32)).to(DEV), R)
    rlo, rrm, rinv = oracle.ep_regroup(c)
    assert lo.cpu().numpy().tolist() == rlo.tolist()
    assert rm.cpu().numpy().tolist() == rrm.tolist()
    assert inv.cpu().numpy().tolist() == rinv.tolist()


def test_gather_rows(moe):
    rng = np.random.default_rng(9)
    src = torch.from_numpy(rng.standard_normal((50, 40)).astype(np.float32)).to(torch.bfloat16).to(DEV)
    index = rng.integers(0, 100, 77)
    index[[3, 9]] = [-1, 100]                            # outside [0, rows * k): zero rows
    out = moe.moe_gather_rows(src, torch.from_numpy(index.astype(np.int32)).to(DEV), 2)
    ref = np.zeros((77, 40), dtype=np.float32)
    ok = (index >= 0) & (index < 100)
    ref[ok] = src.float().cpu().numpy()[index[ok] // 2]
    assert np.array_equal(out.float().cpu().numpy(), ref)
    odd = torch.from_numpy(rng.standard_normal((10, 3)).astype(np.float32)).to(DEV)   # 12-byte rows
    out = moe.moe_gather_rows(odd, torch.tensor([9, 0, 4], dtype=torch.int32, device=DEV))
    assert torch.equal(out, odd[[9, 0, 4]])


def _layer_inputs(G, Tr, d, f, n, k, skew, wid):
    w = workloads.custom(G * Tr, d, f, n, k, "bf16", wid=wid, skew_bias=skew)
    inp = workloads.make_inputs(w)
    return w, inp


def _check_rank_output(y, idx, inp, w, rows):
    f = f32_inputs(inp, w)
    x = f["x"][rows]
    lref = oracle.router_logits(x, f["wg"], inp["bias"])
    gi = idx.cpu().numpy().astype(np.int64)
    check_selection(gi, lref, w.k)
    yref = oracle.moe_layer(x, f["wg"], f["w1"], f["w3"], f["w2"], w.k, inp["bias"], idx=gi,
                            w=gate_weights_for(gi, lref))
    assert_close_rel(to_numpy_f32(y), yref, TOL["bf16"])


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_ep_emulated_ranks_match_oracle(moe, G):
    from sparse_mixture_experts_56_b300 import ep
    Tr, d, f, n, k = 160, 256, 384, 8, 2
    w, inp = _layer_inputs(G, Tr, d, f, n, k, skew=True, wid=480 + G)
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2")}
    bias = torch.from_numpy(inp["bias"]).to(DEV)
    xs = [g["x"][r * Tr:(r + 1) * Tr].contiguous() for r in range(G)]
    ops = ep.NativeOps(DEV)
    ys, stats = ep.ep_layer_forward_emulated(ops, xs, g["wg"], g["w1"], g["w3"], g["w2"], k, n, G, bias)
    torch.cuda.synchronize()
    for r in range(G):
        _check_rank_output(ys[r], stats["topk_idx"][r], inp, w, slice(r * Tr, (r + 1) * Tr))
    plans = oracle.ep_exchange_plan([i.cpu().numpy() for i in stats["topk_idx"]], n, G)
    assert stats["expert_rows"] == oracle.ep_load(plans).tolist()


def test_ep_one_nccl_rank(moe, tmp_path):
    """The SPMD pass over a real NCCL process group of one rank (all experts local): the
    count and row exchanges go through NCCL's all-to-all."""
    import torch.distributed as dist
    from sparse_mixture_experts_56_b300 import ep
    Tr, d, f, n, k = 300, 256, 384, 8, 2
    w, inp = _layer_inputs(1, Tr, d, f, n, k, skew=False, wid=490)
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2")}
    dist.init_process_group("nccl", init_method=f"file://{tmp_path}/store", rank=0, world_size=1,
                            device_id=torch.device(DEV, torch.cuda.current_device()))
    try:
        y, stats = ep.ep_layer_forward(ep.TorchComm(), ep.NativeOps(DEV), g["x"], g["wg"], g["w1"],
                                       g["w3"], g["w2"], k, n)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert stats["expert_rows"] == Tr * k and stats["recv_rows"] == [Tr * k]
    _check_rank_output(y, stats["topk_idx"], inp, w, slice(0, Tr))


def test_ep_ranks_without_tokens_or_rows(moe):
    """Degenerate expert-parallel passes: a rank with no tokens of its own, and ranks whose
    experts receive no rows at all (every token routed to rank 0's experts by the logit
    bias); the others still match the oracle and the empty ones return empty outputs."""
    from sparse_mixture_experts_56_b300 import ep
    G, Tr, d, f, n, k = 4, 96, 256, 384, 8, 2
    w = workloads.custom(G * Tr, d, f, n, k, "bf16", wid=497)
    inp = workloads.make_inputs(w)
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2")}
    ops = ep.NativeOps(DEV)
    # rank 2 has no tokens
    xs = [g["x"][r * Tr:(r + 1) * Tr].contiguous() for r in range(G)]
    xs[2] = g["x"][:0].contiguous()
    ys, stats = ep.ep_layer_forward_emulated(ops, xs, g["wg"], g["w1"], g["w3"], g["w2"], k, n, G)
    torch.cuda.synchronize()
    assert ys[2].shape == (0, d)
    for r in (0, 1, 3):
        _check_rank_output(ys[r], stats["topk_idx"][r], inp, w, slice(r * Tr, (r + 1) * Tr))
    # a bias that sends every token to experts 0 and 1 (both on rank 0): ranks 1-3 get no rows
    bias = torch.tensor([60.0, 50.0] + [0.0] * (n - 2), device=DEV)
    xs = [g["x"][r * Tr:(r + 1) * Tr].contiguous() for r in range(G)]
    ys, stats = ep.ep_layer_forward_emulated(ops, xs, g["wg"], g["w1"], g["w3"], g["w2"], k, n, G, bias)
    torch.cuda.synchronize()
    assert stats["expert_rows"] == [G * Tr * k, 0, 0, 0]
    f32 = f32_inputs(inp, w)
    for r in range(G):
        gi = stats["topk_idx"][r].cpu().numpy().astype(np.int64)
        assert np.all(np.sort(gi, 1) == [0, 1])
        rows = slice(r * Tr, (r + 1) * Tr)
        lref = oracle.router_logits(f32["x"][rows], f32["wg"], bias.cpu().numpy())
        yref = oracle.moe_layer(f32["x"][rows], f32["wg"], f32["w1"], f32["w3"], f32["w2"], k,
                                idx=gi, w=gate_weights_for(gi, lref))
        assert_close_rel(to_numpy_f32(ys[r]), yref, TOL["bf16"])


def test_empty_inputs(moe):
    """T = 0 through the layer, the decoder layer and the attention: nothing launched that
    reads an input, expert offsets all zero, empty outputs."""
    ws = moe.workspace(1, 256, 256, 8, 2, torch.bfloat16, DEV)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    wg = torch.zeros((256, 8), dtype=torch.bfloat16, device=DEV)
    w1 = torch.zeros((8, 256, 256), dtype=torch.bfloat16, device=DEV)
    off = torch.full((9,), -1, dtype=torch.int32, device=DEV)
    y = moe.moe_layer_forward(x, wg, w1, w1, w1, 2, ws, expert_offsets_out=off)
    assert y.shape == (0, 256) and off.cpu().tolist() == [0] * 9
    dws = moe.decoder_workspace(1, 256, 256, 8, 2, 2, 1, DEV)
    wq = torch.zeros((256, 256), dtype=torch.bfloat16, device=DEV)
    wk = torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV)
    y = moe.moe_decoder_layer_forward(x, wq, wk, wk, wq, wg, w1, w1, w1, 2, 2, 1, dws)
    assert y.shape == (0, 256)
    q = torch.empty((0, 2, 128), dtype=torch.bfloat16, device=DEV)
    kv = torch.empty((0, 1, 128), dtype=torch.bfloat16, device=DEV)
    out = moe.moe_attention_gqa(q, kv, kv, torch.zeros(256, dtype=torch.uint8, device=DEV))
    assert out.shape == (0, 2, 128)
    assert moe.moe_check_device_error(ws) == 0
