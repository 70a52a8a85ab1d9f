"""The layer's calls inside CUDA graphs: moe_layer_forward and moe_layer_backward are stream-
ordered with no host synchronisation, so a captured sequence replays them; the replay on new
inputs (copied into the captured buffers) must equal an eager call bit for bit.  The first
call on a device (which sets kernel attributes and queries occupancy) happens before capture,
as the header asks."""
import numpy as np
import pytest

import workloads
from tests.helpers import to_device

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


@pytest.mark.parametrize("T", [32, 2100])
def test_forward_and_backward_replay_in_a_graph(moe, T):
    d, f, n, k = 256, 384, 8, 2
    w = workloads.custom(T, d, f, n, k, "bf16", wid=800 + T, skew_bias=True)
    inp = workloads.make_inputs(w, tensors=("x", "wg", "w1", "w3", "w2", "dy"))
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2", "dy")}
    bias = torch.from_numpy(inp["bias"]).to(DEV)
    ws = moe.workspace(T, d, f, n, k, torch.bfloat16, DEV)
    bws = moe.backward_workspace(T, d, f, n, k, torch.bfloat16, DEV)
    x_static, dy_static = g["x"].clone(), g["dy"].clone()
    y_static = torch.empty_like(x_static)
    outs = {"dx": torch.empty_like(x_static),
            "dw_gate": torch.empty((d, n), dtype=torch.float32, device=DEV),
            "dw1": torch.empty_like(g["w1"]), "dw3": torch.empty_like(g["w3"]),
            "dw2": torch.empty_like(g["w2"])}

    def body():
        moe.moe_layer_forward(x_static, g["wg"], g["w1"], g["w3"], g["w2"], k, ws,
                              logit_bias=bias, y=y_static)
        moe.moe_layer_backward(x_static, g["wg"], g["w1"], g["w3"], g["w2"], k, dy_static, bws,
                               logit_bias=bias, **outs)

    body()                                   # first call outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    # new inputs into the captured buffers, replay, compare with eager calls on them
    rng = np.random.default_rng(T)
    x_new = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(DEV).to(torch.bfloat16)
    dy_new = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(DEV).to(torch.bfloat16)
    x_static.copy_(x_new)
    dy_static.copy_(dy_new)
    graph.replay()
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0 and moe.moe_check_device_error(bws) == 0
    ws2 = moe.workspace(T, d, f, n, k, torch.bfloat16, DEV)
    y_eager = moe.moe_layer_forward(x_new, g["wg"], g["w1"], g["w3"], g["w2"], k, ws2, logit_bias=bias)
    ge = moe.moe_layer_backward(x_new, g["wg"], g["w1"], g["w3"], g["w2"], k, dy_new,
                                moe.backward_workspace(T, d, f, n, k, torch.bfloat16, DEV),
                                logit_bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(y_static.view(torch.int16), y_eager.view(torch.int16))
    for key in outs:
        a, b = outs[key], ge[key]
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), key


def test_decoder_layer_replays_in_a_graph(moe):
    """moe_decoder_layer_forward is stream-ordered with no host synchronisation: a captured
    call replays on new inputs bit for bit like an eager call."""
    T, hq, hkv, f, n, k = 384, 4, 2, 256, 8, 2
    d = hq * 128
    rng = np.random.default_rng(31)
    t = lambda shape, s: (torch.from_numpy((rng.standard_normal(shape) * s).astype(np.float32))
                          .to(torch.bfloat16).to(DEV))
    wq, wk, wv = t((hq * 128, d), d ** -0.5), t((hkv * 128, d), d ** -0.5), t((hkv * 128, d), d ** -0.5)
    wo, wg = t((d, hq * 128), (hq * 128) ** -0.5), t((d, n), 0.02)
    w1, w3, w2 = t((n, f, d), d ** -0.5), t((n, f, d), d ** -0.5), t((n, d, f), f ** -0.5)
    ws = moe.decoder_workspace(T, d, f, n, k, hq, hkv, DEV)
    h_static = t((T, d), 1.0)
    y_static = torch.empty_like(h_static)

    def body():
        moe.moe_decoder_layer_forward(h_static, wq, wk, wv, wo, wg, w1, w3, w2, k, hq, hkv, ws,
                                      seq_len=200, y=y_static)

    body()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    h_new = t((T, d), 1.0)
    h_static.copy_(h_new)
    graph.replay()
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0
    y_eager = moe.moe_decoder_layer_forward(h_new, wq, wk, wv, wo, wg, w1, w3, w2, k, hq, hkv,
                                            moe.decoder_workspace(T, d, f, n, k, hq, hkv, DEV),
                                            seq_len=200)
    torch.cuda.synchronize()
    assert torch.equal(y_static.view(torch.int16), y_eager.view(torch.int16))
