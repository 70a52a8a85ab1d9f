"""Out-of-bounds writes.  Every output buffer of the layer's calls (and the workspace) sits
between two 4 KB guard bands filled with a known byte; after the calls the bands must be
unchanged.  The shapes reach each GEMM form: the swapped form of a decode batch (many experts
without rows), the single-CTA form with ragged weight tiles (f = 320, d = 384: partial n-tiles
in both GEMMs) and the CTA-pair form with ragged 256-row tails; the backward and the attention
core run once each.  Nothing here is compared with the oracle: the other GPU tests do that
on the same kernels."""
import math

import numpy as np
import pytest

import workloads
from tests.helpers import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"
PAD = 4096
FILL = 0x5A


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_56_b300 as m
    m._native.lib()
    return m


class Guarded:
    """A tensor of `shape` placed between two guard bands inside one byte buffer."""

    def __init__(self, shape, dtype):
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.n = math.prod(shape) * itemsize
        self.raw = torch.full((2 * PAD + self.n,), FILL, dtype=torch.uint8, device=DEV)
        self.t = self.raw[PAD:PAD + self.n].view(dtype).view(shape)

    def workspace(self):
        """As a workspace: its 256-byte status header starts at zero, as every workspace's
        must; the rest keeps the fill."""
        self.t[:256].zero_()
        return self

    def check(self, what):
        torch.cuda.synchronize()
        lo = self.raw[:PAD].cpu().numpy()
        hi = self.raw[PAD + self.n:].cpu().numpy()
        assert (lo == FILL).all(), f"{what}: bytes written before the buffer"
        assert (hi == FILL).all(), f"{what}: bytes written after the buffer"


def _inputs(T, d, f, n, k, wid, skew=False):
    w = workloads.custom(T, d, f, n, k, "bf16", wid=wid, skew_bias=skew)
    inp = workloads.make_inputs(w)
    g = {t: to_device(inp[t], w, DEV) for t in ("x", "wg", "w1", "w3", "w2")}
    bias = torch.from_numpy(inp["bias"]).to(DEV) if inp["bias"] is not None else None
    return w, g, bias


@pytest.mark.parametrize("T,d,f,n,k,skew", [
    (20, 256, 384, 32, 2, False),      # swapped form; most experts without rows
    (300, 384, 320, 8, 2, True),       # single-CTA form, ragged weight tiles in both GEMMs
    (1500, 384, 320, 8, 2, True),      # CTA-pair form, ragged 256-row tails
])
def test_layer_calls_write_inside_their_buffers(moe, T, d, f, n, k, skew):
    w, g, bias = _inputs(T, d, f, n, k, 1300 + T, skew)
    A = T * k
    bf = torch.bfloat16
    ws = Guarded((moe.moe_workspace_size(T, d, f, n, k, bf),), torch.uint8).workspace()
    idx, wts = Guarded((T, k), torch.int32), Guarded((T, k), torch.float32)
    logits = Guarded((T, n), torch.float32)
    off, perm, inv = Guarded((n + 1,), torch.int32), Guarded((A,), torch.int32), Guarded((A,), torch.int32)
    h, yp, y = Guarded((A, f), bf), Guarded((A, d), bf), Guarded((T, d), bf)
    y2, idx2, off2 = Guarded((T, d), bf), Guarded((T, k), torch.int32), Guarded((n + 1,), torch.int32)

    moe.moe_router_topk(g["x"], g["wg"], k, bias, want_logits=True, topk_idx=idx.t, topk_w=wts.t,
                        logits=logits.t)
    moe.moe_permute(idx.t, n, ws.t, expert_offsets=off.t, perm=perm.t, inv_perm=inv.t)
    moe.moe_expert_up(g["x"], perm.t, off.t, g["w1"], g["w3"], k, ws.t, h=h.t)
    moe.moe_expert_down(h.t, off.t, g["w2"], k, ws.t, y_perm=yp.t)
    moe.moe_combine(yp.t, inv.t, wts.t, g["x"], y=y.t)
    moe.moe_layer_forward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], k, ws.t, logit_bias=bias,
                          residual=g["x"], y=y2.t, topk_idx_out=idx2.t, expert_offsets_out=off2.t)
    assert moe.moe_check_device_error(ws.t) == 0
    for name, buf in [("workspace", ws), ("topk_idx", idx), ("topk_w", wts), ("logits", logits),
                      ("expert_offsets", off), ("perm", perm), ("inv_perm", inv), ("h", h),
                      ("y_perm", yp), ("y", y), ("layer y", y2), ("layer topk_idx", idx2),
                      ("layer expert_offsets", off2)]:
        buf.check(name)
    # the step-by-step calls and the whole layer agree
    assert torch.equal(y.t.view(torch.int16), y2.t.view(torch.int16))


def test_backward_and_attention_write_inside_their_buffers(moe):
    T, d, f, n, k = 300, 384, 320, 8, 2
    w, g, bias = _inputs(T, d, f, n, k, 1350, True)
    bf = torch.bfloat16
    dy = to_device(workloads.make_inputs(w, tensors=("dy",))["dy"], w, DEV)
    bws = Guarded((moe.moe_backward_workspace_size(T, d, f, n, k, bf),), torch.uint8).workspace()
    dx, dwg = Guarded((T, d), bf), Guarded((d, n), torch.float32)
    dw1, dw3, dw2 = Guarded((n, f, d), bf), Guarded((n, f, d), bf), Guarded((n, d, f), bf)
    db = Guarded((n,), torch.float32)
    moe.moe_layer_backward(g["x"], g["wg"], g["w1"], g["w3"], g["w2"], k, dy, bws.t,
                           logit_bias=bias, want_dbias=True, dx=dx.t, dw_gate=dwg.t, dw1=dw1.t,
                           dw3=dw3.t, dw2=dw2.t, dlogit_bias=db.t)
    assert moe.moe_check_device_error(bws.t) == 0
    for name, buf in [("backward workspace", bws), ("dx", dx), ("dw_gate", dwg), ("dw1", dw1),
                      ("dw3", dw3), ("dw2", dw2), ("dlogit_bias", db)]:
        buf.check(name)

    # attention core: 2 sequences of 200 tokens (a ragged last query and key tile in each)
    Ta, hq, hkv = 400, 4, 2
    rng = np.random.default_rng(5)
    q = torch.from_numpy(rng.standard_normal((Ta, hq, 128), dtype=np.float32)).to(DEV).to(bf)
    kk = torch.from_numpy(rng.standard_normal((Ta, hkv, 128), dtype=np.float32)).to(DEV).to(bf)
    v = torch.from_numpy(rng.standard_normal((Ta, hkv, 128), dtype=np.float32)).to(DEV).to(bf)
    aws = Guarded((256,), torch.uint8).workspace()   # the attention needs only the header
    out = Guarded((Ta, hq, 128), bf)
    moe.moe_attention_gqa(q, kk, v, aws.t, seq_len=200, out=out.t)
    assert moe.moe_check_device_error(aws.t) == 0
    out.check("attention out")
    aws.check("attention workspace")
