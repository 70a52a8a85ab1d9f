"""One decoder layer on the GPU (moe_decoder_layer_forward: RMSNorm, the q/k/v projections
on the grouped tensor-core GEMM with one group, causal GQA attention, the output projection
and residual, then RMSNorm and the MoE layer with its residual) against the oracle's
composition of attention_gqa and the MoE layer, in fp64 on the same bf16 inputs.
Tolerance: max|y - y_ref| <= 2e-2 * max|y_ref| over the tokens whose MoE routing matches;
tokens that route differently must be near ties of the oracle's logits within the band the
bf16 roundings before the router allow (derived as in the stacked-layer test)."""
import numpy as np
import pytest

import oracle
import workloads
from tests.helpers import TOL, assert_close_rel

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


def _bf16(rng, shape, scale):
    bits = workloads.bf16_round_bits((rng.standard_normal(shape) * scale).astype(np.float32))
    return bits, workloads.bf16_bits_to_f32(bits).astype(np.float64)


CASES = [
    # T, hq, hkv, f, n, k, seq_len, skew
    (300, 4, 2, 384, 8, 2, 0, False),
    (520, 8, 2, 256, 8, 2, 256, True),     # two sequences of 256 and a tail of 8
    (96, 2, 1, 128, 4, 1, 0, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{}-hq{}-hkv{}-f{}-n{}-k{}-s{}".format(*c[:7]))
def test_decoder_layer_matches_oracle(moe, case):
    T, hq, hkv, f, n, k, seq, skew = case
    d = hq * 128
    rng = np.random.default_rng(T + hq)
    hb, h = _bf16(rng, (T, d), 1.0)
    wqb, wq = _bf16(rng, (hq * 128, d), d ** -0.5)
    wkb, wk = _bf16(rng, (hkv * 128, d), d ** -0.5)
    wvb, wv = _bf16(rng, (hkv * 128, d), d ** -0.5)
    wob, wo = _bf16(rng, (d, hq * 128), (hq * 128) ** -0.5)
    wgb, wg = _bf16(rng, (d, n), 0.02)
    w1b, w1 = _bf16(rng, (n, f, d), d ** -0.5)
    w3b, w3 = _bf16(rng, (n, f, d), d ** -0.5)
    w2b, w2 = _bf16(rng, (n, d, f), f ** -0.5)
    bias = workloads.logit_bias_vector(n) if skew else None
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(DEV)
    ws = moe.decoder_workspace(T, d, f, n, k, hq, hkv, DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    y = moe.moe_decoder_layer_forward(dev(hb), dev(wqb), dev(wkb), dev(wvb), dev(wob), dev(wgb),
                                      dev(w1b), dev(w3b), dev(w2b), k, hq, hkv, ws, seq_len=seq,
                                      logit_bias=None if bias is None else torch.from_numpy(bias).to(DEV),
                                      topk_idx_out=idx)
    assert moe.moe_check_device_error(ws) == 0
    yref, lref = oracle.decoder_layer(h, wq, wk, wv, wo, wg, w1, w3, w2, k, hq, hkv, seq, bias=bias,
                                      with_logits=True)
    gi = idx.cpu().numpy().astype(np.int64)
    same = np.all(np.sort(gi, 1) == np.sort(oracle.topk_select(lref, k), 1), axis=1)
    # the router input x2 = RMSNorm(h1) reaches the GPU after four bf16 roundings (q/k/v, the
    # attention output, h1, x2), each moving logit e by a random amount of std
    # 2^-9/sqrt(3) * ||x2 * W_g[:, e]||; differing choices must lie within 5 sigma of a tie
    x2 = oracle.rmsnorm(h)   # the router input's scale (unit rms); its exact value is not needed
    sigma = 2.0 ** -9 / np.sqrt(3) * np.sqrt(((x2[:, :, None] * wg[None]) ** 2).sum(1)).max(1)
    band = 5 * sigma * 4
    kth = np.sort(lref, 1)[:, ::-1][:, k - 1]
    chosen = np.take_along_axis(lref, gi, axis=1)
    assert np.all(chosen[~same] >= kth[~same, None] - band[~same, None]), "a routing flip outside the band"
    assert same.sum() >= 0.9 * T, f"{(~same).sum()} of {T} tokens routed differently"
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert_close_rel(got[same], yref[same], TOL["bf16"])


def test_decoder_layer_rejects_fp32_and_odd_sizes(moe):
    from sparse_mixture_experts_56_b300 import _native
    fake = 4096
    lib = _native.lib()
    # fp32 storage: the attention and projections are bf16 tensor-core kernels only
    st = lib.moe_decoder_layer_forward(fake, fake, fake, fake, fake, fake, None, fake, fake, fake,
                                       64, 256, 256, 8, 2, 2, 1, 0, 1e-5, 0, fake, None, fake, 1 << 30, None)
    assert st == 2
    # d not a multiple of 64
    st = lib.moe_decoder_layer_forward(fake, fake, fake, fake, fake, fake, None, fake, fake, fake,
                                       64, 200, 256, 8, 2, 2, 1, 0, 1e-5, 1, fake, None, fake, 1 << 30, None)
    assert st == 2
