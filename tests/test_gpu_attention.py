"""GPU parity of the causal grouped-query attention kernel against the fp64 oracle: head
dimension 128, query / key-value head ratios 4 (the pages' 32 / 8), 1 and 8, single and
multiple sequences with ragged ends (query and key blocks of 128), and one token.
Tolerance: max|o - o_ref| <= 2e-2 * max|o_ref| (bf16 inputs and P, fp32 accumulation)."""
import numpy as np
import pytest

import oracle
import workloads

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


def _bf16(rng, shape):
    bits = workloads.bf16_round_bits(rng.standard_normal(shape).astype(np.float32))
    return bits, workloads.bf16_bits_to_f32(bits).astype(np.float64)


CASES = [
    # (T, hq, hkv, seq_len)
    (300, 8, 2, 0),        # one ragged sequence: 3 query blocks, partial last block
    (256, 4, 4, 0),        # plain multi-head attention
    (1000, 8, 2, 300),     # four sequences of 300 (last 100), blocks straddle nothing
    (640, 32, 8, 0),       # the pages' head counts
    (130, 8, 1, 0),        # one key-value head
    (1, 4, 1, 0),          # a single token attends to itself
    (2048, 32, 8, 2048),   # a long sequence: 16 key blocks for the last query block
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{}-hq{}-hkv{}-s{}".format(*c))
def test_attention_matches_oracle(moe, case):
    T, hq, hkv, seq = case
    rng = np.random.default_rng(T * 7 + hq)
    qb, q = _bf16(rng, (T, hq, 128))
    kb, k = _bf16(rng, (T, hkv, 128))
    vb, v = _bf16(rng, (T, hkv, 128))
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    out = moe.moe_attention_gqa(dev(qb), dev(kb), dev(vb), ws, seq)
    assert moe.moe_check_device_error(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    ref = oracle.attention_gqa(q, k, v, seq)
    err = np.max(np.abs(got - ref))
    assert np.all(np.isfinite(got))
    assert err <= 2e-2 * np.max(np.abs(ref)), f"max err {err:.3e} vs scale {np.max(np.abs(ref)):.3e}"


def test_attention_is_deterministic(moe):
    T, hq, hkv = 700, 8, 2
    rng = np.random.default_rng(5)
    qb, _ = _bf16(rng, (T, hq, 128))
    kb, _ = _bf16(rng, (T, hkv, 128))
    vb, _ = _bf16(rng, (T, hkv, 128))
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    a = moe.moe_attention_gqa(dev(qb), dev(kb), dev(vb), ws)
    b = moe.moe_attention_gqa(dev(qb), dev(kb), dev(vb), ws)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_attention_timeout_path_reports_and_recovers(moe):
    """A wait limit of 1 ns makes the attention's roles give up at their first wait that is not
    already satisfied (barriers, and the exchange of row maxima between the two threads of a
    row): the kernel must stop cleanly (status MOE_ERR_TIMEOUT), drain what it issued, free
    its TMEM, and the next call must be correct."""
    T, hq, hkv = 1024, 32, 8
    rng = np.random.default_rng(11)
    qb, q = _bf16(rng, (T, hq, 128))
    kb, k = _bf16(rng, (T, hkv, 128))
    vb, v = _bf16(rng, (T, hkv, 128))
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    try:
        moe.moe_set_wait_limit_ns(1)
        moe.moe_attention_gqa(dev(qb), dev(kb), dev(vb), ws)
        st = moe.moe_check_device_error(ws)
    finally:
        moe.moe_set_wait_limit_ns(0)
    # 1024 tokens x 32 heads span many CTAs and key blocks: the first MMA of every CTA waits
    # for a TMA copy that cannot have landed within 1 ns, so the limit must fire
    assert st == 5, f"status {st}, expected MOE_ERR_TIMEOUT (5)"
    out = moe.moe_attention_gqa(dev(qb), dev(kb), dev(vb), ws)
    assert moe.moe_check_device_error(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    ref = oracle.attention_gqa(q, k, v)
    assert np.max(np.abs(got - ref)) <= 2e-2 * np.max(np.abs(ref))


@pytest.mark.slow
def test_attention_32k_context(moe):
    """The pages' full dense 32k context: one 32768-token sequence with 32 / 8 heads.  Rows are
    checked where the oracle is cheap: all rows of the first 1024 tokens (the causal prefix
    is a problem of its own), and sampled late rows, each against the plain definition over
    its whole prefix."""
    T, hq, hkv = 32768, 32, 8
    rng = np.random.default_rng(32768)
    qb, q = _bf16(rng, (T, hq, 128))
    kb, k = _bf16(rng, (T, hkv, 128))
    vb, v = _bf16(rng, (T, hkv, 128))
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    out = moe.moe_attention_gqa(dev(qb), dev(kb), dev(vb), ws)
    assert moe.moe_check_device_error(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    pre = 1024
    ref = oracle.attention_gqa(q[:pre], k[:pre], v[:pre])
    assert np.max(np.abs(got[:pre] - ref)) <= 2e-2 * np.max(np.abs(ref))
    rows = np.concatenate([[T - 1, T - 128, T // 2], rng.choice(np.arange(pre, T), size=13, replace=False)])
    ref_rows = oracle.attention_gqa_rows(q, k, v, rows)
    for r, i in enumerate(rows):
        assert np.max(np.abs(got[i] - ref_rows[r])) <= 2e-2 * np.max(np.abs(ref_rows[r])), i


def test_attention_rescales_running_output(moe):
    """Scores that grow along the sequence: key row s is scaled by (1 + s/64), so every later
    key block holds scores several times larger than the earlier ones and the running row
    maximum passes the kernel's lazy-rescaling threshold (2^8 in the exp2 domain, about 5.5 in
    natural units) again and again; the output accumulated in TMEM must then be rescaled
    before the next P·V adds to it.  Checked against the oracle at every row."""
    T, hq, hkv = 1024, 8, 2
    rng = np.random.default_rng(64)
    qb, q = _bf16(rng, (T, hq, 128))
    grow = (1.0 + np.arange(T) / 64.0)[:, None, None]
    kf = rng.standard_normal((T, hkv, 128)) * grow
    kb = workloads.bf16_round_bits(kf.astype(np.float32))
    k = workloads.bf16_bits_to_f32(kb).astype(np.float64)
    vb, v = _bf16(rng, (T, hkv, 128))
    # the premise: for rows past the first block, a later key block's maximum score beats the
    # first block's by more than 8 / log2(e) natural units
    i = T - 1
    sc = k[:i + 1, 0] @ q[i, 0] / np.sqrt(128.0)       # query head 0 reads key-value head 0
    assert sc[128:].max() - sc[:128].max() > 8.0 / np.log2(np.e)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    out = moe.moe_attention_gqa(dev(qb), dev(kb), dev(vb), ws)
    assert moe.moe_check_device_error(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    ref = oracle.attention_gqa(q, k, v)
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - ref))
    assert err <= 2e-2 * np.max(np.abs(ref)), f"max err {err:.3e} vs scale {np.max(np.abs(ref)):.3e}"
