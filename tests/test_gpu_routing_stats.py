"""GPU parity of the routing-statistics kernel (expert load and the repetition of expert
choices between consecutive tokens) against the oracle: integer results, bit-exact."""
import numpy as np
import pytest

import oracle
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


def _random_idx(T, n, k, seed, skew=0.0):
    """k distinct experts per token (random permutation prefix), optionally with runs of
    repeated choices so that the pair counters see both outcomes often."""
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, n)), axis=1)[:, :k]
    if skew > 0 and T > 1:
        rep = rng.random(T) < skew
        rep[0] = False
        for t in np.flatnonzero(rep):
            idx[t] = idx[t - 1]
    return np.ascontiguousarray(idx.astype(np.int32))


CASES = [
    # (T, n, k, seq_len, skew)
    (0, 8, 2, 0, 0.0),
    (1, 8, 2, 0, 0.0),
    (2, 8, 2, 0, 0.0),
    (64, 8, 2, 0, 0.3),
    (4097, 8, 2, 4096, 0.3),       # two sequences, ragged tail
    (2048, 8, 2, 0, 0.28),         # largest single-block case
    (2049, 8, 2, 1000, 0.28),      # first multi-block case
    (16384, 8, 2, 0, 0.28),        # the skewed workload's batch size
    (70001, 8, 2, 8192, 0.1),      # several blocks per SM, ragged sequences
    (500, 32, 4, 7, 0.2),          # n = 32 (full bit mask)
    (333, 5, 5, 0, 0.0),           # K = n: every pair shares an expert
    (257, 8, 1, 1, 0.5),           # seq_len 1: no pairs at all
    (1000, 1, 1, 0, 0.0),          # one expert
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{}-n{}-k{}-s{}".format(*c[:4]))
def test_routing_stats_bit_exact(moe, case):
    T, n, k, seq, skew = case
    idx = _random_idx(T, n, k, seed=T * 31 + n, skew=skew)
    gi = torch.from_numpy(idx).to(DEV) if T else torch.empty((0, k), dtype=torch.int32, device=DEV)
    counts = torch.full((n,), -7, dtype=torch.int64, device=DEV)      # overwritten, not added to
    pairs = torch.full((3,), -7, dtype=torch.int64, device=DEV)
    moe.moe_routing_stats(gi, n, seq, expert_counts=counts, pair_counts=pairs)
    torch.cuda.synchronize()
    c_ref, p_ref, f1_ref, fa_ref = oracle.routing_statistics(idx.reshape(T, k), n, seq)
    assert counts.cpu().tolist() == c_ref.tolist()
    assert pairs.cpu().tolist() == [p_ref, f1_ref, fa_ref]
    if k == n and p_ref:
        assert fa_ref == p_ref


def test_routing_stats_of_the_router_output(moe):
    """Statistics of the GPU router's own selections on a skewed Mixtral-shaped batch: the
    counts agree with the grouping's offsets and the pair counts with the oracle run on
    the same selections; called twice in a row with the same result."""
    w = workloads.custom(2048, 4096, 8, 8, 2, "bf16", wid=210, skew_bias=True)
    inp = workloads.make_inputs(w, tensors=("x", "wg"))
    x, wg = to_device(inp["x"], w, DEV), to_device(inp["wg"], w, DEV)
    bias = torch.from_numpy(inp["bias"]).to(DEV)
    idx, _, _ = moe.moe_router_topk(x, wg, 2, bias)
    ws = moe.workspace(2048, 64, 64, 8, 2, torch.bfloat16, DEV)
    offsets, _, _ = moe.moe_permute(idx, 8, ws)
    c1, p1 = moe.moe_routing_stats(idx, 8, 512)
    c2, p2 = moe.moe_routing_stats(idx, 8, 512)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    c_ref, *pr = oracle.routing_statistics(gi, 8, 512)
    assert c1.cpu().tolist() == c_ref.tolist() == np.diff(offsets.cpu().numpy()).tolist()
    assert p1.cpu().tolist() == pr
    assert c2.cpu().tolist() == c1.cpu().tolist() and p2.cpu().tolist() == p1.cpu().tolist()


def test_routing_stats_skips_indices_out_of_range(moe):
    idx = np.array([[0, 1], [1, 8], [-1, 2], [2, 3]], dtype=np.int32)
    counts, pairs = moe.moe_routing_stats(torch.from_numpy(idx).to(DEV), 8)
    torch.cuda.synchronize()
    # out-of-range entries are not counted; first choices are compared as stored;
    # the shared-expert test sees {0,1}&{1} yes, {1}&{2} no, {2}&{2,3} yes
    assert counts.cpu().tolist() == [1, 2, 2, 1, 0, 0, 0, 0]
    assert pairs.cpu().tolist() == [3, 0, 2]


def test_routing_stats_counts_every_slot(moe):
    """A row that repeats an expert (not a TopK output, but a valid input) counts it once per
    slot, as the oracle's per-assignment histogram does."""
    rng = np.random.default_rng(5)
    idx = rng.integers(0, 4, size=(3000, 3)).astype(np.int32)
    counts, pairs = moe.moe_routing_stats(torch.from_numpy(idx).to(DEV), 4, 100)
    torch.cuda.synchronize()
    c_ref, *pr = oracle.routing_statistics(idx, 4, 100)
    assert counts.cpu().tolist() == c_ref.tolist()
    assert pairs.cpu().tolist() == pr
