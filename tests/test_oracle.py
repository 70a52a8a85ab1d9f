"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each ``check_*`` function takes the oracle module, so that ``test_pins_catch_mutations``
can run the same checks against deliberately broken copies of the oracle (mistakes
planted on the CPU only) and show that every planted mistake fails at least one pin.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.ep as ep_oracle
import oracle.moe as moe_oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _expr(s):
    """Closed-form values stored in fixtures: integers, decimals, fractions, log(q)."""
    s = s.strip()
    if s.startswith("log(") and s.endswith(")"):
        return math.log(float(Fraction(s[4:-1])))
    return float(Fraction(s))


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ------------------------------------------------------------------------------------------
# checks (module-parameterised)
# ------------------------------------------------------------------------------------------
def check_worked_example(o):
    fx = _load("gate_worked_example.json")
    l = np.array([[_expr(v) for v in fx["logits"]]])
    G = o.masked_softmax(o.topk_mask(l, fx["k"]))
    idx = o.topk_select(l, fx["k"])
    assert idx.tolist() == [fx["expected_idx"]]
    np.testing.assert_allclose(G[0], [_expr(v) for v in fx["expected_G"]], rtol=0, atol=1e-15)


def check_gate_invariants(o):
    for n, k, seed in [(8, 2, 0), (8, 1, 1), (8, 8, 2), (5, 3, 3), (32, 2, 4), (1, 1, 5)]:
        x = _rand((64, 16), seed)
        wg = _rand((16, n), seed + 100, 0.5)
        idx, w, G, l = o.gate(x, wg, k)
        assert G.shape == (64, n) and idx.shape == (64, k)
        assert np.all(G >= 0)
        assert np.all(np.count_nonzero(G, axis=1) == k)           # exactly K non-zeros
        np.testing.assert_allclose(G.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        # the non-zero entries sit exactly at the selected experts
        nz = [sorted(np.flatnonzero(r).tolist()) for r in G]
        assert nz == [sorted(r) for r in idx.tolist()]
        # slots are in descending logit order
        kept = np.take_along_axis(l, idx, axis=1)
        assert np.all(np.diff(kept, axis=1) <= 0)


def _rank_count_topk(row, k):
    """Brute force: expert i is selected iff fewer than k experts beat it, where j
    beats i when l_j > l_i, or l_j == l_i and j < i.  Returned in beat-count order."""
    n = len(row)
    beaten_by = [sum(1 for j in range(n) if row[j] > row[i] or (row[j] == row[i] and j < i))
                 for i in range(n)]
    chosen = [i for i in range(n) if beaten_by[i] < k]
    return sorted(chosen, key=lambda i: beaten_by[i])


def check_topk_bruteforce(o):
    vals = [0.0, 1.0, 2.0]
    for n in (1, 2, 3, 4):
        rows = np.array(list(itertools.product(vals, repeat=n)), dtype=np.float64)
        for k in range(1, n + 1):
            got = o.topk_select(rows, k)
            want = np.array([_rank_count_topk(r, k) for r in rows])
            assert np.array_equal(got, want), (n, k)
    # random, continuous, n=8
    rows = _rand((500, 8), 7)
    for k in (1, 2, 3, 8):
        assert np.array_equal(o.topk_select(rows, k), np.array([_rank_count_topk(r, k) for r in rows]))


def check_softmax_order_equivalence(o):
    l = _rand((200, 8), 11, 2.0)
    for k in (1, 2, 4, 8):
        G = o.masked_softmax(o.topk_mask(l, k))
        # independent route: torch softmax over all n, zero outside the top-k, renormalise
        p = torch.softmax(torch.from_numpy(l), dim=1)
        top = torch.topk(p, k, dim=1).indices
        keep = torch.zeros_like(p).scatter(1, top, 1.0)
        ref = (p * keep) / (p * keep).sum(dim=1, keepdim=True)
        np.testing.assert_allclose(G, ref.numpy(), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(o.gate_softmax_then_topk(l, k), ref.numpy(), rtol=1e-13, atol=1e-15)


def _torch_swiglu(x, w1e, w3e, w2e):
    x, w1e, w3e, w2e = (torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (x, w1e, w3e, w2e))
    return F.linear(F.silu(F.linear(x, w1e)) * F.linear(x, w3e), w2e).numpy()


def check_single_expert_is_plain_ffn(o):
    T, d, f = 12, 24, 40
    x = _rand((T, d), 21)
    wg = _rand((d, 1), 22)
    w1 = _rand((1, f, d), 23, d ** -0.5)
    w3 = _rand((1, f, d), 24, d ** -0.5)
    w2 = _rand((1, d, f), 25, f ** -0.5)
    y = o.moe_layer(x, wg, w1, w3, w2, 1)
    np.testing.assert_allclose(y, _torch_swiglu(x, w1[0], w3[0], w2[0]), rtol=1e-12, atol=1e-13)


def check_k_equals_n_is_dense_softmax_mixture(o):
    T, d, f, n = 10, 16, 20, 4
    x = _rand((T, d), 31)
    wg = _rand((d, n), 32, 0.3)
    w1 = _rand((n, f, d), 33, d ** -0.5)
    w3 = _rand((n, f, d), 34, d ** -0.5)
    w2 = _rand((n, d, f), 35, f ** -0.5)
    y = o.moe_layer(x, wg, w1, w3, w2, n)
    p = torch.softmax(torch.from_numpy(x) @ torch.from_numpy(wg), dim=1).numpy()
    ref = sum(p[:, i:i + 1] * _torch_swiglu(x, w1[i], w3[i], w2[i]) for i in range(n))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


def check_sparse_equals_dense(o):
    w = workloads.workload(1)
    inp = workloads.make_inputs(w)
    args = [workloads.as_f32(inp[t], w) for t in ("x", "wg", "w1", "w3", "w2")]
    y = o.moe_layer(*args, w.k)
    yd = o.moe_layer_dense(*args, w.k)
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12)
    # the dense sum with torch ops over all experts and the page's G
    _, _, G, _ = o.gate(args[0], args[1], w.k)
    ref = sum(G[:, i:i + 1] * _torch_swiglu(args[0], args[2][i], args[3][i], args[4][i]) for i in range(w.n))
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)


def check_grouping(o):
    rng = np.random.default_rng(41)
    cases = [
        (rng.integers(0, 8, size=(64, 2)), 8),
        (np.zeros((33, 2), dtype=np.int64), 8),                        # every token to expert 0
        (np.array([[7, 3]] * 5), 8),                                   # empty experts around
        (rng.integers(0, 3, size=(17, 3)), 5),                         # ragged, experts 3,4 empty
        (np.zeros((0, 2), dtype=np.int64), 4),                         # no tokens
        (rng.integers(0, 32, size=(1000, 2)), 32),
    ]
    for idx, n in cases:
        off, perm, inv = o.group_by_expert(idx, n)
        flat = idx.reshape(-1).tolist()
        A = len(flat)
        # brute force by counting
        counts = [flat.count(e) for e in range(n)]
        assert off.tolist() == [sum(counts[:e]) for e in range(n + 1)]
        want = [a for e in range(n) for a in range(A) if flat[a] == e]
        assert perm.tolist() == want
        assert sorted(perm.tolist()) == list(range(A))                  # bijection
        assert all(inv[perm[p]] == p for p in range(A))
        # permute rows then unpermute is the identity
        X = rng.standard_normal((A, 3))
        assert np.array_equal(X[perm][inv], X)


def check_silu(o):
    z = np.concatenate([np.linspace(-40, 40, 2001), [0.0, -1e-300, 1e-300, -745.0, 710.0]])
    np.testing.assert_allclose(o.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-300)
    # odd-part identity: silu(z) - silu(-z) = z
    np.testing.assert_allclose(o.silu(z) - o.silu(-z), z, rtol=1e-13, atol=1e-13)
    # sigmoid(ln 3) = 3/4
    assert abs(o.silu(np.array([math.log(3)]))[0] - 0.75 * math.log(3)) < 1e-15


def check_bias_enters_before_topk(o):
    # logits 0.2 > 0.1 > 0 without bias; a bias of +1 on expert 2 moves it to the top
    x = np.array([[1.0]])
    wg = np.array([[0.2, 0.1, 0.0]])
    b = np.array([0.0, 0.0, 1.0])
    idx, w, G, l = o.gate(x, wg, 2, b)
    assert idx.tolist() == [[2, 0]]
    e = math.exp(1.0 - 0.2)
    np.testing.assert_allclose(w[0], [e / (1 + e), 1 / (1 + e)], rtol=1e-14)
    assert o.gate(x, wg, 2)[0].tolist() == [[0, 1]]


def check_rmsnorm(o):
    h = _rand((9, 64), 51, 3.0)
    ref = F.rms_norm(torch.from_numpy(h), (64,), eps=1e-5).numpy()
    np.testing.assert_allclose(o.rmsnorm(h, 1e-5), ref, rtol=1e-13, atol=1e-14)
    # stacked layer = h + MoE(RMSNorm(h)) with a single always-on expert
    x = _rand((5, 8), 52)
    wg = np.ones((8, 1))
    w1, w3, w2 = _rand((1, 6, 8), 53), _rand((1, 6, 8), 54), _rand((1, 8, 6), 55)
    xn = F.rms_norm(torch.from_numpy(x), (8,), eps=1e-5).numpy()
    np.testing.assert_allclose(o.stacked_layer(x, wg, w1, w3, w2, 1), x + _torch_swiglu(xn, w1[0], w3[0], w2[0]),
                               rtol=1e-12, atol=1e-13)


def check_param_counts(o):
    fx = _load("param_counts.json")
    c = o.param_counts(fx["d"], fx["f"], fx["n"], fx["k"], fx["layers"], fx["heads"], fx["kv_heads"])
    # 32 * 8 * 3 * 4096 * 14336 and 32 * 2 * 3 * 4096 * 14336
    assert c["expert"] == 45_097_156_608 and c["active_expert"] == 11_274_289_152
    rest_total = fx["total_params_printed"] - (c["expert"] + c["attention"])
    rest_active = fx["active_params_printed"] - (c["active_expert"] + c["attention"])
    # what is left (embeddings, norms, router) is small, positive and the same in both counts
    assert 0 < rest_total < 0.6e9 and 0 < rest_active < 0.6e9
    assert abs(rest_total - rest_active) <= 2 * fx["printed_rounding"]


def check_locality_metric(o):
    assert o.consecutive_same_expert_rate(np.array([[0, 1], [0, 2], [1, 0], [1, 3], [1, 0]])) == 0.75
    rng = np.random.default_rng(61)
    r = o.consecutive_same_expert_rate(rng.integers(0, 8, size=(200_000, 2)))
    assert abs(r - 1 / 8) < 0.005          # the random-assignment rate of 12.5% for n = 8


def _pairs_bruteforce(idx, seq_len):
    """Plain loops over token pairs with Python sets (no NumPy): the routing-statistics
    definitions written out directly."""
    rows = [list(map(int, r)) for r in idx]
    pairs = same_first = same_any = 0
    for t in range(len(rows) - 1):
        if seq_len > 0 and (t + 1) % seq_len == 0:
            continue                      # t+1 starts a new sequence
        pairs += 1
        same_first += rows[t][0] == rows[t + 1][0]
        same_any += len(set(rows[t]) & set(rows[t + 1])) > 0
    return pairs, same_first, same_any


def check_routing_statistics(o):
    hand = np.array([[0, 1], [0, 2], [1, 0], [1, 3], [1, 0]])
    c, p, f1, fa = o.routing_statistics(hand, 4)
    assert c.tolist() == [4, 4, 1, 1] and (p, f1, fa) == (4, 3, 4)
    c, p, f1, fa = o.routing_statistics(hand, 4, seq_len=2)   # pairs (0,1) and (2,3) only
    assert (p, f1, fa) == (2, 2, 2)
    assert o.routing_statistics(hand[:1], 4)[1:] == (0, 0, 0)
    rng = np.random.default_rng(62)
    for n, k, T, seq in [(8, 2, 300, 0), (8, 2, 301, 37), (5, 3, 64, 8), (4, 1, 50, 7), (32, 4, 90, 1)]:
        idx = np.argsort(rng.random((T, n)), axis=1)[:, :k]
        c, p, f1, fa = o.routing_statistics(idx, n, seq_len=seq)
        assert (p, f1, fa) == _pairs_bruteforce(idx, seq)
        assert c.tolist() == [int(np.sum(idx == e)) for e in range(n)] and c.sum() == T * k
        if k == 1:
            assert f1 == fa
    # random routing: first choice repeats with probability 1/n, and two independent
    # K-subsets of n share an expert with probability 1 - C(n-K, K) / C(n, K)
    for n, k in [(8, 2), (8, 1), (6, 3)]:
        idx = np.argsort(rng.random((200_000, n)), axis=1)[:, :k]
        _, p, f1, fa = o.routing_statistics(idx, n)
        assert abs(f1 / p - 1 / n) < 0.005
        assert abs(fa / p - (1 - math.comb(n - k, k) / math.comb(n, k))) < 0.005


def _bwd_case(seed, T, d, f, n, k, margin=1e-2, scale=0.4):
    """Random layer whose TopK decisions all have a gap of at least ``margin`` (so small
    perturbations do not flip a selection)."""
    rng = np.random.default_rng(seed)
    while True:
        x = rng.standard_normal((T, d))
        wg = rng.standard_normal((d, n))
        bias = rng.standard_normal(n) * 0.1
        l = np.sort(x @ wg + bias, axis=1)[:, ::-1]
        if k == n or np.all(l[:, k - 1] - l[:, k] > margin):
            break
    w1 = rng.standard_normal((n, f, d)) * scale
    w3 = rng.standard_normal((n, f, d)) * scale
    w2 = rng.standard_normal((n, d, f)) * scale
    dy = rng.standard_normal((T, d))
    return x, wg, w1, w3, w2, bias, dy


def check_backward_finite_differences(o):
    """Every gradient entry against central differences of L = <dy, y> in fp64."""
    x, wg, w1, w3, w2, bias, dy = _bwd_case(70, 5, 6, 7, 4, 2)
    params = {"x": x, "wg": wg, "w1": w1, "w3": w3, "w2": w2, "bias": bias}

    def loss(p):
        return float(np.sum(dy * o.moe_layer(p["x"], p["wg"], p["w1"], p["w3"], p["w2"], 2,
                                             p["bias"])))
    g = o.moe_layer_backward(x, wg, w1, w3, w2, 2, dy, bias)
    names = {"x": "dx", "wg": "dwg", "w1": "dw1", "w3": "dw3", "w2": "dw2", "bias": "dbias"}
    eps = 1e-6
    for name, arr in params.items():
        num = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            p = {kk: v.copy() for kk, v in params.items()}
            p[name][i] += eps
            lp = loss(p)
            p[name][i] -= 2 * eps
            num[i] = (lp - loss(p)) / (2 * eps)
        np.testing.assert_allclose(g[names[name]], num, rtol=1e-6, atol=1e-7, err_msg=name)


def _torch_moe(x, wg, bias, w1, w3, w2, idx):
    """The layer restated with torch ops on a fixed selection, for autograd."""
    l = x @ wg + bias
    gw = torch.softmax(torch.gather(l, 1, idx), dim=1)
    y = torch.zeros_like(x)
    for slot in range(idx.shape[1]):
        e = idx[:, slot]
        a = torch.einsum("td,tfd->tf", x, w1[e])
        b = torch.einsum("td,tfd->tf", x, w3[e])
        o = torch.einsum("tf,tdf->td", F.silu(a) * b, w2[e])
        y = y + gw[:, slot:slot + 1] * o
    return y


def check_backward_autograd(o):
    """The whole backward against torch autograd of a torch restatement of the forward."""
    for seed, (T, d, f, n, k) in [(71, (40, 16, 24, 8, 2)), (72, (23, 8, 12, 5, 3)),
                                  (73, (17, 8, 8, 6, 1))]:
        x, wg, w1, w3, w2, bias, dy = _bwd_case(seed, T, d, f, n, k, margin=1e-6)
        g = o.moe_layer_backward(x, wg, w1, w3, w2, k, dy, bias)
        idx = torch.from_numpy(o.topk_select(x @ wg + bias, k))
        ts = [torch.from_numpy(a).requires_grad_(True) for a in (x, wg, bias, w1, w3, w2)]
        y = _torch_moe(*ts, idx)
        (y * torch.from_numpy(dy)).sum().backward()
        for name, t in zip(("dx", "dwg", "dbias", "dw1", "dw3", "dw2"), ts):
            np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=1e-10, atol=1e-11,
                                       err_msg=name)


def check_backward_special_cases(o):
    # K = 1: the gate is identically 1, so the router gets no gradient
    x, wg, w1, w3, w2, bias, dy = _bwd_case(74, 9, 8, 8, 4, 1)
    g = o.moe_layer_backward(x, wg, w1, w3, w2, 1, dy, bias)
    assert np.all(g["dlogits"] == 0) and np.all(g["dwg"] == 0)
    # the softmax Jacobian keeps the logit gradient of every token summing to zero
    x, wg, w1, w3, w2, bias, dy = _bwd_case(75, 30, 8, 8, 8, 3)
    g = o.moe_layer_backward(x, wg, w1, w3, w2, 3, dy, bias)
    np.testing.assert_allclose(g["dlogits"].sum(axis=1), 0.0, atol=1e-12)
    assert np.all(np.count_nonzero(g["dlogits"], axis=1) <= 3)
    # one expert, K = 1: the backward of a plain SwiGLU FFN (torch autograd of F.linear)
    x, wg, w1, w3, w2, bias, dy = _bwd_case(76, 12, 8, 10, 1, 1)
    g = o.moe_layer_backward(x, wg, w1, w3, w2, 1, dy)
    tx, t1, t3, t2 = (torch.from_numpy(a).requires_grad_(True) for a in (x, w1[0], w3[0], w2[0]))
    yt = F.linear(F.silu(F.linear(tx, t1)) * F.linear(tx, t3), t2)
    (yt * torch.from_numpy(dy)).sum().backward()
    np.testing.assert_allclose(g["dx"], tx.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dw1"][0], t1.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dw3"][0], t3.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dw2"][0], t2.grad.numpy(), rtol=1e-11, atol=1e-12)
    # SiLU'(z) against the symmetric difference of SiLU, and at 0 (= 1/2)
    z = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(o.silu_grad(z), (o.silu(z + 1e-6) - o.silu(z - 1e-6)) / 2e-6,
                               rtol=1e-6, atol=1e-8)
    assert o.silu_grad(np.array([0.0]))[0] == 0.5


def check_attention(o):
    rng = np.random.default_rng(80)
    # torch's scaled_dot_product_attention (causal) on key/value heads repeated per group
    for T, hq, hkv, dh, seq in [(37, 8, 2, 16, 0), (50, 4, 4, 8, 0), (45, 6, 3, 8, 16), (9, 4, 1, 32, 4)]:
        q = rng.standard_normal((T, hq, dh))
        k = rng.standard_normal((T, hkv, dh))
        v = rng.standard_normal((T, hkv, dh))
        out = o.attention_gqa(q, k, v, seq)
        S = T if seq == 0 else seq
        for s0 in range(0, T, S):
            sl = slice(s0, min(T, s0 + S))
            tq = torch.from_numpy(q[sl]).transpose(0, 1)                       # [hq, n, dh]
            tk = torch.from_numpy(k[sl]).transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
            tv = torch.from_numpy(v[sl]).transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
            ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True).transpose(0, 1)
            np.testing.assert_allclose(out[sl], ref.numpy(), rtol=1e-11, atol=1e-12)
    # the first token of every sequence sees only itself: o = v of its head group
    q = rng.standard_normal((24, 4, 8))
    k = rng.standard_normal((24, 2, 8))
    v = rng.standard_normal((24, 2, 8))
    out = o.attention_gqa(q, k, v, 8)
    for s0 in (0, 8, 16):
        for h in range(4):
            np.testing.assert_allclose(out[s0, h], v[s0, h // 2], rtol=0, atol=1e-14)
    # zero queries give equal weights: the mean of the causal prefix of v
    out = o.attention_gqa(np.zeros((12, 2, 8)), k[:12, :1], v[:12, :1], 0)
    for i in range(12):
        np.testing.assert_allclose(out[i, 0], v[:i + 1, 0].mean(axis=0), rtol=1e-13, atol=1e-14)


def check_near_tie_tokens(o):
    """Hand-built logits around the 1e-4 band, with binary-exact gaps (2^-14 = 6.1e-5 is
    inside the band, 2^-13 = 1.22e-4 outside), rows deliberately unsorted."""
    a, b = 2.0 ** -14, 2.0 ** -13
    # n = 4, k = 2: the set gap is between the 2nd and 3rd largest, the order gap between
    # the 1st and 2nd
    l2 = np.array([
        [0.5 - a, 0.0, 3.0, 0.5],        # set gap a            -> set tie
        [0.5 - b, 0.0, 3.0, 0.5],        # set gap b            -> none
        [-1.0, 0.5, -2.0, 0.5 + a],      # kept pair gap a      -> order tie
        [-1.0, 0.5, -2.0, 0.5 + b],      # kept pair gap b      -> none
        [0.0, 3.0, 2.0, 0.0 + a],        # 3rd/4th gap a only   -> none
        [1.0, 1.0, 1.0, 1.0],            # all equal            -> both
        [0.5 + a, 0.5, 0.5 - a, -9.0],   # both gaps a          -> both
    ])
    st, ot = o.near_tie_tokens(l2, 2)
    assert st.tolist() == [True, False, False, False, False, True, True]
    assert ot.tolist() == [False, False, True, False, False, True, True]
    # k = 3: order gaps (1st, 2nd) and (2nd, 3rd); the set gap (3rd, 4th)
    l3 = np.array([
        [5.0, 3.0, 3.0 - a, 0.0],        # 2nd/3rd gap a        -> order tie
        [5.0, 3.0, 1.0, 1.0 - a],        # 3rd/4th gap a        -> set tie only
        [5.0, 5.0 - b, 2.0, 0.0],        # gaps >= b            -> none
    ])
    st, ot = o.near_tie_tokens(l3, 3)
    assert st.tolist() == [False, True, False]
    assert ot.tolist() == [True, False, False]
    # k = n: the selected set cannot be in doubt; k = 1: no slot order to decide
    st, ot = o.near_tie_tokens(l2, 4)
    assert not st.any()
    st, ot = o.near_tie_tokens(l2, 1)
    assert not ot.any() and st.tolist() == [False, False, True, False, False, True, True]
    # a custom band
    st, _ = o.near_tie_tokens(np.array([[1.0, 0.75, 0.5]]), 1, eps=0.3)
    assert st.tolist() == [True]


def check_attention_rows(o):
    """The row-wise evaluation equals the whole-sequence one (itself pinned to torch SDPA
    above) at every row, across sequence boundaries and with grouped heads."""
    rng = np.random.default_rng(81)
    for T, hq, hkv, dh, seq in [(37, 8, 2, 16, 0), (45, 6, 3, 8, 16), (9, 4, 1, 32, 4)]:
        q = rng.standard_normal((T, hq, dh))
        k = rng.standard_normal((T, hkv, dh))
        v = rng.standard_normal((T, hkv, dh))
        full = o.attention_gqa(q, k, v, seq)
        rows = np.arange(T)[::-1]
        np.testing.assert_allclose(o.attention_gqa_rows(q, k, v, rows, seq), full[rows],
                                   rtol=1e-12, atol=1e-13)


def check_ep_plan(o):
    """Expert-parallel bookkeeping against the single-rank grouping: with G ranks of T tokens
    each, the rows a rank's expert receives, in the order the plan evaluates them, are the
    rows the single-rank grouping of all G*T tokens (rank s's tokens at s*T..) gives that
    expert; every assignment is sent exactly once; counts add up; G = 1 is the identity."""
    rng = np.random.default_rng(90)
    for G, T, n, k in [(1, 37, 8, 2), (2, 50, 8, 2), (4, 33, 8, 2), (8, 20, 8, 2), (2, 40, 4, 3),
                       (4, 0, 8, 2)]:
        idx = [rng.integers(0, n, (T, k)) for _ in range(G)]
        if T:
            idx[0][:, 0] = 0                                     # a crowded expert
        plans = ep_oracle.ep_exchange_plan(idx, n, G)
        E = n // G
        off_all, perm_all, _ = o.group_by_expert(np.concatenate(idx) if T else np.zeros((0, k), int), n)
        seen = set()
        for g, p in enumerate(plans):
            # brute-force counts
            for s in range(G):
                for j in range(E):
                    assert p["recv_counts"][s, j] == int(np.count_nonzero(idx[s] == g * E + j))
            assert p["send_counts"].tolist() == [
                int(np.count_nonzero((idx[g] >= h * E) & (idx[g] < (h + 1) * E))) for h in range(G)]
            R = int(p["recv_counts"].sum())
            assert p["local_offsets"][-1] == R and len(p["row_map"]) == R
            assert sorted(p["row_map"].tolist()) == list(range(R))
            for j in range(E):
                e = g * E + j
                rows = p["row_map"][p["local_offsets"][j]:p["local_offsets"][j + 1]]
                got = list(zip(p["recv_src"][rows].tolist(), p["recv_assign"][rows].tolist()))
                want = [divmod(int(a), T * k) for a in perm_all[off_all[e]:off_all[e + 1]]]
                assert got == want
                for sa in got:
                    assert idx[sa[0]].reshape(-1)[sa[1]] == e
                    seen.add(sa)
        assert len(seen) == G * T * k                            # each assignment sent once
        if G == 1:
            off, _, _ = o.group_by_expert(idx[0], n)
            assert plans[0]["row_map"].tolist() == list(range(T * k))
            assert plans[0]["local_offsets"].tolist() == off.tolist()
        assert ep_oracle.ep_load(plans).sum() == G * T * k
        # the receiver's regrouping from its counts alone is the plan's
        for p in plans:
            lo, rm, inv = ep_oracle.ep_regroup(p["recv_counts"])
            assert lo.tolist() == p["local_offsets"].tolist()
            assert rm.tolist() == p["row_map"].tolist()
            assert np.array_equal(rm[inv], np.arange(rm.size))
    # unequal batches per rank: the receive buffer is the sources' blocks in source order
    idx = [np.array([[1, 3], [0, 1]]), np.array([[3, 2]]), np.zeros((0, 2), int)]
    with pytest.raises(ValueError):
        ep_oracle.ep_exchange_plan(idx, 4, 3)                            # 4 experts over 3 ranks
    p = ep_oracle.ep_exchange_plan(idx + [np.array([[2, 0]])], 4, 4)
    assert p[1]["recv_src"].tolist() == [0, 0] and p[1]["recv_assign"].tolist() == [0, 3]
    assert p[3]["recv_src"].tolist() == [0, 1] and p[3]["recv_assign"].tolist() == [1, 0]
    assert p[0]["recv_counts"][:, 0].tolist() == [1, 0, 0, 1]


def check_decoder_layer(o):
    """One decoder layer against torch primitives: F.rms_norm, F.linear, causal SDPA with the
    key-value heads repeated per group, and the MoE written with torch.topk / softmax (ties
    have probability zero with these Gaussian inputs)."""
    rng = np.random.default_rng(95)
    T, hq, hkv, dh, n, k, f, seq = 21, 4, 2, 8, 4, 2, 12, 8
    d = hq * dh
    h = rng.standard_normal((T, d))
    wq, wo = rng.standard_normal((hq * dh, d)) / 4, rng.standard_normal((d, hq * dh)) / 4
    wk, wv = rng.standard_normal((hkv * dh, d)) / 4, rng.standard_normal((hkv * dh, d)) / 4
    wg = rng.standard_normal((d, n))
    w1, w3 = rng.standard_normal((n, f, d)) / 4, rng.standard_normal((n, f, d)) / 4
    w2 = rng.standard_normal((n, d, f)) / 4
    out = o.decoder_layer(h, wq, wk, wv, wo, wg, w1, w3, w2, k, hq, hkv, seq)
    t = torch.from_numpy
    ht = t(h)
    a = F.rms_norm(ht, (d,), eps=1e-5)
    q = F.linear(a, t(wq)).view(T, hq, dh)
    kk = F.linear(a, t(wk)).view(T, hkv, dh)
    v = F.linear(a, t(wv)).view(T, hkv, dh)
    att = torch.zeros(T, hq, dh, dtype=torch.float64)
    for s0 in range(0, T, seq):
        sl = slice(s0, min(T, s0 + seq))
        tq = q[sl].transpose(0, 1)
        tk = kk[sl].transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
        tv = v[sl].transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
        att[sl] = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True).transpose(0, 1)
    h1 = ht + F.linear(att.reshape(T, d), t(wo))
    x2 = F.rms_norm(h1, (d,), eps=1e-5)
    top, ti = torch.topk(x2 @ t(wg), k, dim=1)
    gw = torch.softmax(top, dim=1)
    moe = torch.zeros_like(h1)
    for s in range(k):
        for e in range(n):
            rows = ti[:, s] == e
            if rows.any():
                moe[rows] += gw[rows, s:s + 1] * F.linear(
                    F.silu(F.linear(x2[rows], t(w1[e]))) * F.linear(x2[rows], t(w3[e])), t(w2[e]))
    np.testing.assert_allclose(out, (h1 + moe).numpy(), rtol=1e-10, atol=1e-11)
    # the evaluation on a token sample gives the same rows
    sel = np.array([0, 7, 8, 15, 20])
    np.testing.assert_allclose(o.decoder_layer(h, wq, wk, wv, wo, wg, w1, w3, w2, k, hq, hkv, seq,
                                               tokens=sel), out[sel], rtol=1e-12, atol=1e-12)


CHECKS = [check_worked_example, check_gate_invariants, check_topk_bruteforce,
          check_softmax_order_equivalence, check_single_expert_is_plain_ffn,
          check_k_equals_n_is_dense_softmax_mixture, check_sparse_equals_dense, check_grouping,
          check_silu, check_bias_enters_before_topk, check_rmsnorm, check_param_counts,
          check_locality_metric, check_routing_statistics, check_backward_finite_differences,
          check_backward_autograd, check_backward_special_cases, check_attention,
          check_near_tie_tokens, check_attention_rows, check_ep_plan, check_decoder_layer]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__[6:])
def test_oracle_pin(check):
    check(moe_oracle)


# ------------------------------------------------------------------------------------------
# planted mistakes (CPU only): each must be caught by at least one pin
# ------------------------------------------------------------------------------------------
_ORIG_SWIGLU = moe_oracle.expert_swiglu
_ORIG_GROUP = moe_oracle.group_by_expert


def _mut_sigmoid_for_silu(z):
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def _mut_swap_w1_w3(xs, w1_e, w3_e, w2_e):
    return _ORIG_SWIGLU(xs, w3_e, w1_e, w2_e)


def _mut_drop_w3(xs, w1_e, w3_e, w2_e):
    xs = np.asarray(xs, dtype=np.float64)
    return moe_oracle.silu(xs @ np.asarray(w1_e).T) @ np.asarray(w2_e).T


def _mut_transpose_w2(xs, w1_e, w3_e, w2_e):
    xs = np.asarray(xs, dtype=np.float64)
    h = moe_oracle.silu(xs @ np.asarray(w1_e).T) * (xs @ np.asarray(w3_e).T)
    w2 = np.asarray(w2_e)
    return h @ w2.reshape(w2.shape[1], w2.shape[0])  # a plausible layout mix-up


def _mut_no_topk(logits, k):
    return np.asarray(logits, dtype=np.float64)


def _mut_ties_to_higher(logits, k):
    l = np.asarray(logits, dtype=np.float64)
    n = l.shape[1]
    order = np.argsort(-l[:, ::-1], axis=1, kind="stable")
    return (n - 1 - order)[:, :k].astype(np.int64)


def _mut_unstable_group(idx, n):
    off, perm, inv = _ORIG_GROUP(idx, n)
    for e in range(n):
        perm[off[e]:off[e + 1]] = perm[off[e]:off[e + 1]][::-1].copy()
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return off, perm, inv


def _mut_bias_after_topk(x, wg, bias=None):
    return np.asarray(x, dtype=np.float64) @ np.asarray(wg, dtype=np.float64)


def _mut_softmax_sign(z):
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(-(z - m))
    e[np.isinf(z)] = 0.0
    return e / np.sum(e, axis=-1, keepdims=True)


def _mut_rms_no_sqrt(h, eps=1e-5):
    h = np.asarray(h, dtype=np.float64)
    return h / (np.mean(h * h, axis=-1, keepdims=True) + eps)


_ORIG_STATS = moe_oracle.routing_statistics


def _mut_stats_cross_sequences(idx, n, seq_len=0):
    return _ORIG_STATS(idx, n, 0)


def _mut_stats_slotwise_any(idx, n, seq_len=0):
    c, p, f1, _ = _ORIG_STATS(idx, n, seq_len)
    e = np.asarray(idx)
    t = np.arange(1, e.shape[0])
    inside = np.ones(t.size, bool) if seq_len <= 0 else (t % seq_len) != 0
    return c, p, f1, int(np.count_nonzero((e[:-1] == e[1:]).any(axis=1)[inside]))


_ORIG_SWIGLU_BWD = moe_oracle.expert_swiglu_backward


def _mut_silu_grad_sigmoid_only(z):
    return moe_oracle.sigmoid(z)


def _mut_softmax_bwd_no_centering(p, dp):
    return np.asarray(p, dtype=np.float64) * np.asarray(dp, dtype=np.float64)


def _mut_swiglu_bwd_dw2_transposed(xs, do, w1_e, w3_e, w2_e):
    dxs, dw1, dw3, dw2 = _ORIG_SWIGLU_BWD(xs, do, w1_e, w3_e, w2_e)
    return dxs, dw1, dw3, dw2.reshape(dw2.shape[1], dw2.shape[0]).T.reshape(dw2.shape)


def _mut_swiglu_bwd_swapped_branches(xs, do, w1_e, w3_e, w2_e):
    dxs, dw1, dw3, dw2 = _ORIG_SWIGLU_BWD(xs, do, w1_e, w3_e, w2_e)
    return dxs, dw3, dw1, dw2


_ORIG_ATTN = moe_oracle.attention_gqa


def _mut_attn_heads_modulo(q, k, v, seq_len=0):
    hq, hkv = np.asarray(q).shape[1], np.asarray(k).shape[1]
    perm = [h % hkv * (hq // hkv) + h // hkv for h in range(hq)]   # query head h -> group h % hkv
    out = _ORIG_ATTN(np.asarray(q)[:, perm], k, v, seq_len)
    inv = np.argsort(perm)
    return out[:, inv]


def _mut_attn_no_scale(q, k, v, seq_len=0):
    dh = np.asarray(q).shape[2]
    return _ORIG_ATTN(np.asarray(q, dtype=np.float64) * np.sqrt(dh), k, v, seq_len)


def _mut_attn_one_sequence(q, k, v, seq_len=0):
    return _ORIG_ATTN(q, k, v, 0)


def _mut_attn_anticausal(q, k, v, seq_len=0):
    q, k, v = (np.asarray(a)[::-1] for a in (q, k, v))
    return _ORIG_ATTN(q, k, v, seq_len)[::-1]


_ORIG_NEAR_TIE = moe_oracle.near_tie_tokens


def _mut_near_tie_wrong_gap(logits, k, eps=1e-4):
    """the set gap taken between the (K+1)-th and (K+2)-th largest logits"""
    l = np.sort(np.asarray(logits, dtype=np.float64), axis=1)[:, ::-1]
    _, order_tie = _ORIG_NEAR_TIE(logits, k, eps)
    set_tie = np.zeros(l.shape[0], dtype=bool)
    if k + 1 < l.shape[1]:
        set_tie = (l[:, k] - l[:, k + 1]) < eps
    return set_tie, order_tie


def _mut_near_tie_order_off_by_one(logits, k, eps=1e-4):
    """the slot-order loop runs one gap too far (into the set gap)"""
    l = np.sort(np.asarray(logits, dtype=np.float64), axis=1)[:, ::-1]
    set_tie, _ = _ORIG_NEAR_TIE(logits, k, eps)
    order_tie = np.zeros(l.shape[0], dtype=bool)
    for j in range(min(k, l.shape[1] - 1)):
        order_tie |= (l[:, j] - l[:, j + 1]) < eps
    return set_tie, order_tie


_ORIG_ATTN_ROWS = moe_oracle.attention_gqa_rows


def _mut_attn_rows_excludes_self(q, k, v, rows, seq_len=0):
    """each row attends to the keys strictly before it (the diagonal dropped)"""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    T, hq, dh = q.shape
    group = hq // k.shape[1]
    S = T if seq_len <= 0 else seq_len
    out = np.zeros((len(rows), hq, dh))
    for r, i in enumerate(rows):
        s0 = (i // S) * S
        hi = max(i, s0 + 1)
        for h in range(hq):
            sc = k[s0:hi, h // group] @ q[i, h] / np.sqrt(dh)
            out[r, h] = moe_oracle.masked_softmax(sc) @ v[s0:hi, h // group]
    return out


_ORIG_EP_PLAN = ep_oracle.ep_exchange_plan
_ORIG_EP_OF = ep_oracle.ep_experts_of


def _mut_ep_strided_experts(rank, n, G):
    """rank r holds experts r, r+G, r+2G, ... instead of a contiguous block"""
    if G < 1 or n % G:
        raise ValueError("n must be a multiple of the number of ranks")
    return range(rank, n, G)


def _mut_ep_order_by_assignment(idx_per_rank, n, G):
    """a receiver orders an expert's rows by assignment index before source rank"""
    plans = _ORIG_EP_PLAN(idx_per_rank, n, G)
    for p in plans:
        lo = p["local_offsets"]
        for j in range(len(lo) - 1):
            seg = p["row_map"][lo[j]:lo[j + 1]]
            key = np.lexsort((p["recv_src"][seg], p["recv_assign"][seg]))
            p["row_map"][lo[j]:lo[j + 1]] = seg[key]
    return plans


def _mut_decoder_moe_on_h(h, wq, wk, wv, wo, wg, w1, w3, w2, k, hq, hkv, seq_len=0, eps=1e-5,
                          bias=None, **_):
    """the MoE sub-block normalises the layer input h instead of h1"""
    h = np.asarray(h, dtype=np.float64)
    T = h.shape[0]
    a = moe_oracle.rmsnorm(h, eps)
    q = (a @ np.asarray(wq).T).reshape(T, hq, -1)
    kk = (a @ np.asarray(wk).T).reshape(T, hkv, -1)
    v = (a @ np.asarray(wv).T).reshape(T, hkv, -1)
    h1 = h + moe_oracle.attention_gqa(q, kk, v, seq_len).reshape(T, -1) @ np.asarray(wo).T
    return h1 + moe_oracle.moe_layer(a, wg, w1, w3, w2, k, bias)

MUTATIONS = {
    "silu->sigmoid": ("silu", _mut_sigmoid_for_silu),
    "swap w1/w3": ("expert_swiglu", _mut_swap_w1_w3),
    "drop w3 branch": ("expert_swiglu", _mut_drop_w3),
    "w2 layout mix-up": ("expert_swiglu", _mut_transpose_w2),
    "no TopK mask": ("topk_mask", _mut_no_topk),
    "ties to higher index": ("topk_select", _mut_ties_to_higher),
    "unstable grouping": ("group_by_expert", _mut_unstable_group),
    "bias ignored": ("router_logits", _mut_bias_after_topk),
    "softmax sign flip": ("masked_softmax", _mut_softmax_sign),
    "rmsnorm without sqrt": ("rmsnorm", _mut_rms_no_sqrt),
    "pairs cross sequences": ("routing_statistics", _mut_stats_cross_sequences),
    "either-choice slot by slot": ("routing_statistics", _mut_stats_slotwise_any),
    "SiLU' = sigmoid": ("silu_grad", _mut_silu_grad_sigmoid_only),
    "softmax backward without centering": ("softmax_backward", _mut_softmax_bwd_no_centering),
    "dw2 layout mix-up": ("expert_swiglu_backward", _mut_swiglu_bwd_dw2_transposed),
    "dw1/dw3 swapped": ("expert_swiglu_backward", _mut_swiglu_bwd_swapped_branches),
    "attention heads grouped modulo": ("attention_gqa", _mut_attn_heads_modulo),
    "attention without 1/sqrt(dh)": ("attention_gqa", _mut_attn_no_scale),
    "attention across sequences": ("attention_gqa", _mut_attn_one_sequence),
    "attention anti-causal": ("attention_gqa", _mut_attn_anticausal),
    "near-tie set gap one too deep": ("near_tie_tokens", _mut_near_tie_wrong_gap),
    "near-tie order loop off by one": ("near_tie_tokens", _mut_near_tie_order_off_by_one),
    "attention rows without the diagonal": ("attention_gqa_rows", _mut_attn_rows_excludes_self),
    "EP experts strided over ranks": (ep_oracle, "ep_experts_of", _mut_ep_strided_experts),
    "decoder MoE normalises h, not h1": ("decoder_layer", _mut_decoder_moe_on_h),
    "EP rows ordered by assignment first": (ep_oracle, "ep_exchange_plan", _mut_ep_order_by_assignment),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutations(name, monkeypatch):
    spec = MUTATIONS[name]
    module, attr, fn = spec if len(spec) == 3 else (moe_oracle,) + spec
    monkeypatch.setattr(module, attr, fn)
    failed = []
    for check in CHECKS:
        try:
            check(moe_oracle)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"planted mistake '{name}' passed every pin"
