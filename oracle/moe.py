"""fp64 oracle of the sparse MoE feed-forward layer (test infrastructure only).

Sources, by page title and section:
  [G]   "Mixtral of Experts" (xyznot.com summary), section "Método (con las
        ecuaciones clave)": G(x) := Softmax(TopK(x·W_g)); TopK keeps the K largest
        logits of l = x·W_g in R^n and sets the others to -inf; y = sum_i G(x)_i ·
        SwiGLU_i(x); n = 8 experts, K = 2, hidden 4096, intermediate 14336.
  [CS]  "《Mixtral of Experts》Mixtral 8x7B：稀疏专家混合模型的突破性进展"
        (blog.csdn.net), section "MOE数学公式": §1 W_g in R^{d x n} and
        y = sum_{i=0}^{n-1} G(x)_i E_i(x); §2.1 logits; §2.2 the TopK definition;
        §2.3 the softmax over the TopK output and the worked example with experts
        3 and 5; §3.2 softmax-then-TopK-then-renormalise.
  [JA]  "Mixtral 8x7B: 疎な専門家混合言語モデル" (ja.news.hada.io), sections
        "MoEレイヤーの計算方式" (experts whose gate is 0 need not be computed)
        and "実装と推論効率" (variable token counts per expert; outputs return to
        the original token positions).
  [NF]  newsflash.city digest, section "专家层的混合" (same two facts).

What the pages leave open, and the reading taken here:
  * TopK ties: the lower expert index wins; output slots are in descending
    logit order (stable sort by the key (-l_i, i)).
  * SwiGLU is only named on the pages; it is read as
    E_i(x) = w2_i · (SiLU(w1_i · x) ⊙ (w3_i · x)), SiLU(z) = z·sigmoid(z), no biases,
    with w1_i, w3_i stored [f, d] and w2_i stored [d, f] (out x in).
  * The optional per-expert logit bias is added to x·W_g before TopK and softmax.
  * RMSNorm (h / sqrt(mean(h^2) + eps), unit weight) and the residual of the
    stacked workload are not on the pages; they come from the workload definition.

All arithmetic is float64 on the exact stored input values (bf16 or fp32 values
expanded to float64).  Nothing is blocked, fused or reordered beyond the
definitions; NumPy matmul and argsort serve as library steps.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


# ------------------------------------------------------------------------------------------
# Router: logits, TopK, softmax over the kept logits     [G], [CS] §2.1-§2.3
# ------------------------------------------------------------------------------------------
def router_logits(x, wg, bias=None) -> np.ndarray:
    """l = x · W_g (+ b), W_g in R^{d x n}   ([G] eq. G; [CS] §2.1)."""
    l = _f64(x) @ _f64(wg)
    if bias is not None:
        l = l + _f64(bias)[None, :]
    return l


def topk_select(logits, k: int) -> np.ndarray:
    """Indices of the K largest logits per row, in descending logit order ([CS] §2.2).

    Ties are broken toward the lower expert index (reading: stable order on the
    key (-l_i, i)).  Returns int64 [T, k].
    """
    l = _f64(logits)
    T, n = l.shape
    if not 1 <= k <= n:
        raise ValueError("need 1 <= k <= n")
    # argsort of -l with a stable sort orders by (-l_i, i)
    order = np.argsort(-l, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def topk_mask(logits, k: int) -> np.ndarray:
    """(TopK(l))_i = l_i if i is among the K largest, else -inf   ([G]; [CS] §2.2)."""
    l = _f64(logits)
    idx = topk_select(l, k)
    out = np.full_like(l, -np.inf)
    rows = np.arange(l.shape[0])[:, None]
    out[rows, idx] = l[rows, idx]
    return out


def masked_softmax(z) -> np.ndarray:
    """Softmax over the last axis where -inf entries get exactly 0   ([CS] §2.3)."""
    z = _f64(z)
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)  # exp(-inf) = 0
    return e / np.sum(e, axis=-1, keepdims=True)


def gate(x, wg, k: int, bias=None) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """G(x) = Softmax(TopK(x·W_g)).

    Returns (idx [T,k] int64 in descending logit order, w [T,k] the gate values of
    those experts, G [T,n] the full sparse gate vector, logits [T,n]).
    """
    l = router_logits(x, wg, bias)
    G = masked_softmax(topk_mask(l, k))
    idx = topk_select(l, k)
    w = np.take_along_axis(G, idx, axis=1)
    return idx, w, G, l


def gate_softmax_then_topk(logits, k: int) -> np.ndarray:
    """The alternative order of [CS] §3.2: softmax over all n, keep the K largest
    probabilities, renormalise them to sum 1.  Returns the full [T,n] gate vector.
    The page states both orders give zero weight outside the K kept experts; after
    renormalisation the kept weights equal those of G(x)."""
    l = _f64(logits)
    p = masked_softmax(l)
    idx = topk_select(p, k)  # same ranking as the logits (softmax is monotone)
    rows = np.arange(l.shape[0])[:, None]
    kept = np.zeros_like(p)
    kept[rows, idx] = p[rows, idx]
    return kept / np.sum(kept, axis=1, keepdims=True)


# ------------------------------------------------------------------------------------------
# Experts: SwiGLU FFN                                   [G] (SwiGLU experts, 4096 -> 14336)
# ------------------------------------------------------------------------------------------
def silu(z) -> np.ndarray:
    """SiLU(z) = z · sigmoid(z) = z / (1 + exp(-z)), written to avoid overflow."""
    z = _f64(z)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


def expert_swiglu(xs, w1_e, w3_e, w2_e) -> np.ndarray:
    """E(x) = w2 · (SiLU(w1 · x) ⊙ (w3 · x)) for the rows of ``xs`` [m, d].

    w1_e, w3_e: [f, d]; w2_e: [d, f].  Returns [m, d] float64.
    """
    xs = _f64(xs)
    a = xs @ _f64(w1_e).T
    b = xs @ _f64(w3_e).T
    h = silu(a) * b
    return h @ _f64(w2_e).T


# ------------------------------------------------------------------------------------------
# Grouping by expert                                     [JA] 実装と推論効率; [NF] 专家层的混合
# ------------------------------------------------------------------------------------------
def group_by_expert(idx, n: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Group the T·K assignments a = t·K + k by expert.

    Returns (offsets [n+1], perm [A], inv_perm [A]), all int64:
      offsets[e] = number of assignments to experts < e (exclusive prefix sum of the
                   per-expert counts; offsets[n] = A);
      perm[p]    = the assignment at position p, positions ordered by (expert, a);
      inv_perm[a] = the position of assignment a.
    """
    e = np.asarray(idx, dtype=np.int64).reshape(-1)
    if e.size and (e.min() < 0 or e.max() >= n):
        raise ValueError("expert index out of range")
    counts = np.bincount(e, minlength=n)[:n]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    perm = np.argsort(e, kind="stable").astype(np.int64)
    inv_perm = np.empty_like(perm)
    inv_perm[perm] = np.arange(perm.size, dtype=np.int64)
    return offsets, perm, inv_perm


# ------------------------------------------------------------------------------------------
# The layer                                               [G] eq. y; [CS] §1; [JA] MoEレイヤー
# ------------------------------------------------------------------------------------------
def moe_layer(x, wg, w1, w3, w2, k: int, bias=None, *, idx=None, w=None,
              tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """y = sum_i G(x)_i · E_i(x), evaluated sparsely: only experts with a non-zero
    gate are computed ([JA] MoEレイヤーの計算方式), each on the group of tokens
    routed to it, and each result is added back at its token's position.

    ``idx``/``w`` override the router (shape [T,k], one row per token of ``x``);
    ``tokens`` restricts the evaluation to those token rows (the result then has
    len(tokens) rows).
    """
    x = _f64(x)
    if tokens is not None:
        tokens = np.asarray(tokens, dtype=np.int64)
        xs = x[tokens]
    else:
        xs = x
    if idx is None:
        gi, gw, _, _ = gate(xs, wg, k, bias)
    else:
        # the override always covers every token row of x; it is sliced like x
        gi = np.asarray(idx, dtype=np.int64)
        gw = _f64(w)
        if gi.shape[0] != x.shape[0] or gw.shape != gi.shape:
            raise ValueError("idx/w must have one row per token of x")
        if tokens is not None:
            gi, gw = gi[tokens], gw[tokens]
    n = np.asarray(w1).shape[0]
    y = np.zeros_like(xs)
    offsets, perm, _ = group_by_expert(gi, n)
    kk = gi.shape[1]
    for e in range(n):
        sel = perm[offsets[e]:offsets[e + 1]]
        if sel.size == 0:
            continue  # a zero gate: the expert is not evaluated
        t = sel // kk
        out = expert_swiglu(xs[t], w1[e], w3[e], w2[e])
        np.add.at(y, t, gw.reshape(-1)[sel][:, None] * out)
    return y


def moe_layer_dense(x, wg, w1, w3, w2, k: int, bias=None) -> np.ndarray:
    """The literal dense sum y = sum_{i=0}^{n-1} G(x)_i · E_i(x) over every expert
    ([CS] §1), including those whose gate is exactly zero.  Used to check the
    sparse evaluation on small inputs."""
    x = _f64(x)
    _, _, G, _ = gate(x, wg, k, bias)
    n = np.asarray(w1).shape[0]
    y = np.zeros_like(x)
    for i in range(n):
        y += G[:, i:i + 1] * expert_swiglu(x, w1[i], w3[i], w2[i])
    return y


# ------------------------------------------------------------------------------------------
# Stacked workload (not on the pages): RMSNorm and residual
# ------------------------------------------------------------------------------------------
def rmsnorm(h, eps: float = 1e-5) -> np.ndarray:
    """h / sqrt(mean(h^2) + eps) with unit weight (row-wise)."""
    h = _f64(h)
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)


def stacked_layer(h, wg, w1, w3, w2, k: int, eps: float = 1e-5, *, x_norm=None,
                  tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """h + MoE(RMSNorm(h)).  ``x_norm`` may pass the normalised rows in the
    precision the layer consumes them (the bf16-stored activations)."""
    h = _f64(h)
    xn = rmsnorm(h, eps) if x_norm is None else _f64(x_norm)
    if tokens is not None:
        tokens = np.asarray(tokens, dtype=np.int64)
        return h[tokens] + moe_layer(xn, wg, w1, w3, w2, k, tokens=tokens)
    return h + moe_layer(xn, wg, w1, w3, w2, k)


# ------------------------------------------------------------------------------------------
# Helpers for comparisons
# ------------------------------------------------------------------------------------------
def near_tie_tokens(logits, k: int, eps: float = 1e-4) -> Tuple[np.ndarray, np.ndarray]:
    """Tokens whose K-th and (K+1)-th largest logits differ by less than ``eps``
    (the selected set is then not decided by fp32 vs fp64 rounding), and tokens
    whose kept logits are within ``eps`` of each other (slot order not decided).
    Returns two boolean masks [T]."""
    l = np.sort(_f64(logits), axis=1)[:, ::-1]
    n = l.shape[1]
    set_tie = np.zeros(l.shape[0], dtype=bool)
    if k < n:
        set_tie = (l[:, k - 1] - l[:, k]) < eps
    order_tie = np.zeros(l.shape[0], dtype=bool)
    for j in range(k - 1):
        order_tie |= (l[:, j] - l[:, j + 1]) < eps
    return set_tie, order_tie


def consecutive_same_expert_rate(idx) -> float:
    """Share of consecutive token pairs (t, t+1) whose first-choice expert is the
    same — the routing-locality measure of the routing analysis (newsflash.city
    digest, "路径分析", Table 5; xyznot.com, "Limitaciones": 28.4% at layer 15 vs
    12.5% = 1/8 for random assignment)."""
    first = np.asarray(idx)[:, 0]
    if first.size < 2:
        return float("nan")
    return float(np.mean(first[1:] == first[:-1]))


def param_counts(d: int, f: int, n: int, k: int, layers: int, heads: int, kv_heads: int):
    """Expert and attention parameter counts of the layer stack (per [G]: 32 layers,
    hidden 4096, 32 heads, 8 KV heads, 8 SwiGLU experts of 14336).  Embeddings are
    not counted (the pages give no vocabulary size)."""
    expert = layers * n * 3 * d * f
    active_expert = layers * k * 3 * d * f
    head_dim = d // heads
    attn = layers * (2 * d * d + 2 * d * kv_heads * head_dim)
    return {"expert": expert, "active_expert": active_expert, "attention": attn}


def routing_statistics(idx, n: int, seq_len: int = 0):
    """Routing statistics of one layer from its TopK selections ``idx`` [T, K]:

      counts[e]  number of assignments (token, slot) routed to expert e — the per-layer
                 expert load (newsflash.city digest, "路径分析": how tokens spread over
                 the experts of each layer);
      pairs      consecutive token pairs (t, t+1) inside one sequence;
      same_first pairs whose first-choice experts are equal (the repetition measure of
                 Table 5 in the routing analysis; xyznot.com, "Limitaciones": 28.4% at
                 layer 15 against 12.5% = 1/8 for random assignment);
      same_any   pairs whose K chosen experts have at least one expert in common (the
                 pages define only the first-choice measure; this extension to all K
                 choices takes the plainest reading of "the same expert chosen again").

    ``seq_len`` > 0 splits the T tokens into sequences of that length (the last one may
    be shorter) and no pair crosses a sequence boundary; 0 means one sequence.
    Returns (counts int64 [n], pairs, same_first, same_any)."""
    e = np.asarray(idx, dtype=np.int64)
    if e.ndim != 2:
        raise ValueError("idx must be [T, K]")
    T = e.shape[0]
    if e.size and (e.min() < 0 or e.max() >= n):
        raise ValueError("expert index out of range")
    counts = np.bincount(e.reshape(-1), minlength=n)[:n].astype(np.int64)
    if T < 2:
        return counts, 0, 0, 0
    t_next = np.arange(1, T)
    inside = np.ones(T - 1, dtype=bool) if seq_len <= 0 else (t_next % seq_len) != 0
    a, b = e[:-1][inside], e[1:][inside]
    same_first = int(np.count_nonzero(a[:, 0] == b[:, 0]))
    # any expert of token t among the experts of token t+1
    share = (a[:, :, None] == b[:, None, :]).any(axis=(1, 2))
    return counts, int(inside.sum()), same_first, int(np.count_nonzero(share))


# ------------------------------------------------------------------------------------------
# Backward of the layer (the chain rule applied to the forward definitions above)
# ------------------------------------------------------------------------------------------
def sigmoid(z) -> np.ndarray:
    z = _f64(z)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def silu_grad(z) -> np.ndarray:
    """d/dz SiLU(z) = sigma(z) + z sigma(z) (1 - sigma(z))."""
    z = _f64(z)
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def softmax_backward(p, dp) -> np.ndarray:
    """Vector-Jacobian product of the softmax over the last axis: for p = softmax(z) and
    dL/dp = dp, dL/dz = p (dp - sum_j p_j dp_j)."""
    p, dp = _f64(p), _f64(dp)
    return p * (dp - np.sum(p * dp, axis=-1, keepdims=True))


def expert_swiglu_backward(xs, do, w1_e, w3_e, w2_e):
    """Backward of E(x) = w2 (SiLU(w1 x) ⊙ (w3 x)) for the rows of ``xs`` [m, d] given
    dL/dE = ``do`` [m, d].  Returns (dxs [m,d], dw1 [f,d], dw3 [f,d], dw2 [d,f])."""
    xs, do = _f64(xs), _f64(do)
    w1_e, w3_e, w2_e = _f64(w1_e), _f64(w3_e), _f64(w2_e)
    a, b = xs @ w1_e.T, xs @ w3_e.T
    s = silu(a)
    h = s * b
    dh = do @ w2_e
    da = dh * b * silu_grad(a)
    db = dh * s
    return da @ w1_e + db @ w3_e, da.T @ xs, db.T @ xs, do.T @ h


def moe_layer_backward(x, wg, w1, w3, w2, k: int, dy, bias=None, *, idx=None):
    """Gradients of the scalar L = <dy, y> for y = moe_layer(x, ...), by the chain rule through
    the definitions of [G] / [CS] (the pages train the model but print no backward; the
    derivative of the forward they define is the only reading).  TopK is piecewise constant,
    so logits outside the kept set get no gradient; inside it the softmax Jacobian gives
    dl_i = G_i (dG_i - sum_j G_j dG_j) with dG_i = <dy, E_i(x)>.

    ``idx`` overrides the selection (one row per token).  Returns a dict of float64 arrays:
    dx [T,d], dwg [d,n], dw1 [n,f,d], dw3 [n,f,d], dw2 [n,d,f], dbias [n], dlogits [T,n],
    dgate [T,k] (dG of the kept experts, slot order of idx)."""
    x, dy = _f64(x), _f64(dy)
    wg, w1, w3, w2 = _f64(wg), _f64(w1), _f64(w3), _f64(w2)
    T, d = x.shape
    n, f, _ = w1.shape
    l = router_logits(x, wg, bias)
    gi = topk_select(l, k) if idx is None else np.asarray(idx, dtype=np.int64)
    gw = masked_softmax(np.take_along_axis(l, gi, axis=1))        # G at the kept experts
    dx = np.zeros_like(x)
    dw1, dw3, dw2 = np.zeros_like(w1), np.zeros_like(w3), np.zeros_like(w2)
    dgate = np.zeros((T, gi.shape[1]))
    offsets, perm, _ = group_by_expert(gi, n)
    kk = gi.shape[1]
    for e in range(n):
        sel = perm[offsets[e]:offsets[e + 1]]
        if sel.size == 0:
            continue                                              # no rows, zero gradient
        t, slot = sel // kk, sel % kk
        xs, g = x[t], dy[t]
        dgate[t, slot] = np.sum(g * expert_swiglu(xs, w1[e], w3[e], w2[e]), axis=1)
        dxs, dw1[e], dw3[e], dw2[e] = expert_swiglu_backward(
            xs, gw[t, slot][:, None] * g, w1[e], w3[e], w2[e])    # dL/dE_i(x) = G_i dy
        np.add.at(dx, t, dxs)
    dl = np.zeros((T, n))
    np.put_along_axis(dl, gi, softmax_backward(gw, dgate), axis=1)
    dx += dl @ wg.T
    return {"dx": dx, "dwg": x.T @ dl, "dw1": dw1, "dw3": dw3, "dw2": dw2,
            "dbias": dl.sum(axis=0), "dlogits": dl, "dgate": dgate}


# ------------------------------------------------------------------------------------------
# Attention sub-block of the decoder layer (the other half of each layer)
# ------------------------------------------------------------------------------------------
def attention_gqa(q, k, v, seq_len: int = 0) -> np.ndarray:
    """Causal softmax attention with grouped key/value heads: for query head h, key/value head
    g = h // (Hq / Hkv), token i of a sequence,

        o_i = sum_{j <= i} softmax_j(q_i · k_j / sqrt(dh)) v_j

    over the tokens j of the same sequence ("Mixtral of Experts" (xyznot.com summary), Método:
    32 attention heads, 8 key-value heads, hidden 4096 — so dh = 128; newsflash.city digest:
    the full dense 32k context, i.e. no sliding window).  The pages give no positional
    encoding; positions enter through the causal mask only.
    q [T, Hq, dh], k and v [T, Hkv, dh]; ``seq_len`` > 0 splits the T tokens into sequences of
    that length (the last may be shorter), 0 means one sequence.  Returns [T, Hq, dh]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, hq, dh = q.shape
    hkv = k.shape[1]
    if hq % hkv:
        raise ValueError("query heads must be a multiple of key-value heads")
    group = hq // hkv
    S = T if seq_len <= 0 else seq_len
    out = np.zeros_like(q)
    for s0 in range(0, T, S):
        s1 = min(T, s0 + S)
        n = s1 - s0
        causal = np.tril(np.ones((n, n), dtype=bool))
        for h in range(hq):
            g = h // group
            scores = q[s0:s1, h] @ k[s0:s1, g].T / np.sqrt(dh)
            scores = np.where(causal, scores, -np.inf)
            out[s0:s1, h] = masked_softmax(scores) @ v[s0:s1, g]
    return out


def attention_gqa_rows(q, k, v, rows, seq_len: int = 0) -> np.ndarray:
    """The same definition as ``attention_gqa``, evaluated only at the query positions
    ``rows`` (so that single rows deep inside a long sequence cost O(prefix) each):

        o_i = sum_{j <= i, j in the sequence of i} softmax_j(q_i · k_j / sqrt(dh)) v_j

    for every query head.  q [T, Hq, dh], k and v [T, Hkv, dh]; returns [len(rows), Hq, dh]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, hq, dh = q.shape
    hkv = k.shape[1]
    if hq % hkv:
        raise ValueError("query heads must be a multiple of key-value heads")
    group = hq // hkv
    S = T if seq_len <= 0 else seq_len
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    out = np.zeros((rows.size, hq, dh))
    for r, i in enumerate(rows):
        s0 = (i // S) * S                       # first token of the sequence holding i
        for h in range(hq):
            g = h // group
            scores = k[s0:i + 1, g] @ q[i, h] / np.sqrt(dh)
            out[r, h] = masked_softmax(scores) @ v[s0:i + 1, g]
    return out


# ------------------------------------------------------------------------------------------
# One decoder layer: the attention sub-block and the MoE sub-block, each with a residual
# ------------------------------------------------------------------------------------------
def decoder_layer(h, wq, wk, wv, wo, wg, w1, w3, w2, k: int, hq: int, hkv: int,
                  seq_len: int = 0, eps: float = 1e-5, bias=None, *, with_logits: bool = False,
                  tokens: Optional[Sequence[int]] = None):
    """One decoder layer of the Mixtral stack ("Mixtral of Experts" (xyznot.com summary),
    Método: Mistral 7B's layers of attention (32 query heads, 8 key-value heads, hidden
    4096) with every feed-forward sub-block replaced by the MoE layer):

        a  = RMSNorm(h)
        h1 = h + (attention_gqa(a wqᵀ, a wkᵀ, a wvᵀ) flattened) woᵀ
        h2 = h1 + MoE(RMSNorm(h1))

    The pages give neither the normalisation nor a positional encoding: RMSNorm with unit
    weight before each sub-block (as in the stacked workload) and no positional encoding
    (positions enter through the causal mask).  wq [hq*dh, d], wk / wv [hkv*dh, d],
    wo [d, hq*dh] (out x in), dh = 128 in the pages' shapes.  ``with_logits`` also returns
    the MoE sub-block's router logits; ``tokens`` evaluates only those rows (keys and values
    still come from every token, queries and everything after them only from those rows)."""
    h = _f64(h)
    T = h.shape[0]
    a = rmsnorm(h, eps)
    kk = (a @ _f64(wk).T).reshape(T, hkv, -1)
    v = (a @ _f64(wv).T).reshape(T, hkv, -1)
    if tokens is None:
        q = (a @ _f64(wq).T).reshape(T, hq, -1)
        o = attention_gqa(q, kk, v, seq_len).reshape(T, -1)
        hs = h
    else:
        tokens = np.asarray(tokens, dtype=np.int64)
        q = np.zeros((T, hq, kk.shape[2]))
        q[tokens] = (a[tokens] @ _f64(wq).T).reshape(tokens.size, hq, -1)
        o = attention_gqa_rows(q, kk, v, tokens, seq_len).reshape(tokens.size, -1)
        hs = h[tokens]
    h1 = hs + o @ _f64(wo).T
    x2 = rmsnorm(h1, eps)
    h2 = h1 + moe_layer(x2, wg, w1, w3, w2, k, bias)
    return (h2, router_logits(x2, wg, bias)) if with_logits else h2
