"""fp64 oracle of Expert Parallelism (EP) for the MoE layer (test infrastructure only).

Sources, by page title and section:
  [NF]  newsflash.city digest, section "专家层的混合": besides standard model parallelism the
        layer can be spread over several GPUs by expert parallelism; tokens that a given
        expert must process are routed to the GPU holding it, and the expert outputs return
        to the original token positions.
  [JA]  "Mixtral 8x7B: 疎な専門家混合言語モデル" (ja.news.hada.io), section "実装と推論効率":
        the same two steps, plus: EP has to split the work evenly between the GPUs, so load
        balancing is needed.
  [XY]  "Mixtral of Experts" (xyznot.com summary), "Términos clave" (EP maps different
        experts to different GPUs and sends token activations across devices to their
        expert) and "Limitaciones y preguntas abiertas" (consecutive tokens repeat experts,
        which can overload particular GPUs under EP).

What the pages leave open, and the reading taken here:
  * Which GPU holds which expert: G ranks, n divisible by G, rank r holds the contiguous
    block of experts [r*n/G, (r+1)*n/G).
  * Every rank routes its own tokens (the router weight is replicated); a rank sends each
    destination the rows of its assignments to that destination's experts, in its own
    grouping order (expert, then assignment a = t*K + slot).
  * A receiving rank evaluates its experts on the rows it received, expert by expert, the
    rows of one expert ordered by source rank and then by the source's order.
  * "Load" of a rank = the rows it receives (the work its experts do in one layer pass).

All of this is integer bookkeeping; the arithmetic of the layer is moe.py's.
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np

from .moe import group_by_expert


def ep_experts_of(rank: int, n: int, G: int) -> range:
    """Experts held by ``rank`` of ``G``: the contiguous block [rank*n/G, (rank+1)*n/G)."""
    if G < 1 or n % G:
        raise ValueError("n must be a multiple of the number of ranks")
    E = n // G
    return range(rank * E, (rank + 1) * E)


def ep_send_counts(offsets, n: int, G: int) -> np.ndarray:
    """Rows one rank sends to each destination: the assignments of its grouping (``offsets``
    [n+1] from group_by_expert) to the destination's experts.  Returns int64 [G]."""
    off = np.asarray(offsets, dtype=np.int64)
    return np.array([off[ep_experts_of(g, n, G).stop] - off[ep_experts_of(g, n, G).start]
                     for g in range(G)], dtype=np.int64)


def ep_exchange_plan(idx_per_rank: Sequence, n: int, G: int) -> List[dict]:
    """The exchange of one EP layer pass, for ranks whose TopK selections are
    ``idx_per_rank[s]`` [T_s, K].  For each rank g returns a dict of int64 arrays:

      send_counts [G]      rows g sends to each destination (its grouping order)
      recv_counts [G, E]   rows g receives from each source for each of its E local experts
      local_offsets [E+1]  exclusive prefix sum of the rows of g's local experts
      row_map [R]          row_map[p] = index, in g's receive buffer (the sources' blocks
                           concatenated in source order), of the row at grouped position p
      recv_src [R], recv_assign [R]
                           source rank and source assignment a = t*K + slot of every row of
                           the receive buffer
    Rows of one local expert are ordered by source rank, then by the source's grouping order
    (assignment index), which is the order the experts evaluate them in."""
    groupings = [group_by_expert(np.asarray(i, dtype=np.int64), n) for i in idx_per_rank]
    E = n // G
    plans = []
    for g in range(G):
        mine = ep_experts_of(g, n, G)
        recv_counts = np.zeros((G, E), dtype=np.int64)
        recv_src, recv_assign, recv_expert = [], [], []
        for s, (off, perm, _) in enumerate(groupings):
            # source s's rows for g, in s's grouping order: experts of g in ascending order
            for j, e in enumerate(mine):
                rows = perm[off[e]:off[e + 1]]
                recv_counts[s, j] = rows.size
                recv_src.extend([s] * rows.size)
                recv_assign.extend(rows.tolist())
                recv_expert.extend([j] * rows.size)
        recv_expert = np.asarray(recv_expert, dtype=np.int64)
        # grouped order: by local expert, then by position in the receive buffer (which is
        # already ordered by source, then by the source's order)
        row_map = np.array([q for j in range(E) for q in np.flatnonzero(recv_expert == j)],
                           dtype=np.int64)
        counts = recv_counts.sum(axis=0)
        plans.append({
            "send_counts": ep_send_counts(groupings[g][0], n, G),
            "recv_counts": recv_counts,
            "local_offsets": np.concatenate([[0], np.cumsum(counts)]).astype(np.int64),
            "row_map": row_map,
            "recv_src": np.asarray(recv_src, dtype=np.int64),
            "recv_assign": np.asarray(recv_assign, dtype=np.int64),
        })
    return plans


def ep_load(plans: Sequence[dict]) -> np.ndarray:
    """Rows each rank's experts process in the pass (the load [JA] asks to balance)."""
    return np.array([int(p["recv_counts"].sum()) for p in plans], dtype=np.int64)


def ep_regroup(recv_counts) -> tuple:
    """The receiving side from its counts alone: ``recv_counts`` [G, E] rows from source s
    for local expert j.  The receive buffer lists the sources' blocks in source order, each
    block its experts' rows in expert order; the experts evaluate the rows of local expert j
    source by source.  Returns (local_offsets [E+1], row_map [R], inv_row_map [R]) with
    row_map[p] = receive-buffer row at grouped position p."""
    c = np.maximum(np.asarray(recv_counts, dtype=np.int64), 0)
    G, E = c.shape
    recv_pos = {}
    q = 0
    for s in range(G):
        for j in range(E):
            for i in range(int(c[s, j])):
                recv_pos[(s, j, i)] = q
                q += 1
    row_map = [recv_pos[(s, j, i)] for j in range(E) for s in range(G) for i in range(int(c[s, j]))]
    row_map = np.asarray(row_map, dtype=np.int64)
    inv = np.empty_like(row_map)
    inv[row_map] = np.arange(row_map.size, dtype=np.int64)
    local_offsets = np.concatenate([[0], np.cumsum(c.sum(axis=0))]).astype(np.int64)
    return local_offsets, row_map, inv

