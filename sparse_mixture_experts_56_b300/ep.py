"""Expert parallelism (EP) of the MoE layer: the experts spread over G GPUs.

Tokens an expert must process go to the GPU that holds it and the expert outputs return to
the original token positions (newsflash.city digest, section "专家层的混合"; "Mixtral 8x7B:
疎な専門家混合言語モデル" (ja.news.hada.io), section "実装と推論効率", which adds that the work
has to be balanced between the GPUs; "Mixtral of Experts" (xyznot.com summary), "Términos
clave" and "Limitaciones y preguntas abiertas", on the load imbalance consecutive-token
expert repetition causes).

Rank g of G holds the experts [g*E, (g+1)*E), E = n/G, and routes its own tokens (the
router weight is replicated).  One layer pass on rank g:

  1. route, group and gather its tokens (moe_router_topk, moe_permute, moe_gather_rows):
     rows in grouping order, so the rows for each destination are one contiguous block;
  2. exchange the per-expert counts (all-to-all, E counts per destination), then the rows
     (all-to-all-v, split sizes from the counts);
  3. order the received rows by local expert (moe_ep_regroup; the up-projection reads them
     through its row map), run the local experts (moe_expert_up / moe_expert_down with
     k = 1 and n = E), and put the outputs back in receive order (moe_gather_rows);
  4. send the outputs back (the reverse all-to-all-v) and combine them with the gate
     weights in token order (moe_combine).

Every step of the layer runs in libmoe.so's kernels; the exchanges are the collective
library's (NCCL through torch.distributed on GPUs).  The split sizes of the row exchange
come to the host once per pass (one small device-to-host copy of the counts).

The same phases also run with G ranks emulated in one process (`ep_layer_forward_emulated`):
each phase runs for every rank in turn and the exchanges become device-to-device copies
between the ranks' buffers, so that the whole EP sequence can be checked on one GPU without
any kernel waiting for another rank's.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence

import torch

__all__ = ["expert_block", "TorchComm", "NativeOps", "Dispatch", "dispatch", "expert_phase",
           "ep_layer_forward", "ep_layer_forward_emulated", "send_splits"]


def expert_block(rank: int, n: int, G: int) -> range:
    """Experts held by `rank` of `G`: the contiguous block [rank*n/G, (rank+1)*n/G)."""
    if G < 1 or n % G:
        raise ValueError(f"{n} experts cannot be split evenly over {G} ranks")
    E = n // G
    return range(rank * E, (rank + 1) * E)


def send_splits(offsets_host: Sequence[int], n: int, G: int) -> List[int]:
    """Rows a rank sends to each destination: its grouped rows of that destination's experts."""
    return [int(offsets_host[expert_block(g, n, G).stop]) - int(offsets_host[expert_block(g, n, G).start])
            for g in range(G)]


class TorchComm:
    """The two exchanges over torch.distributed (NCCL for CUDA tensors, gloo for CPU ones)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_to_all_counts(self, send: torch.Tensor) -> torch.Tensor:
        """`send` [G * E]: E counts for each destination; returns the E counts of every source."""
        out = torch.empty_like(send)
        self.dist.all_to_all_single(out, send, group=self.group)
        return out

    def all_to_all_rows(self, out: torch.Tensor, inp: torch.Tensor, out_splits: List[int],
                        in_splits: List[int]) -> None:
        self.dist.all_to_all_single(out, inp, out_splits, in_splits, group=self.group)


class NativeOps:
    """The per-rank steps on libmoe.so (CUDA tensors; bf16 or fp32 activations)."""

    def __init__(self, device):
        from . import _native
        _native.lib()
        self.device = torch.device(device)
        self._ws = {}

    def _workspace(self, key, T, d, f, n, k, dtype):
        from . import moe_workspace_size, workspace
        need = moe_workspace_size(T, d, f, n, k, dtype)
        ws = self._ws.get(key)
        if ws is None or ws.numel() < need:
            ws = workspace(max(T, 1), d, f, n, k, dtype, self.device)
            self._ws[key] = ws
        return ws

    def route(self, x, w_gate, k, bias):
        from . import moe_router_topk
        idx, w, _ = moe_router_topk(x, w_gate, k, bias)
        return idx, w

    def permute(self, idx, n):
        from . import moe_permute
        T, k = idx.shape
        ws = self._workspace("permute", T, 64, 64, n, k, torch.bfloat16)
        return moe_permute(idx, n, ws)

    def gather(self, src, index, k):
        from . import moe_gather_rows
        return moe_gather_rows(src, index, k)

    def regroup(self, recv_counts, R):
        from . import moe_ep_regroup
        return moe_ep_regroup(recv_counts, R)

    def experts(self, rows, row_map, local_offsets, w1, w3, w2):
        """Local experts on the received rows: row_map gives the experts' row order and
        local_offsets their ranges; returns the outputs in that (grouped) order."""
        from . import moe_expert_down, moe_expert_up
        R, d = rows.shape
        E, f, _ = w1.shape
        if R == 0:
            return rows.new_empty((0, d))
        ws = self._workspace("experts", R, d, f, E, 1, rows.dtype)
        h = moe_expert_up(rows, row_map, local_offsets, w1, w3, 1, ws)
        return moe_expert_down(h, local_offsets, w2, 1, ws)

    def combine(self, y_perm, inv_perm, w):
        from . import moe_combine
        return moe_combine(y_perm, inv_perm, w)

    def host_ints(self, t) -> List[int]:
        return [int(v) for v in t.cpu().reshape(-1).tolist()]

    def counts_tensor(self, values: Sequence[int]):
        return torch.tensor(list(values), dtype=torch.int32, device=self.device)


@dataclasses.dataclass
class Dispatch:
    """One rank's state after step 1."""
    idx: torch.Tensor
    gate_w: torch.Tensor
    inv_perm: torch.Tensor
    x_perm: torch.Tensor          # [T*k, d] rows in grouping order
    counts: List[int]             # rows per expert (all n)
    send: List[int]               # rows per destination rank
    valid: int                    # rows with a valid expert (= sum of counts)


def dispatch(ops, x, w_gate, k: int, n: int, G: int, bias=None) -> Dispatch:
    idx, w = ops.route(x, w_gate, k, bias)
    off, perm, inv = ops.permute(idx, n)
    x_perm = ops.gather(x, perm, k)
    off_h = ops.host_ints(off)
    counts = [off_h[e + 1] - off_h[e] for e in range(n)]
    return Dispatch(idx, w, inv, x_perm, counts, send_splits(off_h, n, G), off_h[n])


def expert_phase(ops, x_recv, recv_counts, R: int, w1, w3, w2):
    """Step 3 on one rank: received rows (receive order) -> expert outputs (receive order)."""
    local_offsets, row_map, inv_row_map = ops.regroup(recv_counts, R)
    # the experts take their rows through row_map (the up-projection gathers them), so their
    # outputs come out in grouped order; inv_row_map puts them back in receive order
    y_local = ops.experts(x_recv, row_map, local_offsets, w1, w3, w2)
    return ops.gather(y_local, inv_row_map, 1)


def ep_layer_forward(comm, ops, x, w_gate, w1_local, w3_local, w2_local, k: int, n: int,
                     logit_bias=None):
    """One layer pass of rank `comm.rank`: its tokens x [T, d] in, y [T, d] out.  w*_local are
    this rank's experts (expert_block(rank, n, G)).  Returns (y, stats)."""
    G = comm.world
    E = n // G
    expert_block(comm.rank, n, G)
    disp = dispatch(ops, x, w_gate, k, n, G, logit_bias)
    recv = comm.all_to_all_counts(ops.counts_tensor(disp.counts))
    recv_h = ops.host_ints(recv)
    recv_split = [sum(recv_h[s * E:(s + 1) * E]) for s in range(G)]
    R = sum(recv_split)
    d = x.shape[1]
    x_recv = x.new_empty((R, d))
    comm.all_to_all_rows(x_recv, disp.x_perm[:disp.valid], recv_split, disp.send)
    y_ret = expert_phase(ops, x_recv, recv.view(G, E), R, w1_local, w3_local, w2_local)
    y_perm = x.new_zeros((disp.x_perm.shape[0], d)) if disp.valid < disp.x_perm.shape[0] \
        else x.new_empty((disp.x_perm.shape[0], d))
    comm.all_to_all_rows(y_perm[:disp.valid], y_ret, disp.send, recv_split)
    y = ops.combine(y_perm, disp.inv_perm, disp.gate_w)
    return y, {"send_rows": disp.send, "recv_rows": recv_split, "expert_rows": R,
               "expert_counts": disp.counts, "topk_idx": disp.idx}


def ep_layer_forward_emulated(ops, xs: Sequence, w_gate, w1, w3, w2, k: int, n: int, G: int,
                              logit_bias=None):
    """The same pass for G ranks emulated in one process: xs[r] are rank r's tokens; w1, w3,
    w2 hold all n experts (rank r uses its block).  Returns ([y_r], stats)."""
    E = n // G
    blocks = [expert_block(r, n, G) for r in range(G)]
    disps = [dispatch(ops, xs[r], w_gate, k, n, G, logit_bias) for r in range(G)]
    outs = []
    y_rets = []
    starts = [[sum(ds.send[:g]) for g in range(G)] for ds in disps]
    for g in range(G):
        counts = [disps[s].counts[e] for s in range(G) for e in blocks[g]]
        R = sum(counts)
        parts = [disps[s].x_perm[starts[s][g]:starts[s][g] + disps[s].send[g]] for s in range(G)]
        x_recv = torch.cat(parts) if R else xs[g].new_empty((0, xs[g].shape[1]))
        recv_counts = ops.counts_tensor(counts).view(G, E)
        sl = slice(blocks[g].start, blocks[g].stop)
        y_rets.append(expert_phase(ops, x_recv, recv_counts, R, w1[sl], w3[sl], w2[sl]))
    for s in range(G):
        ds = disps[s]
        d = xs[s].shape[1]
        y_perm = xs[s].new_zeros((ds.x_perm.shape[0], d))
        for g in range(G):
            # source s's rows sit in y_rets[g] after the rows of sources < s
            before = sum(disps[q].send[g] for q in range(s))
            y_perm[starts[s][g]:starts[s][g] + ds.send[g]] = y_rets[g][before:before + ds.send[g]]
        outs.append(ops.combine(y_perm, ds.inv_perm, ds.gate_w))
    load = [sum(disps[s].send[g] for s in range(G)) for g in range(G)]
    return outs, {"expert_rows": load, "send_rows": [ds.send for ds in disps],
                  "topk_idx": [ds.idx for ds in disps]}
