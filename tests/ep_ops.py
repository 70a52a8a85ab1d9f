"""The per-rank steps of the expert-parallel layer done by the fp64 oracle on CPU tensors
(test infrastructure): lets the exchange logic of sparse_mixture_experts_56_b300.ep run on
gloo ranks without a GPU, and gives the emulated multi-rank pass a CPU reference."""
from __future__ import annotations

import numpy as np
import torch

import oracle


class OracleOps:
    def route(self, x, w_gate, k, bias):
        idx, w, _, _ = oracle.gate(x.numpy(), w_gate.numpy(), k,
                                   None if bias is None else bias.numpy())
        return torch.from_numpy(idx.astype(np.int32)), torch.from_numpy(w)

    def permute(self, idx, n):
        off, perm, inv = oracle.group_by_expert(idx.numpy(), n)
        return tuple(torch.from_numpy(a.astype(np.int32)) for a in (off, perm, inv))

    def gather(self, src, index, k):
        return src[index.long() // k]

    def regroup(self, recv_counts, R):
        lo, rm, inv = oracle.ep_regroup(recv_counts.numpy())
        assert rm.size == R
        return tuple(torch.from_numpy(a.astype(np.int32)) for a in (lo, rm, inv))

    def experts(self, rows, row_map, local_offsets, w1, w3, w2):
        out = torch.zeros((row_map.numel(), rows.shape[1]), dtype=torch.float64)
        lo = local_offsets.tolist()
        for j in range(len(lo) - 1):
            sel = row_map[lo[j]:lo[j + 1]].long()
            if sel.numel():
                out[lo[j]:lo[j + 1]] = torch.from_numpy(oracle.expert_swiglu(
                    rows[sel].numpy(), w1[j].numpy(), w3[j].numpy(), w2[j].numpy()))
        return out

    def combine(self, y_perm, inv_perm, w):
        T, k = w.shape
        rows = inv_perm.long().view(T, k)
        y = torch.zeros((T, y_perm.shape[1]), dtype=torch.float64)
        for s in range(k):
            y += w[:, s:s + 1] * y_perm[rows[:, s]]
        return y

    def host_ints(self, t):
        return [int(v) for v in t.reshape(-1).tolist()]

    def counts_tensor(self, values):
        return torch.tensor(list(values), dtype=torch.int64)
