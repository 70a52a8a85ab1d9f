"""Expert parallelism without a GPU: the exchange logic of sparse_mixture_experts_56_b300.ep
(split sizes, the count and row all-to-alls, the return to token order) on gloo ranks and on
ranks emulated in one process, with every per-rank step done by the fp64 oracle
(tests/ep_ops.py).  Each rank's output must equal the single-GPU layer on its tokens, and
the rows exchanged must be the oracle's exchange plan."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_56_b300 import ep
from tests.ep_ops import OracleOps

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(G, T, d, f, n, k, seed=7, skew=False):
    rng = np.random.default_rng(seed)
    xs = [rng.standard_normal((T, d)) for _ in range(G)]
    wg = rng.standard_normal((d, n)) * 0.5
    w1 = rng.standard_normal((n, f, d)) / np.sqrt(d)
    w3 = rng.standard_normal((n, f, d)) / np.sqrt(d)
    w2 = rng.standard_normal((n, d, f)) / np.sqrt(f)
    bias = np.where(np.arange(n) == 0, 2.0, 0.0) if skew else None
    return xs, wg, w1, w3, w2, bias


def _check_rank(y, xs_r, wg, w1, w3, w2, k, bias):
    ref = oracle.moe_layer(xs_r, wg, w1, w3, w2, k, bias)
    np.testing.assert_allclose(np.asarray(y), ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("G,T,n,k,skew", [(1, 20, 8, 2, False), (2, 24, 8, 2, False),
                                          (4, 16, 8, 2, True), (8, 9, 8, 2, False),
                                          (2, 30, 4, 3, True)])
def test_ep_emulated_ranks_match_single_rank(G, T, n, k, skew):
    d, f = 16, 24
    xs, wg, w1, w3, w2, bias = _inputs(G, T, d, f, n, k, seed=G * 10 + T, skew=skew)
    t = torch.from_numpy
    ys, stats = ep.ep_layer_forward_emulated(OracleOps(), [t(x) for x in xs], t(wg), t(w1), t(w3),
                                             t(w2), k, n, G, None if bias is None else t(bias))
    for r in range(G):
        _check_rank(ys[r], xs[r], wg, w1, w3, w2, k, bias)
    idx = [oracle.gate(x, wg, k, bias)[0] for x in xs]
    plans = oracle.ep_exchange_plan(idx, n, G)
    assert stats["expert_rows"] == oracle.ep_load(plans).tolist()
    assert stats["send_rows"] == [p["send_counts"].tolist() for p in plans]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import numpy as np, torch, torch.distributed as dist
from sparse_mixture_experts_56_b300 import ep
from tests.ep_ops import OracleOps
from tests.test_ep_cpu import _inputs
dist.init_process_group("gloo")
r, G = dist.get_rank(), dist.get_world_size()
T, d, f, n, k = 24, 16, 24, 8, 2
xs, wg, w1, w3, w2, bias = _inputs(G, T, d, f, n, k, seed=123, skew=True)
blk = ep.expert_block(r, n, G)
sl = slice(blk.start, blk.stop)
t = torch.from_numpy
y, stats = ep.ep_layer_forward(ep.TorchComm(), OracleOps(), t(xs[r]), t(wg), t(w1[sl]), t(w3[sl]),
                               t(w2[sl]), k, n, t(bias))
np.save(os.environ["OUT"] + f"/y{r}.npy", y.numpy())
stats.pop("topk_idx")
print(json.dumps({"rank": r, "stats": stats}), flush=True)
dist.destroy_process_group()
"""


@pytest.mark.parametrize("world", [2, 4])
def test_ep_gloo_ranks_match_single_rank(world, tmp_path):
    """world gloo ranks, each holding 8/world experts and 24 tokens of its own (skewed routing,
    so the ranks receive unequal loads): every rank's y equals the single-GPU layer on its
    tokens, and the rows each rank sent and received are the oracle plan's."""
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, ROOT=ROOT, RANK=str(r), WORLD_SIZE=str(world), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), OUT=str(tmp_path))
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = {}
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err
        o = json.loads(out.strip().splitlines()[-1])
        outs[o["rank"]] = o["stats"]
    T, d, f, n, k = 24, 16, 24, 8, 2
    xs, wg, w1, w3, w2, bias = _inputs(world, T, d, f, n, k, seed=123, skew=True)
    idx = [oracle.gate(x, wg, k, bias)[0] for x in xs]
    plans = oracle.ep_exchange_plan(idx, n, world)
    for r in range(world):
        _check_rank(np.load(tmp_path / f"y{r}.npy"), xs[r], wg, w1, w3, w2, k, bias)
        assert outs[r]["send_rows"] == plans[r]["send_counts"].tolist()
        assert outs[r]["recv_rows"] == plans[r]["recv_counts"].sum(axis=1).tolist()
        assert outs[r]["expert_rows"] == int(oracle.ep_load(plans)[r])
    # skewed routing loads rank 0 (which holds expert 0) the most
    assert int(oracle.ep_load(plans)[0]) == max(outs[r]["expert_rows"] for r in range(world))
