"""The multi-process path of bench.py on CPU: two gloo ranks (replicas, one per GPU in a real
run) go through the same plumbing -- process group, barriers, max of the per-rank times over
ranks, rank-0-only output -- without a GPU.  The layer itself needs no exchange between
ranks, so the only collectives are the timing ones tested here."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import bench
dist = bench.Dist()
dist.init("gloo")
rank = dist.rank
dist.barrier()
# each rank reports its own time; the job's time is the slowest rank's
t = dist.max(1.0 + 2.0 * rank)
dist.barrier()
print(json.dumps({"rank": rank, "world": dist.world, "max": t}), flush=True)
dist.close()
"""


@pytest.mark.parametrize("world", [2])
def test_bench_plumbing_two_gloo_ranks(world):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, ROOT=ROOT, RANK=str(r), WORLD_SIZE=str(world), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == list(range(world))
    assert all(o["world"] == world for o in outs)
    # max over ranks: every rank sees the slowest rank's time
    assert all(o["max"] == 1.0 + 2.0 * (world - 1) for o in outs)


def test_reference_arm_rank_nonzero_exits_without_work(tmp_path):
    """Under torchrun the oracle (reference) arm runs on rank 0 only; other ranks print
    nothing and exit 0."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "1", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_line_on_cpu():
    """The reference arm times the oracle on the host and prints one JSON line with the
    contract's keys."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "1", "--steps", "2", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
