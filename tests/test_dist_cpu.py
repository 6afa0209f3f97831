"""The multi-rank plumbing of bench.py on CPU: two gloo ranks (spawned
processes, 127.0.0.1) run the barrier and the max-over-ranks reduction the
timed region uses, and the reference arm prints only on rank 0.  The layer
itself has no collective: ranks are independent replicas."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
class A: pass
world, rank, local = bench.dist_setup(A())
assert dist.get_world_size() == 2 and world == 2
bench.barrier(world)
v = bench.max_over_ranks(world, 10.0 + rank)
print(json.dumps({{"rank": rank, "max": v}}), flush=True)
dist.destroy_process_group()
"""


def test_two_gloo_ranks_barrier_and_max():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for pr in procs:
        out, err = pr.communicate(timeout=240)
        assert pr.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["max"] == 11.0 for o in outs)


@pytest.mark.timeout(600)
def test_reference_arm_prints_once_under_two_ranks():
    """--impl reference under two ranks: rank 0 prints one JSON line, the
    other rank exits 0 without output."""
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen(
            [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
             "--steps", "1", "--warmup", "3", "--workload", "tiny_fp32"],
            env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for pr in procs:
        out, err = pr.communicate(timeout=500)
        assert pr.returncode == 0, err[-2000:]
        outs.append(out)
    lines = [ln for o in outs for ln in o.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


CP_WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch, torch.distributed as dist
dist.init_process_group("gloo")
from mamba_selective_state_gb300.context_parallel import DistExchange
ex = DistExchange()
r = dist.get_rank()
assert ex.nshards == 2
g = ex.gather([torch.full((2, 3), float(r + 1))])
ids = ex.gather([torch.tensor([r, 10 + r], dtype=torch.int32)])
s = ex.sum(torch.tensor([1.0 + r, 2.0]))
print(json.dumps({{"rank": r, "g": g.tolist(), "ids": ids.tolist(), "s": s.tolist()}}), flush=True)
dist.destroy_process_group()
"""


def test_context_parallel_exchange_two_gloo_ranks():
    """The exchange of the context-parallel driver across two ranks: gathers
    stack the ranks' parts in rank (= shard) order, for float and int32
    parts, and the parameter-gradient sum adds the ranks' values."""
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", CP_WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for pr in procs:
        out, err = pr.communicate(timeout=240)
        assert pr.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["g"] == [[[1.0] * 3] * 2, [[2.0] * 3] * 2]
        assert o["ids"] == [[0, 10], [1, 11]]
        assert o["s"] == [3.0, 4.0]
