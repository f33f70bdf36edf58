"""Host-side logic of bench.py under several ranks, on CPU with gloo
(world size 2): the job's time is the maximum over ranks, and the reference
arm does its work and prints on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, os.environ["ROOT"])
import torch, torch.distributed as tdist
import bench
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
tdist.init_process_group("gloo", rank=rank, world_size=world)
m = bench.max_over_ranks(1.5 + 2.0 * rank, torch.device("cpu"))
class A: pass
a = A(); a.ref_seconds = 0.0; a.steps = 1; a.warmup = 3
ref = bench.run_reference(a, rank, world) if rank != 0 else "skipped"
print(json.dumps({"rank": rank, "max": m, "ref": ref}), flush=True)
tdist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_max_and_reference_rank0_only():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, ROOT=ROOT, RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            pytest.fail("rank did not finish")
        assert p.returncode == 0, e
        outs.append(o)
    import json
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o in outs), key=lambda r: r["rank"])
    assert [r["max"] for r in res] == [3.5, 3.5]
    assert res[1]["ref"] is None  # the reference arm does no work on rank 1
