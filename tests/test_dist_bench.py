"""The multi-process host logic of bench.py with two gloo ranks on the CPU:
rendezvous from the torchrun environment, the max-over-ranks timing reduction,
the barrier, and the reference arm's rank-0-only rule.  The path shards over
sequences with no collective, so timings are the only thing the ranks share."""
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


RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, os.environ["DFL2_ROOT"])
import bench
world, rank, local = bench.dist_init()
assert (world, rank, local) == (2, int(os.environ["RANK"]), int(os.environ["LOCAL_RANK"]))
mine = 1.5 if rank == 0 else 4.25          # a per-rank step time (ms)
worst = bench.max_over_ranks(mine, world)
bench.barrier(world)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps({"rank": rank, "max": worst}))
"""


def _launch(script, extra_env, port):
    procs = []
    for rank in range(2):
        env = dict(os.environ, DFL2_ROOT=ROOT, RANK=str(rank), LOCAL_RANK=str(rank),
                   WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   CUDA_VISIBLE_DEVICES="", **extra_env)
        procs.append(subprocess.Popen([sys.executable, "-c", script], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_max_over_ranks_and_barrier_with_two_gloo_ranks():
    outs = _launch(RANK_SCRIPT, {}, _free_port())
    got = sorted(json.loads(o.strip().splitlines()[-1])["rank"] for o in outs)
    assert got == [0, 1]
    for o in outs:
        assert json.loads(o.strip().splitlines()[-1])["max"] == 4.25


REF_SCRIPT = r"""
import os, sys
sys.path.insert(0, os.environ["DFL2_ROOT"])
import bench
sys.argv = ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
            "--workload", "tiny_l8_v32k"]
sys.exit(bench.main())
"""


def test_reference_arm_prints_on_rank_zero_only():
    pytest.importorskip("numpy")
    outs = _launch(REF_SCRIPT, {}, _free_port())
    lines = [[l for l in o.splitlines() if l.startswith("{")] for o in outs]
    # rank 1 exits 0 without work; rank 0 prints one JSON line
    assert sorted(len(x) for x in lines) == [0, 1]
    line = json.loads([x for x in lines if x][0][0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
