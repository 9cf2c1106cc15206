"""bench.py's multi-process logic on CPU: two gloo ranks.

The step shards by prompt, so the only cross-rank traffic in bench.py is the
timing: a barrier around the timed region and the max of the ranks' elapsed
times.  These tests run that logic as two processes with the gloo backend
(no GPU), and check that the reference arm runs on rank 0 only.
"""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_RANK_SCRIPT = r'''
import os, sys, json
sys.path.insert(0, os.environ["BENCH_ROOT"])
import bench
world, rank, local = bench.dist_setup(int(os.environ["WORLD_SIZE"]))
bench.barrier(world)
m = bench.max_over_ranks(1.5 + rank, world)
print(json.dumps({"rank": rank, "world": world, "max": m, "seed": bench.input_seed(rank)}))
import torch.distributed as dist
dist.destroy_process_group()
'''


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(script, world, extra_env=None, args=()):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), BENCH_ROOT=ROOT,
                   CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, *script, *args], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=240)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_two_gloo_ranks_barrier_and_max():
    import json
    outs = _run_ranks(["-c", _RANK_SCRIPT], 2)
    got = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert {g["rank"] for g in got} == {0, 1}
    assert all(g["world"] == 2 and g["max"] == 2.5 for g in got)
    assert got[0]["seed"] != got[1]["seed"]  # each rank its own prompts


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    """--impl reference under two ranks: rank 0 times the oracle and prints
    one JSON line; rank 1 exits 0 without work."""
    import json
    outs = _run_ranks(["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1",
                       "--workload", "tiny_v64"], 2)
    lines = [o.strip().splitlines() for o in outs]
    assert len(lines[0]) == 1 and lines[1] == []
    rec = json.loads(lines[0][0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["value"] > 0
