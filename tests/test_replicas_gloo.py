"""The N > 1 path of bench.py on CPU: two replica processes over gloo.

The hot path does not shard across GPUs; with N GPUs the benchmark runs N
independent replicas, synchronises them with a barrier and reports the slowest
replica's time. These tests run that host logic as two processes with the gloo
backend (no GPU), plus the rule that only rank 0 runs the reference arm.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import bench
rank, world = bench.dist_init()
bench.barrier(world)
slowest = bench.max_over_ranks(10.0 + rank, world)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps({"rank": rank, "world": world, "slowest": slowest}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    env = dict(os.environ)
    env.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "CUDA_VISIBLE_DEVICES": ""})
    return env


def test_two_replicas_agree_on_the_slowest_time():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", _CHILD, ROOT], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["world"] == 2 for o in outs)
    assert all(o["slowest"] == 11.0 for o in outs)


def test_reference_arm_runs_on_rank_zero_only():
    code = ("import sys; sys.path.insert(0, sys.argv[1]); import bench; "
            "args = bench.argparse.Namespace(workload='fc400k', steps=1, warmup=0, bin_len=500, learners=16, "
            "cpu_seconds=1.0); "
            "print(bench.run_reference(args))")
    env = _env(1, 2, _free_port())
    out = subprocess.run([sys.executable, "-c", code, ROOT], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip().splitlines()[-1] == "None"
