"""The multi-process side of bench.py on the CPU: under torchrun every rank runs its own replica
(the decode step has no exchange step), the timed region is bracketed by a barrier, the reported
time is the maximum over ranks, and only rank 0 prints. Exercised here with two gloo ranks."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys
sys.path.insert(0, os.environ["ROOT"])
import torch
import bench
rank, local, world, dist = bench.dist_setup(2)
assert (rank, world) == (int(os.environ["RANK"]), 2)
bench.barrier(dist, torch)
# each rank times something different; every rank must see the slowest
m = bench.max_over_ranks(dist, torch, 10.0 * (rank + 1))
assert m == 20.0, m
print(f"rank{rank} max {m}", flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_max_over_ranks():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), BENCH_BACKEND="gloo", ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.STDOUT, text=True))
    outs = []
    for p in procs:
        out, _ = p.communicate(timeout=120)
        outs.append(out)
        assert p.returncode == 0, out
    assert "rank0 max 20.0" in outs[0] and "rank1 max 20.0" in outs[1]


def test_reference_arm_prints_on_rank_zero_only():
    # the reference arm of rank 1 does no work and prints nothing
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--config", "tiny"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    import json
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--config", "tiny"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["higher_is_better"] is True and line["warmup"] == 3
