"""The multi-process replica path of the benchmark on CPU (gloo, two ranks).

Every rank runs the whole step on its own data; the ranks meet only at the barrier around the
timed region and in the reduction of its result: the slowest rank's time, and the units all
ranks processed.  These tests launch real ranks with torch.distributed.run on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(nproc, *argv, timeout=300):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={nproc}", "--master-addr=127.0.0.1",
           f"--master-port={free_port()}", *argv]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


def json_lines(text):
    return [json.loads(l) for l in text.splitlines() if l.startswith("{")]


def test_single_rank_aggregate_is_local():
    ms, units, value = bench.aggregate_replicas(torch, None, 4.0, 3)
    assert (ms, units) == (4.0, 3)
    assert value == pytest.approx(750.0)


def test_two_ranks_take_slowest_time_and_all_units():
    r = torchrun(2, os.path.join("tests", "replica_worker.py"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    line = lines[0]
    assert line["world"] == 2
    assert line["ms"] == pytest.approx(3.0)       # max over ranks (2 ms and 3 ms)
    assert line["units"] == 2                     # one unit per rank
    assert line["value"] == pytest.approx(2 * 1000.0 / 3.0)


def test_reference_arm_runs_on_rank_zero_only():
    r = torchrun(2, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                 "--warmup", "3", "--cpu-seconds", "0.1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["value"] == line["value"]
