"""Replica bookkeeping of bench.py with N > 1, run as two gloo ranks on the CPU.

The decode step does not shard, so N GPUs run N independent replicas: the job
time is the slowest rank's, and the job throughput counts every rank's tokens.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

WORKER = r"""
import json, os, sys, time
sys.path.insert(0, sys.argv[1])
import bench
rank, world, local, dist = bench.dist_setup()
assert dist is not None and dist.get_backend() == "gloo"
bench.barrier(dist)
seconds = [1.5, 4.0][rank]
m = bench.reduce_max(dist, seconds)
value = bench.job_throughput(64, world, m)
bench.barrier(dist)
# the reference arm prints from rank 0 only; other ranks return without work
args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "tiny"])
if rank != 0:
    t0 = time.perf_counter()
    bench.run_reference(args, bench.workload("tiny"), rank, world, dist)
    assert time.perf_counter() - t0 < 0.5
print(json.dumps({"rank": rank, "world": world, "max": m, "value": value}), flush=True)
dist.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.dist_setup() == (0, 1, 0, None)
    assert bench.reduce_max(None, 2.5) == 2.5
    bench.barrier(None)


def test_job_throughput_counts_all_ranks():
    assert bench.job_throughput(100, 1, 2.0) == 50.0
    assert bench.job_throughput(100, 4, 2.0) == 200.0


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER)
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, str(script), ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            pytest.fail("gloo ranks did not finish")
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2
        assert o["max"] == 4.0
        assert o["value"] == pytest.approx(64 * 2 / 4.0)


def test_reference_arm_line_is_a_measured_single_core_sample(capsys):
    """The reference arm times the oracle on one host thread: ms_per_step is the
    measured time of one sample step (so ms_per_step x steps fits the run) and
    value is that time projected to the whole model by weight+KV bytes."""
    import time
    args = bench.parse_args(["--impl", "reference", "--steps", "2", "--warmup", "1", "--workload", "tiny"])
    t0 = time.perf_counter()
    bench.run_reference(args, bench.workload("tiny"), 0, 1, None)
    wall = time.perf_counter() - t0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["cores"] == 1
    assert line["ms_per_step"] * line["steps"] / 1e3 <= wall
    proj = line["projection"]
    assert abs(proj["measured_s_per_sample_step"] * 1e3 - line["ms_per_step"]) < 1e-6
    assert abs(line["value"] * proj["measured_s_per_sample_step"] * proj["factor"] - 1.0) < 1e-9
    assert proj["factor"] > 1.0     # the tiny model's two layers, sampled with one
    assert line["e2e"]["value"] == line["value"]
