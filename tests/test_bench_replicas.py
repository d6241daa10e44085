"""bench.py with N > 1 (one process per GPU, independent replicas): the step
time is the slowest rank's, the value counts every rank's work, and only rank
0 of the reference arm works and prints.  The ranks here are gloo processes
on the CPU; the GPU run uses the same helpers over NCCL."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytest.importorskip("torch")

_WORKER = """
import json, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
r, w = dist.get_rank(), dist.get_world_size()
ms = bench.max_over_ranks(1.0 + 0.5 * r, dist, "cpu")
print(json.dumps({{"rank": r, "ms": ms, "tops": bench.whole_job_tops(2e12, w, ms)}}), flush=True)
dist.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, world: int, port: int) -> dict:
    env = dict(os.environ)
    env.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
               WORLD_SIZE=str(world))
    return env


def test_two_ranks_take_the_slowest_time_and_count_both_replicas():
    port = _free_port()
    code = _WORKER.format(root=ROOT)
    procs = [subprocess.Popen([sys.executable, "-c", code], env=_env(r, 2, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["ms"] == 1.5                              # rank 1's 1.5 ms, not rank 0's 1.0
        assert o["tops"] == pytest.approx(2 * 2e12 / 1.5e-3 / 1e12)


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_tops(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_nonzero_rank_exits_without_work():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "0"],
                         env=_env(1, 2, _free_port()), capture_output=True, text=True, timeout=180)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""
