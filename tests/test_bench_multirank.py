"""The multi-rank path of bench.py on CPU: world size 2 over gloo.

The path shards by (batch, head): each rank runs its own replica and the only
cross-rank operation is the max of the step times, so that is what is tested
here, together with the whole-job rate and the reference arm's rank handling.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = bench.reduce_max(dist, 1.5 * (rank + 1), torch.device("cpu"))
    q.put((rank, ms, bench.whole_job_rate(world, 1000, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_step_time_is_the_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in got] == [0, 1]
    for _, ms, rate in got:
        assert ms == 3.0
        assert rate == pytest.approx(2 * 1000 / 3e-3)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_whole_job_rate_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.whole_job_rate(1, 196704, 0.2) == pytest.approx(196704 / 2e-4)
