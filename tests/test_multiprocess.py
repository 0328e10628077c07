"""The N > 1 path of bench.py on CPU, with two gloo ranks.

The TTT scan shards by (batch, head) with no exchange on the data path: each
rank runs its own copy of the workload (weak scaling), and the only
collectives are the barrier around the timed region and the max over ranks of
the measured time.  These tests run that host logic in two processes:

* the rendezvous of bench.dist_setup (gloo when no GPU is present);
* bench.max_over_ranks returns the slowest rank's time on every rank;
* bench.barrier lets both ranks through;
* under torchrun the reference arm runs on rank 0 only; other ranks return
  without work and without output.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    m = bench.max_over_ranks(times[rank], w)
    out[rank] = m
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    times = [1.25, 3.5]
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.0, 1) == 2.0
    bench.barrier(1)  # no-op


@pytest.mark.parametrize("rank", [1])
def test_reference_arm_is_silent_on_other_ranks(rank):
    # under torchrun only rank 0 runs and prints the reference arm
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
