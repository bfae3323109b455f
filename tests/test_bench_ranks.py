"""The benchmark's multi-process logic on CPU (gloo, two ranks): the job's
time is the slowest rank's, the whole-job figure counts every replica's
layer-tokens, and the reference arm does its work on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.job_max(1.5 + rank, dist)           # rank 1 is the slow one
        out.put((rank, ms, bench.job_us_per_layer_token(ms, world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_figure():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = 2.5 * 1e3 / (bench.N_LAYERS * bench.N_TOKENS) / 2
    assert [g[1] for g in got] == [2.5, 2.5]
    assert all(g[2] == pytest.approx(expect) for g in got)


def test_single_process_job_figure():
    assert bench.job_max(3.0, None) == 3.0
    assert bench.job_us_per_layer_token(5.12, 1) == pytest.approx(1.0)


def test_reference_arm_does_nothing_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
