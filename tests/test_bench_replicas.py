"""The multi-GPU path of bench.py is N independent replicas (rows need no exchange): its host
logic, on CPU with gloo and two ranks -- the slowest rank's time is the one reported and the value
counts every rank's bytes; and the reference arm runs on rank 0 alone."""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slower replica
        slowest = bench.slowest_rank(ms, "cpu")
        value = bench.whole_job_gbs(1e9, world, 4, slowest * 1e-3)
        results[rank] = (slowest, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_report_the_slowest_rank_and_all_bytes():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    for r in range(world):
        slowest, value = res[r]
        assert slowest == 15.0                       # max over ranks, seen by every rank
        assert value == pytest.approx(1e9 * 2 * 4 / 15e-3 / 1e9)


def test_one_process_is_its_own_slowest_rank():
    import bench
    assert bench.slowest_rank(3.5, "cpu") == 3.5
    assert bench.whole_job_gbs(2e9, 1, 2, 1.0) == pytest.approx(4.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
