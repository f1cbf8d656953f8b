"""Host logic of the multi-process benchmark path on CPU: two gloo ranks,
the job time is the slowest rank's (max over ranks), the job rate counts
every rank's work; the reference arm runs on rank 0 only."""
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


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        elapsed = 10.0 + 5.0 * rank  # rank 1 is the slower
        job = bench.max_over_ranks(elapsed, device="cpu")
        out[rank] = (job, bench.job_rate(1e12, 4, world, job))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_count_all_work():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        job, rate = res[rank]
        assert job == 15.0
        # 2 ranks x 4 steps x 1 TFLOP in 15 ms
        assert rate == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_process_is_its_own_max():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, device="cpu") == 3.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-1000:]
    assert r.stdout.strip() == ""
