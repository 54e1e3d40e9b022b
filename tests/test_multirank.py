"""The multi-replica path of bench.py on CPU: two gloo ranks, each with its
own batch; the job's time is the slowest rank's, its throughput the tokens
of all ranks over that time; the reference arm runs on rank 0 only."""
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


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]
    got = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    seeds = bench.rank_seed(7, rank)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, seeds, bench.job_tokens_per_s(128, world, got)))


def test_two_gloo_ranks_take_the_slowest_rank():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [5.0, 5.0]          # max over ranks on every rank
    assert res[0][2] != res[1][2]                      # each rank has its own batches
    assert res[0][3] == pytest.approx(2 * 128 / 5e-3)  # whole-job tokens/s


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    assert bench.job_tokens_per_s(128, 1, 1.0) == pytest.approx(128000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
