"""The multi-rank path of bench.py on CPU: two gloo ranks, each an independent
replica (weak scaling, no data-path collective).  The timing reduces to the slowest
rank, both ranks agree on it, and the whole-job rate counts every rank's steps;
the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 20.0][rank]  # the second replica is the slower one
    bench.sync_ranks(world)
    ms = bench.max_over_ranks(local_ms, world)
    q.put((rank, ms, bench.job_rate(100, world, ms)))
    bench.sync_ranks(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_replica():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for _, ms, rate in out:
        assert ms == 20.0                          # max over ranks, identical on both
        assert rate == pytest.approx(2 * 100 / 0.020)  # every rank's 100 steps in the slowest time


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.25, 1) == 7.25
    bench.sync_ranks(1)
    assert bench.job_rate(400, 1, 500.0) == pytest.approx(800.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.main_reference(args, 1, 2)  # rank 1 of 2: exits without work or output
    assert capsys.readouterr().out == ""
