"""The multi-rank path of bench.py on CPU (gloo, world size 2): each rank scores its own seeded
workload, the slowest rank's time is taken, and the whole-job value counts every rank's work."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(10.0 + rank * 5.0, dist, "cpu")
    case = bench.make_workload("long_decode", 4, rank)
    q.put((rank, t, case.seq_lens_k.tolist()))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_own_workloads():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]           # max over ranks on every rank
    assert res[0][2] != res[1][2]                         # independent per-rank workloads


def test_whole_job_value_counts_every_rank():
    one = bench.whole_job_gops(1000, 10, 1, 2.0)
    two = bench.whole_job_gops(1000, 10, 2, 2.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(1000 * 16384 * 10 / 2e-3 / 1e9)


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
