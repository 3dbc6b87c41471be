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


def test_metric_counts_exactly_the_oracles_visible_pairs():
    """The benchmark's algorithmic work (16384 ops per visible query-key pair) counts the pairs the
    oracle's mask makes visible, over the benchmarked workloads and shapes that exercise the mask
    (BSND with short rows, TND with an empty sequence, compression, both sparse modes)."""
    import oracle
    import workloads as W
    from checker import visible_counts
    cases = [W.long_decode(batch=4), W.fp8_compressed_decode(batch=3),
             W.make_case("m0", batch=3, s1=4, q_lens=[4, 2, 0], seq_lens_k=[300, 3, 64], block_size=16,
                         sparse_count=8, sparse_mode=3, cmp_ratio=4, seed=1),
             W.make_case("m1", layout_q="TND", q_lens=[5, 0, 9], seq_lens_k=[40, 7, 9], block_size=16,
                         sparse_count=8, sparse_mode=3, cmp_ratio=2, seed=2),
             W.make_case("m2", batch=2, s1=3, seq_lens_k=[50, 2], block_size=16, sparse_count=8,
                         sparse_mode=0, cmp_ratio=8, seed=3)]
    for case in cases:
        assert bench.visible_pairs(case) == int(visible_counts(case, oracle).sum()), case.name
