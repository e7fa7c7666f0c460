"""Host logic of bench.py's multi-replica path, run as two gloo ranks on CPU:
each rank draws its own inputs, the job time is the slowest rank's, and the
job throughput counts every rank's bytes."""
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 20.0 - rank, 5.0 * (rank + 1)]
        got = bench.max_over_ranks(mine, world, "cpu")
        q.put((rank, got, bench.layer_seed(rank, 0), bench.layer_seed(rank, 7)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_combine_timings():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, g0, s00, s07), (_, g1, s10, s17) = res
    assert g0 == g1 == [11.0, 20.0, 10.0]          # element-wise max over ranks
    assert len({s00, s07, s10, s17}) == 4            # every rank and layer has its own inputs


def test_job_throughput_counts_all_ranks():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    one = bench.job_gbs(bench.step_bytes(131072), 1, 0.05)
    assert bench.job_gbs(bench.step_bytes(131072), 4, 0.05) == pytest.approx(4 * one)
    assert bench.step_bytes(131072) == 151_032_960
    assert bench.max_over_ranks([1.0, 2.0], 1) == [1.0, 2.0]
