"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks agree on
the slowest rank's time and on the whole-job throughput (no GPU needed)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 100.0 + 50.0 * rank               # rank 1 is the slowest
    ms_max = bench.max_over_ranks(ms)
    out.put((rank, ms_max, bench.job_throughput(65536, 10, world, ms_max)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [150.0, 150.0]
    assert res[0][2] == res[1][2] == pytest.approx(65536 * 10 * 2 / 0.150)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_throughput(1000, 2, 1, 1000.0) == 2000.0
