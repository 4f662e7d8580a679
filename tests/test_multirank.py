"""The N > 1 path of bench.py on CPU: two gloo ranks, each a replica with its
own time; the line reports the slowest rank and counts every rank's rows."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower replica
    slowest = bench.max_over_ranks(local_ms, world)
    value = bench.whole_job_us_per_row(slowest, steps=100, rows_per_rank=4, world=world)
    out[rank] = (slowest, value)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_replica():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]                    # every rank agrees
    slowest, value = res[0]
    assert slowest == pytest.approx(15.0)
    # 100 steps x 4 rows x 2 ranks in 15 ms
    assert value == pytest.approx(15.0 * 1000.0 / (100 * 4 * 2))
