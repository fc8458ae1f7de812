"""bench.py's multi-rank path on CPU: two gloo ranks agree on the slowest rank's time and
the whole-job throughput counts every replica (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup("gloo")
    assert (w, r, local) == (world, rank, rank)
    my_ms = 10.0 + 5.0 * rank                 # rank 1 is the slow one
    total = bench.max_over_ranks(my_ms)
    out[rank] = (total, bench.job_tflops(w, 4, 1e12, total))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    total, tf = res[0]
    assert total == 15.0
    assert tf == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1, 10, 2e12, 20.0) == pytest.approx(1000.0)
