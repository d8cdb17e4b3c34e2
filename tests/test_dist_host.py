"""Host logic of the multi-GPU bench path with two gloo ranks on CPU: each
rank runs an independent replica; the whole-job value uses the slowest
rank's time (max over ranks) and every rank's units."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.init_dist(w, "gloo")
    bench.barrier()
    ms = 1.0 + rank                     # rank 1 is the slow one
    m = bench.reduce_max(ms, "cpu")
    out[rank] = (m, bench.whole_job(256, m / 1e3, w))
    bench.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_whole_job():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        m, value = res[r]
        assert m == pytest.approx(2.0)
        assert value == pytest.approx(2 * 256 / 2e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.whole_job(256, 0.5, 1) == 512
