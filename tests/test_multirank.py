"""The multi-process path of bench.py on CPU: two gloo ranks set up the
process group the way the bench does under torchrun, pass its barriers and
agree on the slowest rank's time; the job throughput counts every rank's
tokens over that time (weak scaling, replicas with no data-path exchange)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(backend="gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    t = 0.5 + rank  # the second rank is the slow one
    out[rank] = (bench.max_over_ranks(t, w), bench.job_throughput(1000, w, bench.max_over_ranks(t, w)))
    bench.barrier(w)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_max_time():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        ctx = mp.get_context("spawn")
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(100)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    slowest, thr = res[0]
    assert slowest == 1.5
    assert thr == pytest.approx(2 * 1000 / 1.5)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(8192, 1, 0.5) == 16384
