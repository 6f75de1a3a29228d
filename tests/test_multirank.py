"""The multi-rank harness of bench.py on CPU: two gloo ranks, the barrier,
the max-over-ranks time and the whole-job throughput.  The data path itself
has no collective (each rank runs its own replica), so nothing else is
exchanged between ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist("gloo")
    assert d.world == world and d.rank == rank
    d.barrier()
    ms = 10.0 + 5.0 * rank          # pretend rank r took 10 + 5r ms
    mx = d.max(ms)
    out[rank] = (mx, bench.whole_job_rate(1000, 4, d.world, mx))
    d.barrier()
    d.close()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_time_and_throughput(world):
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()  # no fork after CUDA is initialised
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        mx, rate = out[r]
        assert mx == 15.0
        assert rate == pytest.approx(1000 * 4 * world / 0.015)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist("gloo")
    assert d.world == 1 and d.pg is None
    assert d.max(3.5) == 3.5
    assert bench.whole_job_rate(8192, 10, 1, 20.0) == pytest.approx(8192 * 10 / 0.020)
