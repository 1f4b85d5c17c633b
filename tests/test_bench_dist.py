"""bench.py's multi-rank host logic on CPU: two gloo ranks, no GPU.

Each rank is an independent replica (sequences shard across GPUs with no
data-path exchange); the only collectives are the barrier and the maximum of
the per-rank timings, and the whole-job rate is all ranks' units over the
slowest rank's time.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

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
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_env()
    t = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)])
    dist.barrier()
    out[rank] = (w, r, lr, t, bench.whole_job_rate(w, 100.0, t[0]))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        w, r, lr, t, rate = res[rank]
        assert (w, r, lr) == (world, rank, rank)
        assert t == [2.0, 10.0, 1.0]            # element-wise max over ranks
        assert rate == pytest.approx(2 * 100.0 / 2.0)


def test_single_process_needs_no_collective():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.whole_job_rate(1, 50.0, 2.0) == 25.0
