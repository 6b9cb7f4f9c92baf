"""The multi-GPU path of bench.py on the CPU: two `gloo` ranks run the same barrier and
max-over-ranks reduction the timed region uses, and the weak-scaling value aggregates the
work of every replica over the slowest rank's time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    w, r, local, pg = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(pg)
    t_ms = 10.0 + 5.0 * rank  # this rank's timed region
    t_max = bench.max_over_ranks(pg, t_ms)
    bench.barrier(pg)
    out[rank] = t_max
    pg.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group():
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    w, r, local, pg = bench.dist_setup(1)
    assert (w, r, local, pg) == (1, 0, 0, None)
    assert bench.max_over_ranks(None, 3.5) == 3.5
