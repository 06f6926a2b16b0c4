"""Multi-rank host logic of bench.py on CPU: two gloo ranks (127.0.0.1).

Each rank runs the same work on its own GPU in the real benchmark (weak
scaling, no collective on the data path); the only cross-rank steps are the
barrier and the max over ranks of the timed duration, tested here."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist = bench.dist_init(w, use_cuda=False)
    dist.barrier()
    m = bench.reduce_max(dist, 1.5 + rank, use_cuda=False)
    out.put((rank, m))
    dist.destroy_process_group()


def test_two_ranks_agree_on_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 2.5), (1, 2.5)]


def test_single_rank_needs_no_process_group():
    assert bench.dist_init(1, use_cuda=False) is None
    assert bench.reduce_max(None, 3.0, use_cuda=False) == 3.0
