"""The benchmark's multi-rank logic on CPU (gloo, world size 2): each rank
serves its own batch of the same recipe (weak scaling, no data-path
collective), and the timed value is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workload as wl

        seed = bench.shard_seed(wl.DEFAULT_SEED["0"], rank)
        w = wl.make("0", seed=seed)
        t = bench.max_over_ranks(1.5 + rank, dist, world, torch.device("cpu"))
        dist.barrier()
        out[rank] = (seed, int(w.prompts[0][:64].sum()), t)
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_and_take_the_max():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (s0, h0, t0), (s1, h1, t1) = out[0], out[1]
    assert s0 != s1 and h0 != h1          # different batches per rank
    assert t0 == t1 == pytest.approx(2.5)  # the slowest rank's time, on every rank
