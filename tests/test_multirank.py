"""The N>1 bench path on CPU: two gloo ranks reduce their timings (max) and
their work (sum) the way bench.py does under torchrun."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, units = bench.reduce_over_ranks(10.0 + 5 * rank, 100 * (rank + 1))
    q.put((rank, ms, units))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_time_and_total_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, units in res:
        assert ms == 15.0 and units == 300.0


def test_single_process_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.0, 7) == (3.0, 7.0)
