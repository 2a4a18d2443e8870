"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks, each with
its own elapsed time and work; the reported figures are the slowest rank's
time and the sum of every rank's units."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, results):
    import torch.distributed as tdist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    ms, units = bench.reduce_over_ranks(10.0 + 5.0 * rank, 1000.0 * (rank + 1))
    results[rank] = (ms, units)
    tdist.barrier()
    tdist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == (15.0, 3000.0) and results[1] == (15.0, 3000.0)


def test_reduce_is_identity_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(7.5, 42) == (7.5, 42.0)
