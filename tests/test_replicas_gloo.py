"""Multi-process path of bench.py (replicas only): two gloo ranks on the CPU
check the max-over-ranks time and the summed work units."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    ms, units = bench.aggregate(1.5 + rank, 100.0 * (rank + 1))
    bench.barrier()
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_aggregate_max_time_sum_units_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, ms, units in res:
        assert ms == pytest.approx(2.5) and units == pytest.approx(300.0)


def test_aggregate_single_process_passthrough():
    import bench
    assert bench.aggregate(3.0, 7.0) == (3.0, 7.0)
