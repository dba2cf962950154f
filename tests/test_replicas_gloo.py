"""Multi-process path of bench.py (replicas only): gloo ranks on the CPU run
bench.main's rank set-up with a stand-in for the GPU section, and check the
max-over-ranks time, the summed work units, that every rank ran the same
workload, and that rank 0 alone prints the JSON line."""
import contextlib
import io
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
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


def _stub_measure(config_for_rank):
    """Stand-in for bench.measure_gpu: fixed per-rank times and units."""
    def measure(args, rank, world, local_rank):
        return {"ms": 2.0 + rank, "units": 1.0e9, "e2e": (3.0 + rank, 100, 50),
                "config": config_for_rank(rank),
                "fields": {"gpu_launches": 80 * args.steps, "rank_seen": rank,
                           "local_rank_seen": local_rank}}
    return measure


def _main_rank(rank, world, port, q, same_config):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    cfg = (lambda r: {"workload": "w"}) if same_config else (lambda r: {"workload": f"w{r}"})
    buf = io.StringIO()
    err = None
    try:
        with contextlib.redirect_stdout(buf):
            bench.main(["--gpus", str(world), "--steps", "4", "--warmup", "3"],
                       backend="gloo", measure=_stub_measure(cfg))
    except RuntimeError as e:
        err = str(e)
    q.put((rank, buf.getvalue(), err))


def _run_main(world, same_config):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_main_rank, args=(r, world, port, q, same_config))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    return sorted(q.get(timeout=10) for _ in range(world))


def test_bench_main_two_ranks_rank0_prints_aggregate():
    res = _run_main(2, same_config=True)
    (r0, out0, err0), (r1, out1, err1) = res
    assert err0 is None and err1 is None
    assert out1 == ""  # rank 1 prints nothing
    lines = [l for l in out0.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["scaling"] == "weak"
    assert d["ms_per_step"] == pytest.approx(3.0)  # max over ranks
    assert d["value"] == pytest.approx(2.0e9 / 3.0e-3 / 1e9, rel=1e-3)  # summed units
    assert d["e2e"]["ms_per_step"] == pytest.approx(4.0)
    assert d["config"] == {"workload": "w"}
    assert d["rank_seen"] == 0 and d["local_rank_seen"] == 0


def test_bench_main_rejects_ranks_with_different_workloads():
    res = _run_main(2, same_config=False)
    for rank, out, err in res:
        assert err is not None and "different workloads" in err
        assert out == ""
