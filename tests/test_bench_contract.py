"""bench.py's reference arm on the CPU: one JSON line with the contract's
keys, on the same metric and config as the GPU arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0

    # same metric and config as the GPU arm's default line (the 40-layer full pool)
    sys.path.insert(0, ROOT)
    import bench
    from fp8_paged_kv_append_gb300 import workloads
    lay = workloads.fullpool_layout(seed=bench.FULLPOOL_SEED)
    assert d["metric"] == bench.METRIC
    assert d["config"] == bench.fullpool_config(lay, 40, "auto")
    assert d["config"]["layers"] == 40 and d["config"]["batch"] == 64


def test_reference_arm_one_layer_workload_config():
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--impl", "reference", "--workload", "1k"])
    w, chunk, sample, desc, config = bench.reference_workload(args)
    assert config == bench.config_of(w, "decode 1K/batch 32", 384, bench.replicas_for(w),
                                     bench.DEFAULT_DECODE)
    assert len(sample) == 2


def test_fullpool_cpu_sample_spans_the_length_range():
    sys.path.insert(0, ROOT)
    import bench
    from fp8_paged_kv_append_gb300 import workloads
    lay = workloads.fullpool_layout(seed=bench.FULLPOOL_SEED)
    w, desc = bench.fullpool_cpu_sample()
    assert w.batch == 8
    assert int(w.seq_lens.min()) == int(lay.seq_lens.min())
    assert int(w.seq_lens.max()) == int(lay.seq_lens.max())
    assert set(w.seq_lens.tolist()) <= set(lay.seq_lens.tolist())
    assert (w.num_qo_heads, w.num_kv_heads, w.head_dim) == (40, 10, 128)


def test_replicas_cover_four_l2():
    sys.path.insert(0, ROOT)
    import bench
    for name in ("1k", "8k"):
        w, _, _ = bench.make_workload(name)
        pool = w.num_pages * w.num_kv_heads * 16 * w.head_dim * 3
        assert bench.replicas_for(w) * pool >= 4 * bench.L2_BYTES


def test_oracle_baselines_report_all_cores_and_one_thread():
    """The host baselines of the default line: the oracle's decode steps on
    every core and on one thread, and the oracle's prefill attention and
    cache write beside the prefill line (tiny workloads here)."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from fp8_paged_kv_append_gb300 import workloads
    w = workloads.make_decode("tiny", 3, [37, 200], num_qo_heads=8, num_kv_heads=2)
    d = bench.run_cpu_baseline(w, 64, np.arange(w.batch), "tiny", budget_s=0.2)
    assert d["kind"] == "oracle" and d["unit"] == "GB/s" and d["cores"] >= 1
    assert d["value"] > 0 and d["single_thread_value"] > 0
    p = workloads.make_prefill("tiny", 4, [70, 33], chunk=64, num_qo_heads=8, num_kv_heads=2)
    d = bench.prefill_cpu_baseline(p, row_stride=4, budget_s=0.2)
    assert d["kind"] == "oracle" and d["unit"] == "TFLOP/s" and d["cores"] >= 1
    assert d["value"] > 0 and d["single_thread_value"] > 0
    assert d["kv_append"]["unit"] == "GB/s" and d["kv_append"]["value"] > 0
