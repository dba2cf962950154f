"""Oracle pool sizing against the slot counts printed on the subject page."""
import json
import os

import oracle
from fp8_paged_kv_append_gb300 import workloads

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pool_slots.json")))


def test_bytes_per_token_from_geometry():
    # FP16 keys (2 B) + E4M3 values (1 B) vs FP16 keys and values (2 + 2 B).
    assert GOLD["kv_heads"] * GOLD["head_dim"] * 3 == GOLD["k16v8_bytes_per_token"]
    assert GOLD["kv_heads"] * GOLD["head_dim"] * 4 == GOLD["fp16_bytes_per_token"]


def test_pool_slots_match_printed_figures():
    s8 = oracle.pool_slots(GOLD["budget_bytes"], GOLD["layers"],
                           GOLD["k16v8_bytes_per_token"], GOLD["page_size"])
    s16 = oracle.pool_slots(GOLD["budget_bytes"], GOLD["layers"],
                            GOLD["fp16_bytes_per_token"], GOLD["page_size"])
    assert s8 == GOLD["k16v8_slots_per_layer"]
    assert s16 == GOLD["fp16_slots_per_layer"]
    assert s8 % 16 == 0 and s16 % 16 == 0
    # "approximately one third more"
    assert abs(s8 / s16 - 4.0 / 3.0) < 1e-3


def test_workload_pool_sizing_agrees():
    assert workloads.pool_pages_per_layer() * 16 == GOLD["k16v8_slots_per_layer"]
    assert workloads.pool_pages_per_layer(v_bytes=2) * 16 == GOLD["fp16_slots_per_layer"]
