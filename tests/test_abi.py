"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

from fp8_paged_kv_append_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    libbuild.build()
    from fp8_paged_kv_append_gb300 import k16v8
    k16v8.load_library()
    return k16v8


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(k16v8_\w+)\s*\(", txt))
    return names


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ["k16v8_kv_append", "k16v8_paged_decode_split", "k16v8_merge_states",
              "k16v8_paged_decode_attention", "k16v8_decode_workspace_size"]:
        assert n in names


def test_library_exports_every_declared_symbol(K):
    lib = ctypes.CDLL(K.LIB_PATH)
    for n in declared_symbols():
        assert hasattr(lib, n), n
        assert n in K.SIGNATURES, f"binding lacks {n}"


def test_status_strings(K):
    assert K.status_string(0) == "ok"
    assert "workspace" in K.status_string(3)
    assert K.status_string(99) == "unknown status"


def test_workspace_size_and_layout(K):
    B, H, D, L, C = 16, 40, 128, 8300, 512
    chunks = -(-L // C)
    o_bytes = B * H * chunks * D * 4
    lse_bytes = B * H * chunks * 4
    r256 = lambda x: -(-x // 256) * 256
    assert K.k16v8_decode_workspace_size(B, H, D, L, C) == r256(o_bytes) + r256(lse_bytes)
    assert K.k16v8_decode_workspace_layout(B, H, D, L, C) == (0, r256(o_bytes), chunks)
    assert K.k16v8_decode_workspace_size(B, H, D, 0, C) > 0  # one chunk minimum
    assert K.k16v8_decode_workspace_size(B, H, D, L, 24) == 0  # not a page multiple


def test_host_validation_without_gpu(K):
    lib = K.load_library()
    # head_dim 64 is not supported
    assert lib.k16v8_kv_append(1, 0, 1, 0, 0, 1, 4, 1, 1, 1, 8, 2, 64, None, None) == 2
    # bad v dtype
    assert lib.k16v8_kv_append(1, 0, 1, 7, 0, 1, 4, 1, 1, 1, 8, 2, 128, None, None) == 1
    # zero tokens is a no-op
    assert lib.k16v8_kv_append(None, 0, None, 0, 0, None, 0, None, None, None, 8, 2, 128,
                               None, None) == 0
    # GQA group other than 4
    args = [1, 1, 1, 1, 1, 4, 1, 64, 2, 8, 4, 128, 8, 0.1, 64, 1, 1 << 20, None, None]
    assert lib.k16v8_paged_decode_split(*args) == 2
    args[10] = 2  # 8 query heads over 2 KV heads
    args[14] = 40  # split not a page multiple
    assert lib.k16v8_paged_decode_split(*args) == 1
    args[14] = 64
    args[5] = 2  # max_pages_per_seq too small for max_seq_len
    assert lib.k16v8_paged_decode_split(*args) == 1
    args[5] = 4
    args[16] = 16  # workspace too small
    assert lib.k16v8_paged_decode_split(*args) == 3
    assert lib.k16v8_merge_states(1, 1, 2, 8, 1, 64, 1, 64, 1, None, None) == 2
    assert lib.k16v8_merge_states(1, 1, -1, 8, 1, 128, 1, 64, 1, None, None) == 1


def declared_parameter_counts():
    """Number of parameters of every k16v8_* function the headers declare."""
    counts = {}
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            txt = re.sub(r"//[^\n]*", "", txt)
            for m in re.finditer(r"\b(k16v8_\w+)\s*\(([^;{]*?)\)\s*;", txt, flags=re.S):
                params = m.group(2).strip()
                counts[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_binding_signatures_match_header_parameter_counts():
    """Every ctypes signature takes as many arguments as the C declaration, so
    a parameter added on one side only fails here, on the CPU."""
    from fp8_paged_kv_append_gb300 import k16v8
    counts = declared_parameter_counts()
    assert len(counts) >= 20
    for name, n in counts.items():
        assert name in k16v8.SIGNATURES, name
        assert len(k16v8.SIGNATURES[name][1]) == n, (name, n, len(k16v8.SIGNATURES[name][1]))


def test_host_validation_of_split_prefill_and_fused_balanced_without_gpu(K):
    """The newer entry points refuse bad arguments before any CUDA call."""
    lib = K.load_library()
    # k16v8_paged_prefill_attention_split: kv_splits / max_seq_len < 0, then shapes
    pre = [1, 1, 64, 64, 1, 1, 1, 1, 8, 1, 1, 40, 10, 128, 100, 0.1, 0, 0, None, 0, 1, None,
           None, None]
    pre[16] = -1
    assert lib.k16v8_paged_prefill_attention_split(*pre) == 1
    pre[16], pre[17] = 0, -1
    assert lib.k16v8_paged_prefill_attention_split(*pre) == 1
    pre[17], pre[13] = 0, 64  # head_dim 64
    assert lib.k16v8_paged_prefill_attention_split(*pre) == 2
    pre[13], pre[12] = 128, 40  # 40 query heads over 40 KV heads: GQA group 1
    assert lib.k16v8_paged_prefill_attention_split(*pre) == 2
    pre[12] = 10  # valid shape, but the pointers are not 16-byte aligned
    assert lib.k16v8_paged_prefill_attention_split(*pre) == 1
    # k16v8_prefill_workspace_size: 0 for what the call would refuse
    assert lib.k16v8_prefill_workspace_size(1024, 1, 40, 10, 64, 0, 0) == 0
    assert lib.k16v8_prefill_workspace_size(1024, 1, 40, 10, 128, -1, 0) == 0
    assert lib.k16v8_prefill_workspace_size(1024, 1, 40, 10, 128, 0, -1) == 0
    assert lib.k16v8_prefill_workspace_size(0, 1, 40, 10, 128, 0, 0) == 0
    # k16v8_paged_decode_append_balanced_split: shapes and batch bound
    dec = [1, 1, 1, 1, 1, 1, 1, 8, 1, 4, 40, 10, 64, 100, 0.1, 1, 1 << 20, 1, None, 0, None,
           None]
    assert lib.k16v8_paged_decode_append_balanced_split(*dec) == 2  # head_dim 64
    dec[12], dec[9] = 128, 8193
    assert lib.k16v8_paged_decode_append_balanced_split(*dec) == 1  # batch above 8192
    assert lib.k16v8_decode_balanced_workspace_size(8193, 40, 128) == 0
