"""Decode with the new token's cache write fused into the attention kernel:
the cache bytes must equal the oracle's append (bit-exact, whole pool), and
the outputs the oracle's append-then-attend (tolerance as for decode)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import check_close, dev, gpu_poisoned_caches, host_bits, oracle_cache, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from fp8_paged_kv_append_gb300 import k16v8
    k16v8.load_library()
    return k16v8


def cache_without_new_tokens(w, K):
    """GPU and oracle caches holding every token except each sequence's last."""
    keep = np.ones(w.k_tok.shape[0], bool)
    keep[w.new_rows[w.new_rows >= 0]] = False
    kc, vc = gpu_poisoned_caches(w.num_pages, w.num_kv_heads, w.head_dim)
    idx = np.flatnonzero(keep)
    K.k16v8_kv_append(to_dev(w.k_tok[idx]), to_dev(w.v_tok[idx]), to_dev(w.slot_mapping[idx]),
                      to_dev(w.v_scale), kc, vc)
    from cases import poisoned_caches
    okc, ovc = poisoned_caches(w.num_pages, w.num_kv_heads, w.head_dim)
    oracle.kv_append(w.k_tok[idx], w.v_tok[idx], w.slot_mapping[idx], w.v_scale, okc, ovc)
    return kc, vc, okc, ovc


@pytest.mark.parametrize("maker,chunk", [
    (lambda: workloads.make_decode("ragged", 51, [1, 16, 17, 200, 513, 1000], num_qo_heads=8,
                                   num_kv_heads=2), 64),
    (workloads.decode_1k_b32, 384),
    (workloads.decode_8k_b16, 512)])
def test_fused_append_decode_matches_oracle(K, maker, chunk):
    w = maker()
    w.v_tok = w.v_tok.astype(np.float16)  # decode activations are fp16
    kc, vc, okc, ovc = cache_without_new_tokens(w, K)
    B, hq, d = w.q.shape
    L = int(w.seq_lens.max())
    nr = w.new_rows
    ws = torch.empty(K.k16v8_decode_workspace_size(B, hq, d, L, chunk), dtype=torch.uint8,
                     device=dev())
    out = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    K.k16v8_paged_decode_append_attention(
        to_dev(w.q), to_dev(w.k_tok[nr]), to_dev(w.v_tok[nr]), kc, vc, to_dev(w.v_scale),
        to_dev(w.block_table), to_dev(w.seq_lens), L, w.sm_scale, chunk, ws, out, lse, err)
    assert K.k16v8_read_device_error(err) == 0
    oracle.kv_append(w.k_tok[nr], w.v_tok[nr], w.slot_mapping[nr], w.v_scale, okc, ovc)
    hk, hv = host_bits(kc, vc)
    assert np.array_equal(hk, okc.view(np.uint16)) and np.array_equal(hv, ovc)
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    check_close(out.float().cpu().numpy(), ref["out"], lse.cpu().numpy(), ref["lse"])


def test_fused_append_equals_separate_append(K):
    w = workloads.decode_1k_b32(7)
    kc, vc, _, _ = cache_without_new_tokens(w, K)
    kc2, vc2 = kc.clone(), vc.clone()
    B, hq, d = w.q.shape
    L, chunk, nr = int(w.seq_lens.max()), 384, w.new_rows
    ws = torch.empty(K.k16v8_decode_workspace_size(B, hq, d, L, chunk), dtype=torch.uint8,
                     device=dev())
    o1 = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    o2 = torch.empty_like(o1)
    args = (to_dev(w.v_scale), to_dev(w.block_table), to_dev(w.seq_lens), L, w.sm_scale, chunk)
    K.k16v8_paged_decode_append_attention(to_dev(w.q), to_dev(w.k_tok[nr]), to_dev(w.v_tok[nr]),
                                          kc, vc, *args, ws, o1)
    K.k16v8_kv_append(to_dev(w.k_tok[nr]), to_dev(w.v_tok[nr]), to_dev(w.slot_mapping[nr]),
                      to_dev(w.v_scale), kc2, vc2)
    K.k16v8_paged_decode_attention(to_dev(w.q), kc2, vc2, *args, ws, o2)
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16)) and torch.equal(vc, vc2)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("maker", [
    lambda: workloads.make_decode("ragged with empty", 53, [1, 0, 16, 17, 200, 0, 513, 1000],
                                  num_qo_heads=8, num_kv_heads=2),
    workloads.decode_1k_b32])
def test_fused_append_single_chunk_writes_output_directly(K, maker):
    """Lengths that fit one chunk: the fused split writes the cache row and the
    output itself (one launch).  Cache bytes and outputs equal the fused
    split + merge bit for bit; outputs match the oracle."""
    w = maker()
    w.v_tok = w.v_tok.astype(np.float16)
    kc, vc, okc, ovc = cache_without_new_tokens(w, K)
    kc2, vc2 = kc.clone(), vc.clone()
    B, hq, d = w.q.shape
    L = int(w.seq_lens.max())
    has_new = w.new_rows >= 0
    nr = np.where(has_new, w.new_rows, 0)  # rows of empty sequences are never read
    chunk = -(-L // 16) * 16
    ws = torch.zeros(K.k16v8_decode_workspace_size(B, hq, d, L, chunk), dtype=torch.uint8,
                     device=dev())
    ws2 = torch.zeros_like(ws)
    o1 = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    l1 = torch.empty((B, hq), dtype=torch.float32, device=dev())
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    kn = to_dev(np.ascontiguousarray(w.k_tok[nr]))
    vn = to_dev(np.ascontiguousarray(w.v_tok[nr]))
    args = (to_dev(w.v_scale), to_dev(w.block_table), to_dev(w.seq_lens), L, w.sm_scale, chunk)
    K.k16v8_paged_decode_append_attention(to_dev(w.q), kn, vn, kc, vc, *args, ws, o1, l1, err)
    assert not torch.any(ws)  # no partials written
    K.k16v8_paged_decode_append_split(to_dev(w.q), kn, vn, kc2, vc2, *args, ws2, err)
    po, pl = K.workspace_views(ws2, B, hq, d, L, chunk)
    K.k16v8_merge_states(po, pl, to_dev(w.seq_lens), chunk, o2, l2)
    assert K.k16v8_read_device_error(err) == 0
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16)) and torch.equal(vc, vc2)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    sel = w.new_rows[has_new]
    oracle.kv_append(w.k_tok[sel], w.v_tok[sel], w.slot_mapping[sel], w.v_scale, okc, ovc)
    hk, hv = host_bits(kc, vc)
    assert np.array_equal(hk, okc.view(np.uint16)) and np.array_equal(hv, ovc)
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    check_close(o1.float().cpu().numpy(), ref["out"], l1.cpu().numpy(), ref["lse"])


@pytest.mark.parametrize("maker,flags", [
    (lambda: workloads.make_decode("ragged with empty", 52, [1, 0, 16, 17, 200, 0, 513, 1000],
                                   num_qo_heads=8, num_kv_heads=2), 0),
    (workloads.decode_1k_b32, 1),
    (workloads.decode_8k_b16, 1)])
def test_fused_append_balanced_matches_oracle(K, maker, flags):
    """The load-balanced split with the append folded in: cache bytes equal
    the oracle's append (whole pool, bit-exact), outputs its decode."""
    w = maker()
    w.v_tok = w.v_tok.astype(np.float16)
    kc, vc, okc, ovc = cache_without_new_tokens(w, K)
    B, hq, d = w.q.shape
    has_new = w.new_rows >= 0
    nr = np.where(has_new, w.new_rows, 0)  # rows of empty sequences are never read
    ws = torch.empty(K.k16v8_decode_balanced_workspace_size(B, hq, d), dtype=torch.uint8,
                     device=dev())
    out = torch.full((B, hq, d), float("nan"), dtype=torch.float16, device=dev())
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    k_new = np.ascontiguousarray(w.k_tok[nr])
    v_new = np.ascontiguousarray(w.v_tok[nr])
    K.k16v8_paged_decode_append_attention_balanced(
        to_dev(w.q), to_dev(k_new), to_dev(v_new), kc, vc, to_dev(w.v_scale),
        to_dev(w.block_table), to_dev(w.seq_lens), w.sm_scale, ws, out, lse, err, flags=flags)
    assert K.k16v8_read_device_error(err) == 0
    sel = w.new_rows[has_new]
    oracle.kv_append(w.k_tok[sel], w.v_tok[sel], w.slot_mapping[sel], w.v_scale, okc, ovc)
    hk, hv = host_bits(kc, vc)
    assert np.array_equal(hk, okc.view(np.uint16)) and np.array_equal(hv, ovc)
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    check_close(out.float().cpu().numpy(), ref["out"], lse.cpu().numpy(), ref["lse"])


def test_fused_append_balanced_equals_separate_append(K):
    """Same cache bytes and bit-identical outputs as kv_append followed by
    the load-balanced decode."""
    w = workloads.decode_1k_b32(8)
    kc, vc, _, _ = cache_without_new_tokens(w, K)
    kc2, vc2 = kc.clone(), vc.clone()
    B, hq, d = w.q.shape
    nr = w.new_rows
    ws = torch.empty(K.k16v8_decode_balanced_workspace_size(B, hq, d), dtype=torch.uint8,
                     device=dev())
    o1 = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    o2 = torch.empty_like(o1)
    l1 = torch.empty((B, hq), dtype=torch.float32, device=dev())
    l2 = torch.empty_like(l1)
    args = (to_dev(w.v_scale), to_dev(w.block_table), to_dev(w.seq_lens), w.sm_scale, ws)
    K.k16v8_paged_decode_append_attention_balanced(
        to_dev(w.q), to_dev(w.k_tok[nr]), to_dev(w.v_tok[nr].astype(np.float16)), kc, vc, *args,
        o1, l1)
    K.k16v8_kv_append(to_dev(w.k_tok[nr]), to_dev(w.v_tok[nr].astype(np.float16)),
                      to_dev(w.slot_mapping[nr]), to_dev(w.v_scale), kc2, vc2)
    K.k16v8_paged_decode_attention_balanced(to_dev(w.q), kc2, vc2, *args, o2, l2)
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16)) and torch.equal(vc, vc2)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_fused_append_balanced_host_checks(K):
    w = workloads.tiny_decode(0)
    B, hq, d = w.q.shape
    kc, vc = gpu_poisoned_caches(w.num_pages, w.num_kv_heads, w.head_dim)
    ws = torch.empty(K.k16v8_decode_balanced_workspace_size(B, hq, d), dtype=torch.uint8,
                     device=dev())
    out = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    kn = torch.zeros((B, w.num_kv_heads, d), dtype=torch.float16, device=dev())
    with pytest.raises(K.K16V8Error) as e:  # v_new missing
        K.k16v8_paged_decode_append_balanced_split(
            to_dev(w.q), kn, None, kc, vc, to_dev(w.v_scale), to_dev(w.block_table),
            to_dev(w.seq_lens), w.sm_scale, ws, out)
    assert e.value.status == K.K16V8_ERR_INVALID_ARG


def test_fused_append_balanced_bad_page_is_flagged(K):
    """A rejected page id on the page that receives the new token: flagged,
    and that row lands nowhere in the pool (every other byte as the oracle's
    append of the other sequences' tokens)."""
    w = workloads.tiny_decode(5)
    w.v_tok = w.v_tok.astype(np.float16)
    kc, vc, okc, ovc = cache_without_new_tokens(w, K)
    B, hq, d = w.q.shape
    bt = w.block_table.copy()
    last = (int(w.seq_lens[1]) - 1) // 16
    bt[1, last] = w.num_pages + 3
    nr = w.new_rows
    ws = torch.empty(K.k16v8_decode_balanced_workspace_size(B, hq, d), dtype=torch.uint8,
                     device=dev())
    out = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    K.k16v8_paged_decode_append_attention_balanced(
        to_dev(w.q), to_dev(w.k_tok[nr]), to_dev(w.v_tok[nr]), kc, vc, to_dev(w.v_scale),
        to_dev(bt), to_dev(w.seq_lens), w.sm_scale, ws, out, None, err)
    assert K.k16v8_read_device_error(err) & K.DEVERR_PAGE
    oracle.kv_append(w.k_tok[nr[:1]], w.v_tok[nr[:1]], w.slot_mapping[nr[:1]], w.v_scale, okc, ovc)
    hk, hv = host_bits(kc, vc)
    assert np.array_equal(hk, okc.view(np.uint16)) and np.array_equal(hv, ovc)
