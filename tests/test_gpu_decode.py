"""Paged split-KV decode and the LSE merge on the GPU against the oracle.

Tolerance: |out - ref| <= 4e-3 + 4e-3 |ref| elementwise, |lse - ref| <= 1e-4;
bit-exact for the merge's indexing (marker partials)."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import (check_close, dev, gpu_cache, host_bits, oracle_cache, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from fp8_paged_kv_append_gb300 import k16v8
    k16v8.load_library()
    return k16v8


def run_decode(K, w, kc, vc, chunk, err=None, max_seq_len=None, block_table=None,
               seq_lens=None):
    B, hq, d = w.q.shape
    L = w.seq_lens if seq_lens is None else seq_lens
    max_len = int(L.max(initial=0)) if max_seq_len is None else max_seq_len
    ws = torch.zeros(K.k16v8_decode_workspace_size(B, hq, d, max_len, chunk),
                     dtype=torch.uint8, device=dev())
    out = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev())
    bt = w.block_table if block_table is None else block_table
    K.k16v8_paged_decode_attention(to_dev(w.q), kc, vc, to_dev(w.v_scale), to_dev(bt),
                                   to_dev(L), max_len, w.sm_scale, chunk, ws, out, lse, err)
    po, pl = K.workspace_views(ws, B, hq, d, max_len, chunk)
    return out, lse, po, pl


def split_then_merge(K, w, kc, vc, chunk, max_len):
    """The same call as two launches: the split's partials, then the merge."""
    B, hq, d = w.q.shape
    ws = torch.zeros(K.k16v8_decode_workspace_size(B, hq, d, max_len, chunk),
                     dtype=torch.uint8, device=dev())
    K.k16v8_paged_decode_split(to_dev(w.q), kc, vc, to_dev(w.v_scale), to_dev(w.block_table),
                               to_dev(w.seq_lens), max_len, w.sm_scale, chunk, ws)
    po, pl = K.workspace_views(ws, B, hq, d, max_len, chunk)
    out = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev())
    K.k16v8_merge_states(po, pl, to_dev(w.seq_lens), chunk, out, lse)
    return out, lse, po, pl


def compare_workload(K, w, chunk, check_partials=True):
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    kc, vc = gpu_cache(w, K, err)
    okc, ovc = oracle_cache(w)
    hk, hv = host_bits(kc, vc)
    assert np.array_equal(hk, okc.view(np.uint16)) and np.array_equal(hv, ovc)
    out, lse, po, pl = run_decode(K, w, kc, vc, chunk, err)
    assert K.k16v8_read_device_error(err) == 0
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens,
                              w.sm_scale, split_chunk=chunk if check_partials else 0)
    check_close(out.float().cpu().numpy(), ref["out"], lse.cpu().numpy(), ref["lse"])
    max_len = int(w.seq_lens.max(initial=0))
    if check_partials and max_len <= chunk:
        # One chunk: the split kernel wrote the rows itself and no partials
        # (the workspace stays as allocated, zero).  The same call as split +
        # merge gives the same bits, and its partials are checked below.
        assert not torch.any(po) and not torch.any(pl)
        o2, l2, po, pl = split_then_merge(K, w, kc, vc, chunk, max_len)
        assert torch.equal(out.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), l2.view(torch.int32))
    if check_partials:
        nc = -(-w.seq_lens // chunk)
        po_h, pl_h = po.cpu().numpy(), pl.cpu().numpy()
        for b in range(w.batch):
            n = int(nc[b])
            check_close(po_h[b, :, :n], ref["partial_o"][b, :, :n], pl_h[b, :, :n],
                        ref["partial_lse"][b, :, :n])


@pytest.mark.parametrize("chunk", [16, 64, 512, 8192])
def test_decode_tiny(K, chunk):
    compare_workload(K, workloads.tiny_decode(0), chunk)


def test_decode_1k_b32(K):
    compare_workload(K, workloads.decode_1k_b32(), 512)


def test_decode_1k_b32_chunk256(K):
    compare_workload(K, workloads.decode_1k_b32(), 256, check_partials=False)


def test_decode_8k_b16(K):
    compare_workload(K, workloads.decode_8k_b16(), 512)


def test_decode_ragged_edges(K):
    """Lengths 0, 1, 15, 16, 17, a page boundary and a chunk boundary in one
    batch; an empty sequence gives out 0 and lse -inf."""
    lens = [0, 1, 15, 16, 17, 511, 512, 513, 1000]
    w = workloads.make_decode("ragged", 31, lens, num_qo_heads=8, num_kv_heads=2)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    kc, vc = gpu_cache(w, K, err)
    okc, ovc = oracle_cache(w)
    out, lse, _, _ = run_decode(K, w, kc, vc, 512, err)
    assert K.k16v8_read_device_error(err) == 0
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    check_close(o, ref["out"], l, ref["lse"])


@pytest.mark.parametrize("maker,chunk", [
    (lambda: workloads.make_decode("ragged", 33, [0, 1, 15, 16, 17, 511, 512, 513, 1000],
                                   num_qo_heads=8, num_kv_heads=2), 1008),
    (workloads.decode_1k_b32, 1152),
    (workloads.decode_1k_b32, 8192)])
def test_decode_single_chunk_writes_output_directly(K, maker, chunk):
    """Lengths that fit one chunk: the combined call launches the split kernel
    alone, which writes out / lse (an empty sequence: 0 and -inf), bit-equal
    to the split + merge of its one partial and within tolerance of the
    oracle."""
    compare_workload(K, maker(), chunk)


def test_decode_uniform_keys_gives_mean_of_values(K):
    w = workloads.make_decode("uniform", 32, [300, 77], num_qo_heads=4, num_kv_heads=1)
    w.k_tok[:] = w.k_tok[0]
    kc, vc = gpu_cache(w, K)
    okc, ovc = oracle_cache(w)
    out, lse, _, _ = run_decode(K, w, kc, vc, 64)
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    check_close(out.float().cpu().numpy(), ref["out"], lse.cpu().numpy(), ref["lse"])


def test_decode_bad_page_id_is_flagged_not_dereferenced(K):
    w = workloads.tiny_decode(5)
    kc, vc = gpu_cache(w, K)
    bt = w.block_table.copy()
    bt[1, 3] = w.num_pages + 1000
    bt[0, 0] = -7
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    run_decode(K, w, kc, vc, 64, err, block_table=bt)
    assert K.k16v8_read_device_error(err) & K.DEVERR_PAGE


def test_decode_seq_len_beyond_hint_is_flagged(K):
    w = workloads.tiny_decode(6)
    kc, vc = gpu_cache(w, K)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    lens = w.seq_lens.copy()
    lens[1] = w.block_table.shape[1] * 16 + 5  # beyond the page table
    run_decode(K, w, kc, vc, 64, err, max_seq_len=int(w.seq_lens.max()), seq_lens=lens)
    assert K.k16v8_read_device_error(err) & K.DEVERR_SEQLEN


def test_merge_indexing_bit_exact(K):
    """Marker partials: row r, chunk c holds values that encode (r, c); one
    live chunk per row must come out exactly (fp16-representable markers)."""
    B, H, C, D, chunk = 3, 8, 5, 128, 64
    rng = np.random.Generator(np.random.PCG64(40))
    lens = np.array([C * chunk, 3 * chunk - 7, 1], np.int32)
    nc = -(-lens // chunk)
    po = np.zeros((B, H, C, D), np.float32)
    pl = np.full((B, H, C), -np.inf, np.float32)
    live = np.zeros((B, H), np.int64)
    for b in range(B):
        for h in range(H):
            c = int(rng.integers(0, nc[b]))
            live[b, h] = c
            for cc in range(C):
                po[b, h, cc] = (b * 64 + h * 8 + cc) + np.arange(D) / 256.0
            pl[b, h, c] = np.float32(0.375 * h)
    out = torch.empty((B, H, D), dtype=torch.float16, device=dev())
    lse = torch.empty((B, H), dtype=torch.float32, device=dev())
    K.k16v8_merge_states(to_dev(po), to_dev(pl), to_dev(lens), chunk, out, lse)
    o = out.cpu().numpy()
    for b in range(B):
        for h in range(H):
            exp = po[b, h, live[b, h]].astype(np.float16)
            assert np.array_equal(o[b, h], exp), (b, h)
    assert np.array_equal(lse.cpu().numpy(), pl.max(axis=2))
    # against the oracle merge on random partials
    po = rng.standard_normal((B, H, C, D)).astype(np.float32)
    pl = (rng.standard_normal((B, H, C)) * 3).astype(np.float32)
    K.k16v8_merge_states(to_dev(po), to_dev(pl), to_dev(lens), chunk, out, lse)
    ro, rl = oracle.merge(po.astype(np.float64), pl.astype(np.float64), nc)
    check_close(out.float().cpu().numpy(), ro, lse.cpu().numpy(), rl)


def _page_sum_stress(seed):
    """Near-uniform scores (queries scaled by 0.1: softmax weights within a
    page between about 0.3 and 1, so every product p*v carries many
    significant bits) over values that all quantise to the extreme codes
    +-448: every per-page product sum the kernels accumulate in fp16 runs up
    to 16 x 448 = 7,168, where an fp16 ulp is 4.  Even KV heads hold +v only
    (no cancellation: the largest sums), odd heads random signs.  Lengths 1,
    16, 17 and 8,192."""
    w = workloads.make_decode("page-sum stress", seed, [1, 16, 17, 8192])
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    w.q = (w.q.astype(np.float32) * np.float32(0.1)).astype(np.float16)
    sign = np.where(rng.integers(0, 2, w.v_tok.shape) == 1, 1.0, -1.0).astype(np.float32)
    sign[:, 0::2, :] = 1.0
    w.v_tok = (sign * np.float32(0.75)).astype(np.float16)
    w.v_scale = workloads.calibrate_v_scale(w.v_tok)
    return w


@pytest.mark.parametrize("chunk", [16, 512])
def test_decode_fp16_page_sums_at_code_448(K, chunk):
    w = _page_sum_stress(21)
    okc, ovc = oracle_cache(w)
    slots = w.slot_mapping
    written = ovc.transpose(0, 2, 1, 3).reshape(-1, w.num_kv_heads, w.head_dim)[slots]
    assert set(np.unique(written).tolist()) == {0x7E, 0xFE}  # +-448 only
    compare_workload(K, w, chunk)


def test_decode_balanced_fp16_page_sums_at_code_448(K):
    w = _page_sum_stress(22)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    kc, vc = gpu_cache(w, K, err)
    okc, ovc = oracle_cache(w)
    B, hq, d = w.q.shape
    ws = torch.empty(K.k16v8_decode_balanced_workspace_size(B, hq, d), dtype=torch.uint8,
                     device=dev())
    out = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev())
    K.k16v8_paged_decode_attention_balanced(to_dev(w.q), kc, vc, to_dev(w.v_scale),
                                            to_dev(w.block_table), to_dev(w.seq_lens),
                                            w.sm_scale, ws, out, lse, err)
    assert K.k16v8_read_device_error(err) == 0
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    check_close(out.float().cpu().numpy(), ref["out"], lse.cpu().numpy(), ref["lse"])
