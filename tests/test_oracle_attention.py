"""Oracle kv_append placement, decode, merge and prefill pinned to library
routines, brute force and closed forms (no GPU)."""
import math

import numpy as np
import pytest

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import (K_POISON, V_POISON, lib_table, library_dequant_v, oracle_cache,
                   sdpa_reference, seq_rows)


@pytest.fixture(scope="module")
def tiny():
    w = workloads.tiny_decode(0)
    kc, vc = oracle_cache(w)
    return w, kc, vc


def test_kv_append_placement_brute_force(tiny):
    w, kc, vc = tiny
    slot = w.slot_mapping
    page, off = slot // 16, slot % 16
    # numpy fancy indexing into the [page, head, offset, d] layout
    assert np.array_equal(kc[page, :, off, :].view(np.uint16), w.k_tok.view(np.uint16))
    x = w.v_tok.astype(np.float32) / w.v_scale[None, :, None]
    import torch
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(vc[page, :, off, :], ref)
    touched = np.zeros(kc.shape[0] * 16, bool)
    touched[slot] = True
    touched = touched.reshape(-1, 16)
    untouched_k = kc.view(np.uint16).transpose(0, 2, 1, 3)[~touched]
    untouched_v = vc.transpose(0, 2, 1, 3)[~touched]
    assert np.all(untouched_k == K_POISON) and np.all(untouched_v == V_POISON)
    assert untouched_k.size > 0


def test_kv_append_skips_negative_slots_and_rejects_out_of_range(tiny):
    w, _, _ = tiny
    kc, vc = oracle_cache(w)
    kc2, vc2 = kc.copy(), vc.copy()
    sm = w.slot_mapping.copy()
    sm[:] = -1
    oracle.kv_append(w.k_tok, w.v_tok, sm, w.v_scale, kc2, vc2)
    assert np.array_equal(kc2.view(np.uint16), kc.view(np.uint16)) and np.array_equal(vc2, vc)
    sm[0] = w.num_pages * 16
    with pytest.raises(oracle.OracleError):
        oracle.kv_append(w.k_tok[:1], w.v_tok[:1], sm[:1], w.v_scale, kc2, vc2)


def _unpaged(w, b):
    lo, hi = seq_rows(w.seq_lens)[b]
    k = w.k_tok[lo:hi].astype(np.float64).transpose(1, 0, 2)
    v = library_dequant_v(w.v_tok[lo:hi], w.v_scale).transpose(1, 0, 2)
    return k, v


def test_decode_matches_library_sdpa_unpaged(tiny):
    w, kc, vc = tiny
    r = oracle.paged_decode(w.q, kc, vc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    for b in range(w.batch):
        k, v = _unpaged(w, b)
        q = w.q[b].astype(np.float64)[:, None, :]
        out, lse = sdpa_reference(q, k, v, w.sm_scale)
        np.testing.assert_allclose(r["out"][b], out[:, 0], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(r["lse"][b], lse[:, 0], rtol=1e-12, atol=1e-12)


def test_decode_gqa_mapping_detects_swapped_heads(tiny):
    # q heads 0..3 read KV head 0, 4..7 read KV head 1: swapping the KV heads
    # of the reference must break agreement (guards the head index).
    w, kc, vc = tiny
    r = oracle.paged_decode(w.q, kc, vc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    k, v = _unpaged(w, 1)
    out, _ = sdpa_reference(w.q[1].astype(np.float64)[:, None, :], k[::-1], v[::-1], w.sm_scale)
    assert not np.allclose(r["out"][1], out[:, 0], atol=1e-3)


def test_decode_uniform_keys_closed_form():
    w = workloads.make_decode("uniform", 3, [53], num_qo_heads=4, num_kv_heads=1)
    w.k_tok[:] = w.k_tok[0]
    kc, vc = oracle_cache(w)
    r = oracle.paged_decode(w.q, kc, vc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    vdq = library_dequant_v(w.v_tok, w.v_scale)[:, 0, :]
    mean_v = vdq.mean(axis=0)
    k0 = w.k_tok[0, 0].astype(np.float64)
    for h in range(4):
        s = float(w.sm_scale) * float(w.q[0, h].astype(np.float64) @ k0)
        np.testing.assert_allclose(r["out"][0, h], mean_v, rtol=1e-12, atol=1e-13)
        assert abs(r["lse"][0, h] - (s + math.log(53))) < 1e-12


def test_decode_one_hot_score_closed_form():
    L, sel = 77, 41
    w = workloads.make_decode("onehot", 4, [L], num_qo_heads=4, num_kv_heads=1)
    w.q[0, 1:] = w.q[0, 0]
    qv = w.q[0, 0].astype(np.float64)
    w.k_tok[:] = 0
    w.k_tok[sel, 0] = (30.0 * qv / np.linalg.norm(qv)).astype(np.float16)
    kc, vc = oracle_cache(w)
    r = oracle.paged_decode(w.q, kc, vc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    vdq = library_dequant_v(w.v_tok, w.v_scale)[:, 0, :]
    s = float(w.sm_scale) * float(qv @ w.k_tok[sel, 0].astype(np.float64))
    e = math.exp(s)
    others = vdq.sum(axis=0) - vdq[sel]
    expect = (e * vdq[sel] + others) / (e + (L - 1))
    np.testing.assert_allclose(r["out"][0, 0], expect, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["out"][0, 0], vdq[sel], atol=1e-9)
    assert abs(r["lse"][0, 0] - math.log(e + L - 1)) < 1e-12


def test_decode_invariant_under_page_permutation(tiny):
    w, kc, vc = tiny
    r0 = oracle.paged_decode(w.q, kc, vc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    perm = np.random.Generator(np.random.PCG64(9)).permutation(w.num_pages)
    inv = np.argsort(perm)
    kc2, vc2 = kc[perm], vc[perm]  # new page p holds old page perm[p]
    bt2 = np.where(w.block_table >= 0, inv[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    r1 = oracle.paged_decode(w.q, np.ascontiguousarray(kc2), np.ascontiguousarray(vc2),
                             w.v_scale, bt2, w.seq_lens, w.sm_scale)
    assert np.array_equal(r0["out"], r1["out"]) and np.array_equal(r0["lse"], r1["lse"])


@pytest.mark.parametrize("chunk", [16, 48, 512])
def test_split_then_merge_equals_unsplit(tiny, chunk):
    w, kc, vc = tiny
    r = oracle.paged_decode(w.q, kc, vc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale,
                            split_chunk=chunk)
    nc = -(-w.seq_lens // chunk)
    out, lse = oracle.merge(r["partial_o"], r["partial_lse"], nc)
    np.testing.assert_allclose(out, r["out"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, r["lse"], rtol=1e-13, atol=1e-13)
    # chunks past the end are empty: lse -inf, o = 0
    C = r["partial_lse"].shape[2]
    for b in range(w.batch):
        for c in range(int(nc[b]), C):
            assert np.all(np.isneginf(r["partial_lse"][b, :, c]))
            assert np.all(r["partial_o"][b, :, c] == 0)


def test_merge_marker_partials():
    B, H, C, D = 2, 3, 4, 8
    po = np.arange(B * H * C * D, dtype=np.float64).reshape(B, H, C, D)
    pl = np.full((B, H, C), -np.inf)
    pl[0, :, 2] = 0.5                       # single live chunk -> copied
    pl[1, :, 0] = pl[1, :, 3] = 1.25        # two equal chunks -> average
    pl[1, 2, 3] = 1.25 + math.log(3.0)      # weights 1/4, 3/4
    out, lse = oracle.merge(po, pl, np.array([4, 4], np.int32))
    assert np.array_equal(out[0], po[0, :, 2]) and np.all(lse[0] == 0.5)
    np.testing.assert_allclose(out[1, :2], (po[1, :2, 0] + po[1, :2, 3]) / 2, rtol=1e-15)
    np.testing.assert_allclose(out[1, 2], 0.25 * po[1, 2, 0] + 0.75 * po[1, 2, 3], rtol=1e-15)
    np.testing.assert_allclose(lse[1, :2], 1.25 + math.log(2.0), rtol=1e-15)
    # chunks beyond n_chunks are ignored; zero live chunks -> 0 / -inf
    out2, lse2 = oracle.merge(po, pl, np.array([2, 0], np.int32))
    assert np.all(out2 == 0) and np.all(np.isneginf(lse2))


def test_decode_empty_sequence():
    w = workloads.make_decode("empty", 5, [0, 20], num_qo_heads=4, num_kv_heads=1)
    kc, vc = oracle_cache(w)
    r = oracle.paged_decode(w.q, kc, vc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    assert np.all(r["out"][0] == 0) and np.all(np.isneginf(r["lse"][0]))
    assert np.all(np.isfinite(r["out"][1]))


def test_decode_rejects_bad_page_id(tiny):
    w, kc, vc = tiny
    bt = w.block_table.copy()
    bt[1, 2] = w.num_pages
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(w.q, kc, vc, w.v_scale, bt, w.seq_lens, w.sm_scale)


@pytest.fixture(scope="module")
def small_prefill():
    p = workloads.make_prefill("small prefill", 7, [70, 33, 130], chunk=48,
                               num_qo_heads=8, num_kv_heads=2, num_pages=40)
    kc, vc = oracle_cache(p)
    return p, kc, vc


def test_prefill_matches_library_causal_sdpa(small_prefill):
    p, kc, vc = small_prefill
    offs = np.concatenate([[0], np.cumsum(p.prompt_lens.astype(np.int64))])
    for call in p.calls:
        out, lse = oracle.paged_prefill(p.q[call.rows], call.qo_indptr, kc, vc, p.v_scale,
                                        call.block_table, call.seq_lens, p.sm_scale)
        for i, b in enumerate(call.seqs.tolist()):
            lo, hi = int(call.qo_indptr[i]), int(call.qo_indptr[i + 1])
            L = int(call.seq_lens[i])
            base = int(offs[b])
            k = p.k_tok[base:base + L].astype(np.float64).transpose(1, 0, 2)
            v = library_dequant_v(p.v_tok[base:base + L], p.v_scale).transpose(1, 0, 2)
            q = p.q[call.rows[lo:hi]].astype(np.float64).transpose(1, 0, 2)
            qpos = L - (hi - lo) + np.arange(hi - lo)
            mask = np.arange(L)[None, :] <= qpos[:, None]
            ro, rl = sdpa_reference(q, k, v, p.sm_scale, mask)
            np.testing.assert_allclose(out[lo:hi], ro.transpose(1, 0, 2), rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(lse[lo:hi], rl.T, rtol=1e-12, atol=1e-12)


def test_prefill_last_row_equals_decode_and_rows_subset(small_prefill):
    p, kc, vc = small_prefill
    call = p.calls[-1]
    out, lse = oracle.paged_prefill(p.q[call.rows], call.qo_indptr, kc, vc, p.v_scale,
                                    call.block_table, call.seq_lens, p.sm_scale)
    last = call.qo_indptr[1:] - 1
    r = oracle.paged_decode(np.ascontiguousarray(p.q[call.rows][last]), kc, vc, p.v_scale,
                            call.block_table, call.seq_lens, p.sm_scale)
    assert np.array_equal(out[last], r["out"]) and np.array_equal(lse[last], r["lse"])
    sub = np.array([0, 5, int(last[-1])], np.int64)
    o2, l2 = oracle.paged_prefill(p.q[call.rows], call.qo_indptr, kc, vc, p.v_scale,
                                  call.block_table, call.seq_lens, p.sm_scale, rows=sub)
    assert np.array_equal(o2, out[sub]) and np.array_equal(l2, lse[sub])


def test_prefill_chunked_equals_unchunked():
    a = workloads.make_prefill("a", 8, [100, 64], chunk=32, num_qo_heads=4,
                               num_kv_heads=1, num_pages=20)
    kc, vc = oracle_cache(a)
    full_o = {}
    for call in a.calls:
        o, l = oracle.paged_prefill(a.q[call.rows], call.qo_indptr, kc, vc, a.v_scale,
                                    call.block_table, call.seq_lens, a.sm_scale)
        for r, oo, ll in zip(call.rows.tolist(), o, l):
            full_o[r] = (oo, ll)
    offs = np.concatenate([[0], np.cumsum(a.prompt_lens.astype(np.int64))]).astype(np.int32)
    o, l = oracle.paged_prefill(a.q, offs, kc, vc, a.v_scale, a.block_table,
                                a.prompt_lens, a.sm_scale)
    for r in range(a.q.shape[0]):
        assert np.array_equal(full_o[r][0], o[r]) and np.array_equal(full_o[r][1], l[r])


def test_fp16_kv_control_decode_matches_library_sdpa():
    """FP16-KV control (values stored exactly in fp16): placement and
    attention pinned to numpy indexing and torch SDPA."""
    w = workloads.make_decode("v16", 12, [45, 130], num_qo_heads=8, num_kv_heads=2, num_pages=20)
    v16 = w.v_tok.astype(np.float16)
    kc = np.full((w.num_pages, 2, 16, 128), 0x7E00, np.uint16).view(np.float16)
    vc = np.full((w.num_pages, 2, 16, 128), 0x7E00, np.uint16).view(np.float16)
    oracle.kv_append_v16(w.k_tok, v16, w.slot_mapping, kc, vc)
    page, off = w.slot_mapping // 16, w.slot_mapping % 16
    assert np.array_equal(vc[page, :, off, :].view(np.uint16), v16.view(np.uint16))
    out, lse = oracle.paged_decode_v16(w.q, kc, vc, w.block_table, w.seq_lens, w.sm_scale)
    for b in range(w.batch):
        lo, hi = seq_rows(w.seq_lens)[b]
        k = w.k_tok[lo:hi].astype(np.float64).transpose(1, 0, 2)
        v = v16[lo:hi].astype(np.float64).transpose(1, 0, 2)
        ro, rl = sdpa_reference(w.q[b].astype(np.float64)[:, None, :], k, v, w.sm_scale)
        np.testing.assert_allclose(out[b], ro[:, 0], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl[:, 0], rtol=1e-12, atol=1e-12)
