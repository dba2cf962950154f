"""Paged causal prefill on tensor cores against the oracle.

The cache is written call by call by kv_append (as a chunked prefill does),
then each call's queries attend to their prefix.  Tolerance as for decode:
|out - ref| <= 4e-3 + 4e-3 |ref|, |lse - ref| <= 1e-4."""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import check_close, dev, gpu_poisoned_caches, oracle_cache, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from fp8_paged_kv_append_gb300 import k16v8
    k16v8.load_library()
    return k16v8


def run_calls(K, p, rows_to_check=None, err=None, kv_splits=None, max_seq_len_hint=False):
    """Append + prefill for every call of a PrefillInputs; returns
    {call index: (out, lse)} on the host.  kv_splits: None for the plain
    call, else the split call with that count (0 = its own choice) and one
    zero-filled workspace shared by all calls."""
    kc, vc = gpu_poisoned_caches(p.num_pages, p.num_kv_heads, p.head_dim)
    vs = to_dev(p.v_scale)
    ws = None
    if kv_splits is not None:
        n = max(K.k16v8_prefill_workspace_size(int(c.qlens.max()), len(c.seq_lens),
                                               p.num_qo_heads, p.num_kv_heads, p.head_dim,
                                               kv_splits) for c in p.calls)
        ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=dev())
    res = []
    for call in p.calls:
        rows = call.rows
        K.k16v8_kv_append(to_dev(p.k_tok[rows]), to_dev(p.v_tok[rows]),
                          to_dev(p.slot_mapping[rows]), vs, kc, vc, err)
        q = to_dev(p.q[rows])
        out = torch.full(q.shape, float("nan"), dtype=torch.float16, device=dev())
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev())
        if kv_splits is None:
            K.k16v8_paged_prefill_attention(q, to_dev(call.qo_indptr), int(call.qlens.max()), kc,
                                            vc, vs, to_dev(call.block_table),
                                            to_dev(call.seq_lens), p.sm_scale, out, lse, err)
        else:
            K.k16v8_paged_prefill_attention_split(
                q, to_dev(call.qo_indptr), int(call.qlens.max()), kc, vc, vs,
                to_dev(call.block_table), to_dev(call.seq_lens), p.sm_scale, ws, out, lse, err,
                kv_splits=kv_splits, max_seq_len=max_seq_len_hint and int(call.seq_lens.max()))
        res.append((out.float().cpu().numpy(), lse.cpu().numpy()))
    return res


def check_against_oracle(p, res, sample=None, full_calls=()):
    """Every call against the oracle: all rows, or every `sample`-th row plus
    each sequence's last row (all rows of the calls in full_calls)."""
    okc, ovc = oracle_cache(p)
    for ci, call in enumerate(p.calls):
        o, l = res[ci]
        rows = None
        if sample is not None and ci not in full_calls:
            rows = np.unique(np.concatenate([np.arange(0, len(call.rows), sample),
                                             call.qo_indptr[1:] - 1])).astype(np.int64)
        ro, rl = oracle.paged_prefill(np.ascontiguousarray(p.q[call.rows]), call.qo_indptr, okc,
                                      ovc, p.v_scale, call.block_table, call.seq_lens,
                                      p.sm_scale, rows=rows)
        if rows is not None:
            o, l = o[rows], l[rows]
        check_close(o, ro, l, rl)


def test_prefill_small_ragged_chunks(K):
    p = workloads.make_prefill("small", 7, [70, 33, 130, 1, 256], chunk=48, num_qo_heads=8,
                               num_kv_heads=2)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    res = run_calls(K, p, err=err)
    assert K.k16v8_read_device_error(err) == 0
    check_against_oracle(p, res)


def test_prefill_single_long_chunk_tile_edges(K):
    # lengths around the 32-token query tile and 128-token KV tile edges
    p = workloads.make_prefill("edges", 8, [31, 32, 33, 127, 128, 129, 300], chunk=1024,
                               num_qo_heads=8, num_kv_heads=2)
    res = run_calls(K, p)
    check_against_oracle(p, res)


def test_prefill_8x1k(K):
    p = workloads.prefill_8x1k()
    res = run_calls(K, p)
    check_against_oracle(p, res)


def test_prefill_1x8k_in_8_chunks_last_chunk_complete(K):
    """The 8192-token prompt in 8 chunks: every row of the last chunk (prefix
    7,169..8,192 positions), every 41st row of the others."""
    p = workloads.prefill_1x8k()
    res = run_calls(K, p)
    check_against_oracle(p, res, sample=41, full_calls=(len(p.calls) - 1,))


@pytest.mark.parametrize("kv_splits", [None, 4])
def test_prefill_prefix_beyond_staged_page_ids(K, kv_splits):
    """A 9,000-token prompt in chunks of 1,024: the last chunk's query-tile
    pairs see up to 563 pages, more than the kernel stages in shared memory
    (512), so the plain call reads the rest of the page ids from the block
    table in global memory.  Every row of the last chunk is checked; the
    KV-split form (4 parts) runs the same calls with short parts."""
    p = workloads.make_prefill("beyond ids", 12, [9000], chunk=1024, num_qo_heads=8,
                               num_kv_heads=2)
    assert -(-9000 // 16) > 512
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    res = run_calls(K, p, err=err, kv_splits=kv_splits)
    assert K.k16v8_read_device_error(err) == 0
    check_against_oracle(p, res, sample=29, full_calls=(len(p.calls) - 1,))


def test_prefill_bad_page_is_flagged(K):
    p = workloads.make_prefill("bad", 9, [100], chunk=1024, num_qo_heads=8, num_kv_heads=2)
    call = p.calls[0]
    call.block_table = call.block_table.copy()
    call.block_table[0, 2] = p.num_pages + 5
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    run_calls(K, p, err=err)
    assert K.k16v8_read_device_error(err) & K.DEVERR_PAGE


@pytest.mark.parametrize("kv_splits", [2, 3, 4])
def test_prefill_kv_split_forced(K, kv_splits):
    """Long prefixes (up to 4,600 positions: up to 36 KV tiles, so up to 4
    parts of >= 8) and short ones (not split) in the same calls; one
    workspace across the calls, so the per-item counters must come back to
    zero after every call."""
    p = workloads.make_prefill("split", 10, [4600, 2100, 700], chunk=1024, num_qo_heads=8,
                               num_kv_heads=2)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    res = run_calls(K, p, err=err, kv_splits=kv_splits)
    assert K.k16v8_read_device_error(err) == 0
    check_against_oracle(p, res, sample=5)


def test_prefill_1x8k_kv_split_auto_sampled(K):
    """The 8192-token prompt in 8 chunks: 160 items per call on the GPU's SMs,
    so the split call picks more than one part (no length hint here); with
    a length bound the first chunk (prefix <= 1024: 8 KV tiles) is not
    split."""
    p = workloads.prefill_1x8k()
    call = p.calls[-1]
    assert K.k16v8_prefill_workspace_size(int(call.qlens.max()), 1, 40, 10, 128, 0) > 0
    assert K.k16v8_prefill_workspace_size(1024, 1, 40, 10, 128, 0, 1024) == 0
    assert K.k16v8_prefill_workspace_size(1024, 1, 40, 10, 128, 0, 8192) > 0
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    res = run_calls(K, p, err=err, kv_splits=0)
    assert K.k16v8_read_device_error(err) == 0
    check_against_oracle(p, res, sample=41, full_calls=(len(p.calls) - 1,))
    res2 = run_calls(K, p, err=err, kv_splits=0, max_seq_len_hint=True)
    assert K.k16v8_read_device_error(err) == 0
    check_against_oracle(p, res2, sample=41)


def test_prefill_kv_split_host_checks(K):
    p = workloads.make_prefill("hc", 11, [2048], chunk=1024, num_qo_heads=8, num_kv_heads=2)
    call = p.calls[0]
    n = K.k16v8_prefill_workspace_size(1024, 1, 8, 2, 128, 2)
    assert n > 0 and K.k16v8_prefill_workspace_size(1024, 1, 8, 2, 128, 1) == 0
    assert K.k16v8_prefill_workspace_size(1024, 1, 8, 2, 64, 2) == 0
    kc, vc = gpu_poisoned_caches(p.num_pages, p.num_kv_heads, p.head_dim)
    q = to_dev(p.q[call.rows])
    out = torch.empty(q.shape, dtype=torch.float16, device=dev())
    small = torch.zeros(n - 256, dtype=torch.uint8, device=dev())
    args = (q, to_dev(call.qo_indptr), 1024, kc, vc, to_dev(p.v_scale), to_dev(call.block_table),
            to_dev(call.seq_lens), p.sm_scale)
    with pytest.raises(K.K16V8Error) as e:
        K.k16v8_paged_prefill_attention_split(*args, small, out, kv_splits=2)
    assert e.value.status == K.K16V8_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(K.K16V8Error) as e:
        K.k16v8_paged_prefill_attention_split(*args, None, out, kv_splits=2)
    assert e.value.status == K.K16V8_ERR_INVALID_ARG
    with pytest.raises(K.K16V8Error) as e:
        K.k16v8_paged_prefill_attention_split(*args, small, out, kv_splits=-1)
    assert e.value.status == K.K16V8_ERR_INVALID_ARG
    with pytest.raises(K.K16V8Error) as e:
        K.k16v8_paged_prefill_attention_split(*args, small, out, max_seq_len=-1)
    assert e.value.status == K.K16V8_ERR_INVALID_ARG
