"""The bounded waits' error path, reached without any fault: the test hooks
run the chunked decode split and the prefill kernel with one copy of the
first CTA withheld (nothing issued, no arrival), so that CTA's wait expires
after a short poll limit.  The kernel must report K16V8_DEVERR_TIMEOUT,
drain what it did issue and return; the stream must stay usable, and a
normal call right after it on the same stream must match the oracle."""
import time

import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import check_close, dev, gpu_cache, oracle_cache, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from fp8_paged_kv_append_gb300 import k16v8
    k16v8.load_library()
    return k16v8


def test_decode_split_wait_expiry_reports_and_recovers(K):
    w = workloads.tiny_decode(3)
    kc, vc = gpu_cache(w, K)
    B, hq, d = w.q.shape
    L = int(w.seq_lens.max())
    chunk = 64
    ws = torch.zeros(K.k16v8_decode_workspace_size(B, hq, d, L, chunk), dtype=torch.uint8,
                     device=dev())
    args = (to_dev(w.q), kc, vc, to_dev(w.v_scale), to_dev(w.block_table), to_dev(w.seq_lens),
            L, w.sm_scale, chunk)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    t0 = time.perf_counter()
    K.k16v8_paged_decode_split_wait_test(*args, ws, err)
    v = K.k16v8_read_device_error(err)
    assert v == K.DEVERR_TIMEOUT, v  # the expired wait, and nothing else
    assert time.perf_counter() - t0 < 30.0
    # the same stream, a normal call: complete and correct
    err.zero_()
    out = torch.full((B, hq, d), float("nan"), dtype=torch.float16, device=dev())
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device=dev())
    K.k16v8_paged_decode_attention(*args, ws, out, lse, err)
    assert K.k16v8_read_device_error(err) == 0
    okc, ovc = oracle_cache(w)
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    check_close(out.float().cpu().numpy(), ref["out"], lse.cpu().numpy(), ref["lse"])


def test_prefill_wait_expiry_reports_and_recovers(K):
    # one sequence: 300 cached positions, the last 100 new (3 KV tiles for the
    # last query-tile pair, the CTA that withholds its first tile)
    p = workloads.make_prefill("expiry", 13, [300], chunk=1024, num_qo_heads=8, num_kv_heads=2)
    call = p.calls[0]
    rows = call.rows[200:]
    indptr = np.array([0, 100], np.int32)
    kc, vc = gpu_cache(p, K)
    q = to_dev(p.q[rows])
    vs = to_dev(p.v_scale)
    args = (q, to_dev(indptr), 100, kc, vc, vs, to_dev(call.block_table), to_dev(call.seq_lens),
            p.sm_scale)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device=dev())
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev())
    t0 = time.perf_counter()
    K.k16v8_paged_prefill_attention_wait_test(*args, out, lse, err)
    v = K.k16v8_read_device_error(err)
    assert v == K.DEVERR_TIMEOUT, v
    assert time.perf_counter() - t0 < 30.0
    # rows of the CTAs that did not withhold anything (the first query-tile
    # pair, both KV heads; and KV head 1 of the second pair) are complete
    okc, ovc = oracle_cache(p)
    ro, rl = oracle.paged_prefill(np.ascontiguousarray(p.q[rows]), indptr, okc, ovc, p.v_scale,
                                  call.block_table, call.seq_lens, p.sm_scale)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    check_close(o[:64], ro[:64], l[:64], rl[:64])
    check_close(o[64:, 4:], ro[64:, 4:], l[64:, 4:], rl[64:, 4:])
    # the same stream, a normal call: complete and correct
    err.zero_()
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    K.k16v8_paged_prefill_attention(*args, out, lse, err)
    assert K.k16v8_read_device_error(err) == 0
    check_close(out.float().cpu().numpy(), ro, lse.cpu().numpy(), rl)
