"""The no-allocation decode entry point (partials in the library's built-in
device scratch, for callers that cannot allocate device memory) against the
workspace entry point and against the oracle, through the C ABI, on two
calls in a row.

Kept in its own file, collected last, so a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import ATOL, LSE_TOL, RTOL, check_close, dev, gpu_cache, oracle_cache, to_dev


@pytest.fixture(scope="module")
def K():
    from fp8_paged_kv_append_gb300 import k16v8
    k16v8.load_library()
    return k16v8


def _run_both(K, w, chunk):
    kc, vc = gpu_cache(w, K)
    B, hq, d = w.q.shape
    L = int(w.seq_lens.max())
    args = (to_dev(w.q), kc, vc, to_dev(w.v_scale), to_dev(w.block_table), to_dev(w.seq_lens), L,
            w.sm_scale, chunk)
    ws = torch.empty(K.k16v8_decode_workspace_size(B, hq, d, L, chunk), dtype=torch.uint8,
                     device=dev())
    ref_o = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    ref_l = torch.empty((B, hq), dtype=torch.float32, device=dev())
    K.k16v8_paged_decode_attention(*args, ws, ref_o, ref_l)
    results = []
    for _ in range(2):  # the scratch keeps the previous call's contents
        o = torch.full((B, hq, d), float("nan"), dtype=torch.float16, device=dev())
        l = torch.full((B, hq), float("nan"), dtype=torch.float32, device=dev())
        err = torch.zeros(1, dtype=torch.int32, device=dev())
        K.k16v8_paged_decode_attention_static(*args, o, l, err)
        assert K.k16v8_read_device_error(err) == 0
        results.append((o.float().cpu().numpy(), l.cpu().numpy()))
    return ref_o.float().cpu().numpy(), ref_l.cpu().numpy(), results


@pytest.mark.gpu
@pytest.mark.parametrize("maker,chunk", [(workloads.tiny_decode, 64),
                                         (workloads.decode_1k_b32, 384)])
def test_static_scratch_matches_workspace_entry_and_oracle(K, maker, chunk):
    w = maker()
    ref_o, ref_l, results = _run_both(K, w, chunk)
    okc, ovc = oracle_cache(w)
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    for o, l in results:
        assert np.all(np.abs(o - ref_o) <= ATOL + RTOL * np.abs(ref_o))
        assert np.all(np.abs(l - ref_l) <= LSE_TOL)
        check_close(o, ref["out"], l, ref["lse"])


@pytest.mark.gpu
def test_static_scratch_empty_batch_is_accepted(K):
    """batch 0 needs no scratch: accepted like the workspace call (nothing
    launched)."""
    lib = K.load_library()
    st = lib.k16v8_paged_decode_attention_static(None, None, None, None, None, 1, None, 0, 0, 40,
                                                 10, 128, 8, 0.1, 16, None, None, None, None)
    assert st == K.K16V8_OK


@pytest.mark.gpu
def test_static_scratch_rejects_oversized_problem(K):
    """512 sequences x 40 heads x 64 chunks of partials exceed the built-in
    scratch.  The arguments are real (small) device tensors, so a check
    reordered after the launch would fail on the host, not on the GPU."""
    B, chunk, L = 512, 16, 64 * 16
    need = K.k16v8_decode_workspace_size(B, 40, 128, L, chunk)
    assert need > K.STATIC_SCRATCH_BYTES
    w = workloads.make_decode("oversized", 23, [L] * 2)
    kc, vc = gpu_cache(w, K)
    q = torch.zeros((B, 40, 128), dtype=torch.float16, device=dev())
    bt = torch.zeros((B, L // 16), dtype=torch.int32, device=dev())
    lens = torch.zeros(B, dtype=torch.int32, device=dev())
    out = torch.empty((B, 40, 128), dtype=torch.float16, device=dev())
    lse = torch.empty((B, 40), dtype=torch.float32, device=dev())
    with pytest.raises(K.K16V8Error) as e:
        K.k16v8_paged_decode_attention_static(q, kc, vc, to_dev(w.v_scale), bt, lens, L,
                                              w.sm_scale, chunk, out, lse)
    assert e.value.status == K.K16V8_ERR_STATIC_SCRATCH_LIMIT
