"""Load-balanced decode (one full wave of equal CTA ranges over the flat
(sequence, KV head, page) tile list) on the GPU against the oracle.

Tolerance as for the chunked decode: |out - ref| <= 4e-3 + 4e-3 |ref|,
|lse - ref| <= 1e-4.  The work plan the kernel stores (tile total, tiles per
CTA, per-sequence page offsets) is integer work and is checked bit-exactly
against a numpy restatement of the rule."""
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


def ctas():
    return torch.cuda.get_device_properties(0).multi_processor_count * 4


def expected_plan(seq_lens, hkv, max_pages):
    L = np.clip(np.asarray(seq_lens, np.int64), 0, max_pages * 16)
    np_b = -(-L // 16)
    P = np.concatenate([[0], np.cumsum(np_b)])
    T = int(P[-1]) * hkv
    W = max(-(-T // ctas()), 4)
    return T, W, P


def run_balanced(K, w, kc, vc, err=None, block_table=None, seq_lens=None, flags=0):
    B, hq, d = w.q.shape
    n = K.k16v8_decode_balanced_workspace_size(B, hq, d)
    assert n > 0
    ws = torch.full((n,), 0xA5, dtype=torch.uint8, device=dev())  # contents must not matter
    out = torch.full((B, hq, d), float("nan"), dtype=torch.float16, device=dev())
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device=dev())
    bt = w.block_table if block_table is None else block_table
    L = w.seq_lens if seq_lens is None else seq_lens
    K.k16v8_paged_decode_attention_balanced(to_dev(w.q), kc, vc, to_dev(w.v_scale), to_dev(bt),
                                            to_dev(L), w.sm_scale, ws, out, lse, err, flags=flags)
    return out, lse, ws


def compare(K, w, flags=0):
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    kc, vc = gpu_cache(w, K, err)
    okc, ovc = oracle_cache(w)
    out, lse, ws = run_balanced(K, w, kc, vc, err, flags=flags)
    assert K.k16v8_read_device_error(err) == 0
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    check_close(out.float().cpu().numpy(), ref["out"], lse.cpu().numpy(), ref["lse"])
    T, W, P = expected_plan(w.seq_lens, w.num_kv_heads, w.block_table.shape[1])
    plan = ws[: 4 * (w.batch + 3)].cpu().numpy().view(np.int32)
    assert plan[0] == T and plan[1] == W
    assert np.array_equal(plan[2:3 + w.batch], P)
    return T, W


def test_balanced_tiny(K):
    compare(K, workloads.tiny_decode(0))


@pytest.mark.parametrize("flags", [0, 1])
def test_balanced_1k_b32(K, flags):
    T, W = compare(K, workloads.decode_1k_b32(), flags)
    assert W < int(np.min(-(-workloads.decode_1k_b32().seq_lens // 16)))  # segments are cut


@pytest.mark.parametrize("flags", [0, 1])
def test_balanced_8k_b16(K, flags):
    compare(K, workloads.decode_8k_b16(), flags)


def test_balanced_ragged_whole_and_cut_segments(K):
    """Many short sequences (held whole by one CTA, written directly) mixed
    with long ones (cut between CTAs, merged), zero-length sequences among
    them, and lengths on and off page boundaries."""
    rng = np.random.Generator(np.random.PCG64(71))
    lens = rng.integers(0, 80, 300).astype(np.int32)
    lens[[3, 50, 51, 299]] = 0
    lens[[10, 150]] = [4000, 2500]
    lens[[20, 21, 22]] = [1, 16, 17]
    w = workloads.make_decode("balanced ragged", 72, lens, num_qo_heads=8, num_kv_heads=2)
    T, W = compare(K, w, flags=1)
    _, _, P = expected_plan(w.seq_lens, w.num_kv_heads, w.block_table.shape[1])
    whole = cut = 0
    for b in range(w.batch):
        n = int(P[b + 1] - P[b])
        for g in range(w.num_kv_heads):
            if n:
                s0 = int(P[b]) * w.num_kv_heads + g * n
                if s0 // W == (s0 + n - 1) // W:
                    whole += 1
                else:
                    cut += 1
    assert whole > 0 and cut > 0


def test_balanced_all_empty(K):
    w = workloads.make_decode("empty", 73, [5, 0, 0], num_qo_heads=8, num_kv_heads=2)
    kc, vc = gpu_cache(w, K)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    out, lse, _ = run_balanced(K, w, kc, vc, err, seq_lens=np.zeros(3, np.int32))
    assert K.k16v8_read_device_error(err) == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_balanced_max_batch_scan(K):
    """8192 sequences: the in-kernel scan runs over 64 tiles of 128."""
    rng = np.random.Generator(np.random.PCG64(74))
    lens = rng.integers(0, 40, 8192).astype(np.int32)
    w = workloads.make_decode("8192 short", 75, lens, num_qo_heads=4, num_kv_heads=1)
    compare(K, w, flags=1)


def test_balanced_fullpool_layer_sampled(K):
    """One layer of the full-pool ragged batch (64 sequences, L in [1, 8192]):
    sampled sequences against the oracle (pages copied to the host before
    any kernel runs)."""
    lay = workloads.fullpool_layout(seed=4)
    kc, vc, vs = workloads.device_layer_pool(2024, lay.num_pages, dev())
    B = len(lay.seq_lens)
    rng = np.random.Generator(np.random.PCG64(76))
    q = rng.standard_normal((B, 40, 128), dtype=np.float32).astype(np.float16)
    order = np.argsort(lay.seq_lens)
    seqs = sorted({int(order[0]), int(order[1]), int(order[-1]), int(order[B // 2]), 7, 33})
    host = {}
    for b in seqs:
        n = -(-int(lay.seq_lens[b]) // 16)
        pages = torch.from_numpy(lay.block_table[b, :n].astype(np.int64)).to(dev())
        host[b] = (kc[pages].cpu().numpy(), vc[pages].cpu().numpy())
    vs_h = vs.cpu().numpy()
    n = K.k16v8_decode_balanced_workspace_size(B, 40, 128)
    ws = torch.empty(n, dtype=torch.uint8, device=dev())
    out = torch.empty((B, 40, 128), dtype=torch.float16, device=dev())
    lse = torch.empty((B, 40), dtype=torch.float32, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    K.k16v8_paged_decode_attention_balanced(to_dev(q), kc, vc, vs, to_dev(lay.block_table),
                                            to_dev(lay.seq_lens), 1 / np.sqrt(128), ws, out, lse,
                                            err)
    assert K.k16v8_read_device_error(err) == 0
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in seqs:
        hk, hv = host[b]
        bt = np.arange(hk.shape[0], dtype=np.int32)[None, :]
        r = oracle.paged_decode(q[b:b + 1], hk, hv, vs_h, bt,
                                np.array([lay.seq_lens[b]], np.int32), 1 / np.sqrt(128))
        check_close(o[b], r["out"][0], l[b], r["lse"][0])


def test_balanced_bad_page_id_is_flagged(K):
    w = workloads.tiny_decode(5)
    kc, vc = gpu_cache(w, K)
    bt = w.block_table.copy()
    bt[1, 3] = w.num_pages + 1000
    bt[0, 0] = -7
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    run_balanced(K, w, kc, vc, err, block_table=bt)
    assert K.k16v8_read_device_error(err) & K.DEVERR_PAGE


def test_balanced_seq_len_beyond_table_is_flagged(K):
    w = workloads.tiny_decode(6)
    kc, vc = gpu_cache(w, K)
    lens = w.seq_lens.copy()
    lens[1] = w.block_table.shape[1] * 16 + 5
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    run_balanced(K, w, kc, vc, err, seq_lens=lens)
    assert K.k16v8_read_device_error(err) & K.DEVERR_SEQLEN


def test_balanced_host_checks(K):
    w = workloads.tiny_decode(0)
    kc, vc = gpu_cache(w, K)
    B, hq, d = w.q.shape
    n = K.k16v8_decode_balanced_workspace_size(B, hq, d)
    small = torch.empty(n - 256, dtype=torch.uint8, device=dev())
    out = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    with pytest.raises(K.K16V8Error) as e:
        K.k16v8_paged_decode_attention_balanced(to_dev(w.q), kc, vc, to_dev(w.v_scale),
                                                to_dev(w.block_table), to_dev(w.seq_lens),
                                                w.sm_scale, small, out)
    assert e.value.status == K.K16V8_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(K.K16V8Error) as e:
        K.k16v8_paged_decode_attention_balanced(to_dev(w.q), kc, vc, to_dev(w.v_scale),
                                                to_dev(w.block_table), to_dev(w.seq_lens),
                                                w.sm_scale, small, out, flags=2)
    assert e.value.status == K.K16V8_ERR_INVALID_ARG
    assert K.k16v8_decode_balanced_workspace_size(8193, hq, d) == 0
    assert K.k16v8_decode_balanced_workspace_size(B, hq, 64) == 0


def test_metadata_ready_flag_in_a_graph_is_bit_identical(K):
    """The decode step as the bench and MultiLayerDecode run it: the fused
    load-balanced split and its merge captured in one CUDA graph, steps back
    to back (programmatic launch overlap between them), once with the
    block table and lengths read before the wait on the preceding kernel
    (K16V8_DECODE_METADATA_READY) and once without.  Outputs, LSEs and cache
    bytes must be bit-identical, and match the oracle."""
    w = workloads.decode_1k_b32()
    nr = w.new_rows
    B, hq, d = w.q.shape
    results = []
    for flags in (0, K.DECODE_METADATA_READY):
        kc, vc = gpu_cache(w, K)
        ws = torch.empty(K.k16v8_decode_balanced_workspace_size(B, hq, d), dtype=torch.uint8,
                         device=dev())
        out = torch.full((B, hq, d), float("nan"), dtype=torch.float16, device=dev())
        lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device=dev())
        err = torch.zeros(1, dtype=torch.int32, device=dev())
        args = (to_dev(w.q), to_dev(w.k_tok[nr]), to_dev(w.v_tok[nr].astype(np.float16)), kc, vc,
                to_dev(w.v_scale), to_dev(w.block_table), to_dev(w.seq_lens), w.sm_scale, ws)

        def step():
            K.k16v8_paged_decode_append_balanced_split(*args, out, lse, err, flags=flags)
            K.k16v8_merge_balanced(ws, w.num_kv_heads, out, lse)

        step()  # eager run configures the kernels
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream(), capture_error_mode="thread_local"):
            for _ in range(4):
                step()
        out.fill_(float("nan"))
        g.replay()
        assert K.k16v8_read_device_error(err) == 0
        results.append((out.clone(), lse.clone(), kc.clone(), vc.clone()))
    (o0, l0, k0, v0), (o1, l1, k1, v1) = results
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert torch.equal(k0.view(torch.int16), k1.view(torch.int16)) and torch.equal(v0, v1)
    okc, ovc = oracle_cache(w)
    ref = oracle.paged_decode(w.q, okc, ovc, w.v_scale, w.block_table, w.seq_lens, w.sm_scale)
    check_close(o1.float().cpu().numpy(), ref["out"], l1.cpu().numpy(), ref["lse"])
