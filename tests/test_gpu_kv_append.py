"""kv_append on the GPU against the oracle: bit-exact cache bytes and page
placement over the whole pool (untouched slots keep their poison)."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import (K_POISON, V_POISON, dev, gpu_cache, gpu_poisoned_caches, host_bits,
                   oracle_cache, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from fp8_paged_kv_append_gb300 import k16v8
    k16v8.load_library()
    return k16v8


def assert_same_pool(kc, vc, okc, ovc):
    hk, hv = host_bits(kc, vc)
    assert np.array_equal(hk, okc.view(np.uint16)), "k_cache bytes differ"
    assert np.array_equal(hv, ovc), "v_cache bytes differ"


@pytest.mark.parametrize("maker", [workloads.tiny_decode, workloads.decode_1k_b32])
def test_kv_append_bit_exact(K, maker):
    w = maker()
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    kc, vc = gpu_cache(w, K, err)
    okc, ovc = oracle_cache(w)
    assert_same_pool(kc, vc, okc, ovc)
    assert K.k16v8_read_device_error(err) == 0


def test_kv_append_prefill_sized_batch(K):
    p = workloads.prefill_8x1k()
    kc, vc = gpu_cache(p, K)
    okc, ovc = oracle_cache(p)
    assert_same_pool(kc, vc, okc, ovc)


def test_kv_append_strided_fused_qkv_rows(K):
    """k and v as column slices of a fused [T, (Hq + 2 Hkv) * D] projection."""
    w = workloads.tiny_decode(3)
    T, hkv, d = w.k_tok.shape
    hq = w.num_qo_heads
    rng = np.random.Generator(np.random.PCG64(21))
    fused = rng.standard_normal((T, (hq + 2 * hkv) * d)).astype(np.float16)
    fused[:, hq * d:(hq + hkv) * d] = w.k_tok.reshape(T, -1)
    fused[:, (hq + hkv) * d:] = w.v_tok.astype(np.float16).reshape(T, -1)
    fd = to_dev(fused)
    k_view = fd[:, hq * d:(hq + hkv) * d].view(T, hkv, d)
    v_view = fd[:, (hq + hkv) * d:].view(T, hkv, d)
    kc, vc = gpu_poisoned_caches(w.num_pages, hkv, d)
    K.k16v8_kv_append(k_view, v_view, to_dev(w.slot_mapping), to_dev(w.v_scale), kc, vc)
    from cases import poisoned_caches
    okc, ovc = poisoned_caches(w.num_pages, hkv, d)
    oracle.kv_append(w.k_tok, w.v_tok.astype(np.float16), w.slot_mapping, w.v_scale, okc, ovc)
    assert_same_pool(kc, vc, okc, ovc)


def test_kv_append_padding_and_out_of_range_slots(K):
    w = workloads.tiny_decode(4)
    sm = w.slot_mapping.copy()
    sm[::3] = -1                       # padding tokens are skipped
    bad = np.flatnonzero(sm >= 0)[:2]
    sm[bad[0]] = w.num_pages * 16      # one past the pool
    sm[bad[1]] = 1 << 40               # far out
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    kc, vc = gpu_poisoned_caches(w.num_pages, w.num_kv_heads, w.head_dim)
    K.k16v8_kv_append(to_dev(w.k_tok), to_dev(w.v_tok), to_dev(sm), to_dev(w.v_scale),
                      kc, vc, err)
    assert K.k16v8_read_device_error(err) & K.DEVERR_SLOT
    sm_ok = sm.copy()
    sm_ok[bad] = -1
    from cases import poisoned_caches
    okc, ovc = poisoned_caches(w.num_pages, w.num_kv_heads, w.head_dim)
    oracle.kv_append(w.k_tok, w.v_tok, sm_ok, w.v_scale, okc, ovc)
    assert_same_pool(kc, vc, okc, ovc)


def test_kv_append_special_values(K):
    """NaN, infinities, overflow, subnormal-range values, signed zeros and
    exact E4M3 midpoints through the fp32 and fp16 value paths."""
    table = oracle.e4m3_decode_table()
    fin = table[np.isfinite(table)]
    pos = np.unique(fin[fin >= 0])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 448, 449, 464, 465, 1e30,
                         -1e30, 2 ** -10, 2 ** -11, 3 * 2 ** -11, 1e-40, -1e-45], np.float32)
    vals = np.concatenate([specials, mids, -mids, np.nextafter(mids, np.float32(1e9))])
    n = -(-vals.size // 128) * 128
    vals = np.concatenate([vals, np.zeros(n - vals.size, np.float32)])
    T = n // 128
    v = vals.reshape(T, 1, 128)
    k = np.zeros((T, 1, 128), np.float16)
    slots = np.arange(T, dtype=np.int64)
    P = -(-T // 16)
    for vdtype in (np.float32, np.float16):
        vv = v.astype(vdtype)
        scale = np.array([1.0], np.float32)
        kc, vc = gpu_poisoned_caches(P, 1, 128)
        K.k16v8_kv_append(to_dev(k), to_dev(vv), to_dev(slots), to_dev(scale), kc, vc)
        from cases import poisoned_caches
        okc, ovc = poisoned_caches(P, 1, 128)
        oracle.kv_append(k, vv, slots, scale, okc, ovc)
        got = vc.cpu().numpy()
        nan_in = np.zeros(P * 16 * 128, bool)
        nan_in[:vv.size] = np.isnan(vv.astype(np.float32).ravel())
        nan_in = nan_in.reshape(got.shape)
        assert np.array_equal(got[~nan_in], ovc[~nan_in])
        assert np.all((got[nan_in] & 0x7F) == 0x7F)


def test_e4m3_rounding_all_fp32_bit_patterns(K):
    """Every one of the 2^32 fp32 bit patterns through kv_append (scale 1) vs
    the oracle's encoder; NaN inputs may map to either NaN code."""
    n_chunk = 1 << 26
    T = n_chunk // 128
    k = torch.zeros((T, 1, 128), dtype=torch.float16, device=dev())
    slots = torch.arange(T, dtype=torch.int64, device=dev())
    scale = torch.ones(1, dtype=torch.float32, device=dev())
    kc = torch.empty((T // 16, 1, 16, 128), dtype=torch.float16, device=dev())
    vc = torch.empty((T // 16, 1, 16, 128), dtype=torch.uint8, device=dev())
    pool = cf.ThreadPoolExecutor(8)
    for c in range(1 << 32 >> 26):
        lo = c * n_chunk
        bits = torch.arange(lo, lo + n_chunk, dtype=torch.int64, device=dev())
        bits = torch.where(bits >= 2 ** 31, bits - 2 ** 32, bits)  # two's complement
        v = bits.to(torch.int32).view(torch.float32).view(T, 1, 128)
        K.k16v8_kv_append(k, v, slots, scale, kc, vc)
        got = vc.view(-1).cpu().numpy()
        x = np.arange(lo, lo + n_chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        parts = np.array_split(np.arange(n_chunk), 8)
        exp = np.empty(n_chunk, np.uint8)

        def enc(ix):
            exp[ix[0]:ix[-1] + 1] = oracle.e4m3_encode_array(x[ix[0]:ix[-1] + 1])
        list(pool.map(enc, parts))
        nan = np.isnan(x)
        assert np.array_equal(got[~nan], exp[~nan]), f"chunk {c}"
        assert np.all((got[nan] & 0x7F) == 0x7F)
