"""Shared helpers for the tests: caches built by the oracle from the seeded
workload arrays, unpaged reference tensors, tolerances."""
import numpy as np
import torch

import oracle

K_POISON = np.uint16(0x7E00)   # fp16 NaN
V_POISON = np.uint8(0x7F)      # E4M3 NaN

# Attention output tolerance |out - ref| <= ATOL + RTOL*|ref|, LSE |d| <= LSE_TOL
ATOL = 4e-3
RTOL = 4e-3
LSE_TOL = 1e-4


def poisoned_caches(num_pages, hkv, d, page=16):
    kc = np.full((num_pages, hkv, page, d), K_POISON, np.uint16).view(np.float16)
    vc = np.full((num_pages, hkv, page, d), V_POISON, np.uint8)
    return kc, vc


def oracle_cache(w):
    """Caches of a DecodeInputs/PrefillInputs built by the oracle's kv_append."""
    kc, vc = poisoned_caches(w.num_pages, w.num_kv_heads, w.head_dim, w.page_size)
    oracle.kv_append(w.k_tok, w.v_tok, w.slot_mapping, w.v_scale, kc, vc, w.page_size)
    return kc, vc


def lib_table():
    return (torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
            .to(torch.float64).numpy())


def library_dequant_v(v_tok, v_scale):
    """Dequantised values from the library fp8 cast (inputs stay below 464)."""
    x = v_tok.astype(np.float32) / v_scale.astype(np.float32)[None, :, None]
    assert np.abs(x).max() < 464
    codes = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return lib_table()[codes] * v_scale.astype(np.float64)[None, :, None]


def seq_rows(seq_lens):
    offs = np.concatenate([[0], np.cumsum(seq_lens.astype(np.int64))])
    return [(int(offs[b]), int(offs[b + 1])) for b in range(len(seq_lens))]


def sdpa_reference(q, k, v, sm_scale, mask=None):
    """torch scaled_dot_product_attention in float64 on unpaged tensors.
    q [Hq, Tq, D], k/v [Hkv, Tk, D] (GQA expanded here); returns out
    [Hq, Tq, D] and lse [Hq, Tq] via library matmul + logsumexp."""
    hq, hk = q.shape[0], k.shape[0]
    qt = torch.from_numpy(np.ascontiguousarray(q, np.float64))
    kt = torch.from_numpy(np.ascontiguousarray(k, np.float64)).repeat_interleave(hq // hk, 0)
    vt = torch.from_numpy(np.ascontiguousarray(v, np.float64)).repeat_interleave(hq // hk, 0)
    m = None if mask is None else torch.from_numpy(mask)
    out = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=m, scale=float(sm_scale))
    s = torch.matmul(qt, kt.transpose(-1, -2)) * float(sm_scale)
    if m is not None:
        s = s.masked_fill(~m, float("-inf"))
    return out.numpy(), torch.logsumexp(s, dim=-1).numpy()


def check_close(out, ref, lse=None, lse_ref=None, atol=ATOL, rtol=RTOL, lse_tol=LSE_TOL):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(out - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outputs off; worst err "
                           f"{err.max():.3e} (bound there {bound.flat[err.argmax()]:.3e})")
    if lse is not None:
        lse = np.asarray(lse, np.float64)
        lse_ref = np.asarray(lse_ref, np.float64)
        inf = np.isinf(lse_ref)
        assert np.array_equal(np.isinf(lse), inf)
        d = np.abs(lse[~inf] - lse_ref[~inf])
        assert d.size == 0 or d.max() <= lse_tol, f"lse err {d.max():.3e}"


# ---- GPU-side helpers (torch only moves memory; compute is in libk16v8) ----

def dev():
    return torch.device("cuda:0")


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def gpu_poisoned_caches(num_pages, hkv, d, page=16):
    kc = torch.full((num_pages, hkv, page, d), int(np.int16(K_POISON.view(np.int16))),
                    dtype=torch.int16, device=dev()).view(torch.float16)
    vc = torch.full((num_pages, hkv, page, d), int(V_POISON), dtype=torch.uint8, device=dev())
    return kc, vc


def gpu_cache(w, K, err=None):
    """Caches of a workload written by the library's kv_append."""
    kc, vc = gpu_poisoned_caches(w.num_pages, w.num_kv_heads, w.head_dim, w.page_size)
    K.k16v8_kv_append(to_dev(w.k_tok), to_dev(w.v_tok), to_dev(w.slot_mapping),
                      to_dev(w.v_scale), kc, vc, err)
    return kc, vc


def host_bits(kc, vc):
    return (kc.view(torch.int16).cpu().numpy().view(np.uint16), vc.cpu().numpy())
