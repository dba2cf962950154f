"""The oracle: a plain float64 CPU restatement of the K16/V8 paged attention
path.  TEST INFRASTRUCTURE ONLY -- the tests, the smoke check and the
benchmark's CPU-baseline leg use it; the product path never imports it.

The arithmetic lives in ``k16v8_oracle.c`` (plain C11, float64); this module
builds it with gcc when needed and wraps it with ctypes and numpy.  It shares
no code with the CUDA library.  Inputs come from the seeded generators in
``fp8_paged_kv_append_gb300.workloads`` and are passed in as numpy arrays.

Subject page: "Phi-4: quality transfer and interrupted throughput studies"
(intro: K16/V8 storage format, geometry, pool sizes; "Matched diagnostic
profiles": attention, merge and compressed-cache write kernels).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k16v8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libk16v8_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-D_DEFAULT_SOURCE"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (idempotent).  Returns the library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.k16v8o_half_to_double.argtypes = [ctypes.c_uint16]
            lib.k16v8o_half_to_double.restype = f64
            lib.k16v8o_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.k16v8o_e4m3_to_double.restype = f64
            lib.k16v8o_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.k16v8o_e4m3_from_float.restype = ctypes.c_uint8
            lib.k16v8o_quantize_value.argtypes = [ctypes.c_float, ctypes.c_float]
            lib.k16v8o_quantize_value.restype = ctypes.c_uint8
            lib.k16v8o_e4m3_encode_n.argtypes = [P, P, i64]
            lib.k16v8o_e4m3_encode_n.restype = None
            lib.k16v8o_quantize_n.argtypes = [P, ctypes.c_float, P, i64]
            lib.k16v8o_quantize_n.restype = None
            lib.k16v8o_pool_slots.argtypes = [f64, i32, i64, i32]
            lib.k16v8o_pool_slots.restype = i64
            lib.k16v8o_kv_append.argtypes = [P, i64, P, i32, i64, P, i32, P, P, P,
                                             i32, i32, i32, i32]
            lib.k16v8o_kv_append.restype = ctypes.c_int
            lib.k16v8o_paged_decode.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32,
                                                i32, i32, i32, f64, i32, i32, P, P, P,
                                                P, i32]
            lib.k16v8o_paged_decode.restype = ctypes.c_int
            lib.k16v8o_paged_decode_v16.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32,
                                                    i32, i32, f64, P, P, i32]
            lib.k16v8o_paged_decode_v16.restype = ctypes.c_int
            lib.k16v8o_kv_append_v16.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32]
            lib.k16v8o_kv_append_v16.restype = ctypes.c_int
            lib.k16v8o_merge.argtypes = [P, P, P, i32, i32, i32, i32, P, P]
            lib.k16v8o_merge.restype = ctypes.c_int
            lib.k16v8o_paged_prefill.argtypes = [P, P, i32, P, P, P, P, i32, P, i32,
                                                 i32, i32, i32, i32, f64, P, i64, P, P,
                                                 i32]
            lib.k16v8o_paged_prefill.restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what}: oracle returned status {rc}")


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _bits16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype in (np.float16, np.uint16, np.int16)
    return a.view(np.uint16)


# ---- number formats -------------------------------------------------------

def half_to_double(bits: int) -> float:
    return _load().k16v8o_half_to_double(int(bits) & 0xFFFF)


def e4m3_to_double(code: int) -> float:
    return _load().k16v8o_e4m3_to_double(int(code) & 0xFF)


def e4m3_decode_table() -> np.ndarray:
    """float64 value of each of the 256 E4M3FN codes (NaN for 0x7F, 0xFF)."""
    lib = _load()
    return np.array([lib.k16v8o_e4m3_to_double(c) for c in range(256)], np.float64)


def e4m3_from_float(x: float) -> int:
    return int(_load().k16v8o_e4m3_from_float(float(np.float32(x))))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    """Element-wise fp32 -> E4M3 code (uint8)."""
    xf = np.ascontiguousarray(np.asarray(x, np.float32).ravel())
    out = np.empty(xf.shape, np.uint8)
    _load().k16v8o_e4m3_encode_n(_ptr(xf), _ptr(out), xf.size)
    return out.reshape(np.shape(x))


def quantize_array(v: np.ndarray, scale: float) -> np.ndarray:
    """Element-wise E4M3(fl32(v / scale)) for fp16 or fp32 v."""
    vf = np.ascontiguousarray(np.asarray(v).astype(np.float32).ravel())
    out = np.empty(vf.shape, np.uint8)
    _load().k16v8o_quantize_n(_ptr(vf), float(np.float32(scale)), _ptr(out), vf.size)
    return out.reshape(np.shape(v))


def quantize_value(v: float, scale: float) -> int:
    return int(_load().k16v8o_quantize_value(float(np.float32(v)),
                                             float(np.float32(scale))))


# ---- pool sizing ------------------------------------------------------------

def pool_slots(budget_bytes: float, layers: int, bytes_per_token: int,
               page_size: int = 16) -> int:
    return int(_load().k16v8o_pool_slots(float(budget_bytes), layers,
                                         bytes_per_token, page_size))


# ---- kv_append --------------------------------------------------------------

def kv_append(k: np.ndarray, v: np.ndarray, slot_mapping: np.ndarray,
              v_scale: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
              page_size: int = 16) -> None:
    """Write tokens into the caches in place.  k: fp16 [T, Hkv, D]; v: fp16 or
    fp32 [T, Hkv, D]; slot_mapping int64 [T]; v_scale fp32 [Hkv];
    k_cache fp16 [P, Hkv, page, D]; v_cache uint8 same shape."""
    T, Hkv, D = k.shape
    assert v.shape == k.shape and k_cache.shape[1:] == (Hkv, page_size, D)
    assert v_cache.shape == k_cache.shape and v_cache.dtype == np.uint8
    kb = _bits16(k)
    v = np.ascontiguousarray(v)
    v_is_f32 = int(v.dtype == np.float32)
    vb = v if v_is_f32 else _bits16(v)
    sm = np.ascontiguousarray(slot_mapping, np.int64)
    vs = np.ascontiguousarray(v_scale, np.float32)
    kc = k_cache.view(np.uint16)
    rc = _load().k16v8o_kv_append(_ptr(kb), Hkv * D, _ptr(vb), v_is_f32, Hkv * D,
                                  _ptr(sm), T, _ptr(vs), _ptr(kc), _ptr(v_cache),
                                  k_cache.shape[0], Hkv, D, page_size)
    _check(rc, "kv_append")


# ---- decode -----------------------------------------------------------------

def paged_decode(q, k_cache, v_cache, v_scale, block_table, seq_lens, sm_scale,
                 split_chunk: int = 0, page_size: int = 16, nthreads: int = 0,
                 want_full: bool = True):
    """Exact float64 attention over the paged cache.

    Returns dict with ``out`` [B,Hq,D], ``lse`` [B,Hq] (natural log) and, when
    split_chunk > 0, ``partial_o`` [B,Hq,C,D] / ``partial_lse`` [B,Hq,C] with
    C = ceil(max(seq_lens) / split_chunk)."""
    qb = _bits16(q)
    B, Hq, D = q.shape
    P, Hkv = k_cache.shape[:2]
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    vs = np.ascontiguousarray(v_scale, np.float32)
    res = {}
    out = lse = po = pl = None
    if want_full:
        out = np.zeros((B, Hq, D), np.float64)
        lse = np.zeros((B, Hq), np.float64)
        res.update(out=out, lse=lse)
    C = 0
    if split_chunk > 0:
        C = max(1, -(-int(sl.max(initial=0)) // split_chunk))
        po = np.zeros((B, Hq, C, D), np.float64)
        pl = np.zeros((B, Hq, C), np.float64)
        res.update(partial_o=po, partial_lse=pl)
    rc = _load().k16v8o_paged_decode(
        _ptr(qb), _ptr(k_cache.view(np.uint16)), _ptr(v_cache), _ptr(vs), _ptr(bt),
        bt.shape[1], _ptr(sl), B, Hq, Hkv, D, page_size, P, float(sm_scale),
        split_chunk, C, _ptr(out), _ptr(lse), _ptr(po), _ptr(pl), nthreads)
    _check(rc, "paged_decode")
    return res


def kv_append_v16(k, v, slot_mapping, k_cache, v_cache16, page_size: int = 16) -> None:
    """FP16-KV control cache write: K and V copied (v fp16 [T, Hkv, D])."""
    T, Hkv, D = k.shape
    kb, vb = _bits16(k), _bits16(np.asarray(v).astype(np.float16))
    sm = np.ascontiguousarray(slot_mapping, np.int64)
    rc = _load().k16v8o_kv_append_v16(_ptr(kb), _ptr(vb), _ptr(sm), T,
                                      _ptr(k_cache.view(np.uint16)),
                                      _ptr(v_cache16.view(np.uint16)), k_cache.shape[0], Hkv, D,
                                      page_size)
    _check(rc, "kv_append_v16")


def paged_decode_v16(q, k_cache, v_cache16, block_table, seq_lens, sm_scale, page_size=16,
                     nthreads: int = 0):
    """FP16-KV control: exact attention over a cache with fp16 values."""
    qb = _bits16(q)
    B, Hq, D = q.shape
    P, Hkv = k_cache.shape[:2]
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = _load().k16v8o_paged_decode_v16(
        _ptr(qb), _ptr(k_cache.view(np.uint16)), _ptr(v_cache16.view(np.uint16)), _ptr(bt),
        bt.shape[1], _ptr(sl), B, Hq, Hkv, D, page_size, P, float(sm_scale), _ptr(out),
        _ptr(lse), nthreads)
    _check(rc, "paged_decode_v16")
    return out, lse


def merge(partial_o: np.ndarray, partial_lse: np.ndarray, n_chunks: np.ndarray):
    """Log-sum-exp merge of the first n_chunks[b] partials of each row."""
    po = np.ascontiguousarray(partial_o, np.float64)
    pl = np.ascontiguousarray(partial_lse, np.float64)
    nc = np.ascontiguousarray(n_chunks, np.int32)
    B, Hq, C, D = po.shape
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = _load().k16v8o_merge(_ptr(po), _ptr(pl), _ptr(nc), B, Hq, C, D,
                              _ptr(out), _ptr(lse))
    _check(rc, "merge")
    return out, lse


# ---- prefill ----------------------------------------------------------------

def paged_prefill(q, qo_indptr, k_cache, v_cache, v_scale, block_table, seq_lens,
                  sm_scale, rows=None, page_size: int = 16, nthreads: int = 0):
    """Causal attention of ragged query rows against the paged cache.
    rows: optional int64 array of query-row indices to evaluate."""
    qb = _bits16(q)
    Tq, Hq, D = q.shape
    P, Hkv = k_cache.shape[:2]
    qi = np.ascontiguousarray(qo_indptr, np.int32)
    B = qi.shape[0] - 1
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    vs = np.ascontiguousarray(v_scale, np.float32)
    r = None if rows is None else np.ascontiguousarray(rows, np.int64)
    n = Tq if r is None else r.shape[0]
    out = np.zeros((n, Hq, D), np.float64)
    lse = np.zeros((n, Hq), np.float64)
    rc = _load().k16v8o_paged_prefill(
        _ptr(qb), _ptr(qi), B, _ptr(k_cache.view(np.uint16)), _ptr(v_cache),
        _ptr(vs), _ptr(bt), bt.shape[1], _ptr(sl), Hq, Hkv, D, page_size, P,
        float(sm_scale), _ptr(r), n, _ptr(out), _ptr(lse), nthreads)
    _check(rc, "paged_prefill")
    return out, lse
