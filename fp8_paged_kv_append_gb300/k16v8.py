"""Thin Python binding of libk16v8.so (the C ABI in include/k16v8.h).

Argument marshalling only: shapes and strides are read from torch tensors,
device pointers and the current CUDA stream are passed through ctypes, and
every status is turned into an exception.  All computation runs in the
library's CUDA kernels; there is no fallback of any kind -- importing this
module on a machine without the built library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libk16v8.so")

K16V8_OK = 0
K16V8_ERR_INVALID_ARG = 1
K16V8_ERR_UNSUPPORTED_SHAPE = 2
K16V8_ERR_WORKSPACE_TOO_SMALL = 3
K16V8_ERR_CUDA = 4
K16V8_ERR_DEVICE_BOUNDS = 5
K16V8_ERR_STATIC_SCRATCH_LIMIT = 6
STATIC_SCRATCH_BYTES = 32 << 20
K16V8_F16 = 0
K16V8_F32 = 1
DECODE_METADATA_READY = 1
DEVERR_SLOT, DEVERR_PAGE, DEVERR_SEQLEN, DEVERR_TIMEOUT, DEVERR_INTERNAL = 1, 2, 4, 8, 16
PAGE_SIZE = 16
HEAD_DIM = 128
MAX_SPLIT_CHUNK = 8192  # K16V8_MAX_SPLIT_CHUNK

# Every symbol include/k16v8.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_i32, _i64, _sz, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "k16v8_kv_append": (_i32, [_P, _i64, _P, _i32, _i64, _P, _i32, _P, _P, _P, _i32, _i32,
                               _i32, _P, _P]),
    "k16v8_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "k16v8_decode_workspace_layout": (_i32, [_i32, _i32, _i32, _i32, _i32,
                                             ctypes.POINTER(_sz), ctypes.POINTER(_sz),
                                             ctypes.POINTER(_i32)]),
    "k16v8_paged_decode_split": (_i32, [_P, _P, _P, _P, _P, _i32, _P, _i32, _i32, _i32, _i32,
                                        _i32, _i32, _f32, _i32, _P, _sz, _P, _P]),
    "k16v8_merge_states": (_i32, [_P, _P, _i32, _i32, _i32, _i32, _P, _i32, _P, _P, _P]),
    "k16v8_paged_decode_attention": (_i32, [_P, _P, _P, _P, _P, _i32, _P, _i32, _i32, _i32,
                                            _i32, _i32, _i32, _f32, _i32, _P, _sz, _P, _P,
                                            _P, _P]),
    "k16v8_paged_decode_attention_static": (_i32, [_P, _P, _P, _P, _P, _i32, _P, _i32, _i32,
                                                   _i32, _i32, _i32, _i32, _f32, _i32, _P, _P,
                                                   _P, _P]),
    "k16v8_paged_decode_append_split": (_i32, [_P, _P, _P, _P, _P, _P, _P, _i32, _P, _i32, _i32,
                                               _i32, _i32, _i32, _i32, _f32, _i32, _P, _sz, _P,
                                               _P]),
    "k16v8_paged_decode_append_attention": (_i32, [_P, _P, _P, _P, _P, _P, _P, _i32, _P, _i32,
                                                   _i32, _i32, _i32, _i32, _i32, _f32, _i32, _P,
                                                   _sz, _P, _P, _P, _P]),
    "k16v8_kv_append_v16": (_i32, [_P, _i64, _P, _i64, _P, _i32, _P, _P, _i32, _i32, _i32, _P,
                                   _P]),
    "k16v8_paged_decode_split_v16": (_i32, [_P, _P, _P, _P, _i32, _P, _i32, _i32, _i32, _i32,
                                            _i32, _i32, _f32, _i32, _P, _sz, _P, _P]),
    "k16v8_paged_decode_attention_v16": (_i32, [_P, _P, _P, _P, _i32, _P, _i32, _i32, _i32,
                                                _i32, _i32, _i32, _f32, _i32, _P, _sz, _P, _P,
                                                _P, _P]),
    "k16v8_paged_prefill_attention": (_i32, [_P, _P, _i32, _i32, _P, _P, _P, _P, _i32, _P,
                                             _i32, _i32, _i32, _i32, _i32, _f32, _P, _P, _P,
                                             _P]),
    "k16v8_prefill_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "k16v8_paged_prefill_attention_split": (_i32, [_P, _P, _i32, _i32, _P, _P, _P, _P, _i32,
                                                   _P, _i32, _i32, _i32, _i32, _i32, _f32,
                                                   _i32, _i32, _P, _sz, _P, _P, _P, _P]),
    "k16v8_decode_balanced_workspace_size": (_sz, [_i32, _i32, _i32]),
    "k16v8_paged_decode_attention_balanced": (_i32, [_P, _P, _P, _P, _P, _i32, _P, _i32, _i32,
                                                     _i32, _i32, _i32, _f32, _P, _sz, _P, _P,
                                                     _i32, _P, _P]),
    "k16v8_paged_decode_balanced_split": (_i32, [_P, _P, _P, _P, _P, _i32, _P, _i32, _i32,
                                                 _i32, _i32, _i32, _f32, _P, _sz, _P, _P, _i32,
                                                 _P, _P]),
    "k16v8_merge_balanced": (_i32, [_P, _sz, _i32, _i32, _i32, _i32, _P, _P, _P]),
    "k16v8_paged_decode_append_balanced_split": (_i32, [_P, _P, _P, _P, _P, _P, _P, _i32, _P,
                                                        _i32, _i32, _i32, _i32, _i32, _f32, _P,
                                                        _sz, _P, _P, _i32, _P, _P]),
    "k16v8_paged_decode_append_attention_balanced": (_i32, [_P, _P, _P, _P, _P, _P, _P, _i32,
                                                            _P, _i32, _i32, _i32, _i32, _i32,
                                                            _f32, _P, _sz, _P, _P, _i32, _P,
                                                            _P]),
    "k16v8_paged_decode_split_wait_test": (_i32, [_P, _P, _P, _P, _P, _i32, _P, _i32, _i32,
                                                  _i32, _i32, _i32, _i32, _f32, _i32, _P, _sz,
                                                  _P, _P]),
    "k16v8_paged_prefill_attention_wait_test": (_i32, [_P, _P, _i32, _i32, _P, _P, _P, _P,
                                                       _i32, _P, _i32, _i32, _i32, _i32, _i32,
                                                       _f32, _P, _P, _P, _P]),
    "k16v8_read_device_error": (_i32, [_P, _P, ctypes.POINTER(_i32)]),
    "k16v8_status_string": (ctypes.c_char_p, [_i32]),
}

_lib = None


class K16V8Error(RuntimeError):
    def __init__(self, name: str, status: int):
        self.status = status
        super().__init__(f"{name}: {status_string(status)} (status {status})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libk16v8.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"libk16v8.so not found at {path}: build it with "
                "`python -m fp8_paged_kv_append_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().k16v8_status_string(int(status)).decode()


k16v8_status_string = status_string


def _check(name: str, status: int) -> None:
    if status != K16V8_OK:
        raise K16V8Error(name, status)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _row_stride(t: torch.Tensor, name: str) -> int:
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name} must be [tokens, heads, head_dim] with dense rows")
    return t.stride(0)


# ---- kv_append ---------------------------------------------------------------

def k16v8_kv_append(k, v, slot_mapping, v_scale, k_cache, v_cache, dev_error=None,
                    stream=None) -> None:
    """k fp16 [T,Hkv,D]; v fp16/fp32 [T,Hkv,D] (token stride may exceed the
    row, e.g. a slice of a fused QKV); slot_mapping int64 [T]; v_scale fp32
    [Hkv]; k_cache fp16 / v_cache uint8 [P,Hkv,16,D]."""
    T, hkv, d = k.shape
    vd = {torch.float16: K16V8_F16, torch.float32: K16V8_F32}[v.dtype]
    st = load_library().k16v8_kv_append(
        _ptr(k), _row_stride(k, "k"), _ptr(v), vd, _row_stride(v, "v"), _ptr(slot_mapping), T,
        _ptr(v_scale), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], hkv, d,
        _ptr(dev_error), _stream(stream))
    _check("k16v8_kv_append", st)


# ---- decode --------------------------------------------------------------------

def k16v8_decode_workspace_size(batch, num_qo_heads, head_dim, max_seq_len, split_chunk) -> int:
    return int(load_library().k16v8_decode_workspace_size(batch, num_qo_heads, head_dim,
                                                          max_seq_len, split_chunk))


def k16v8_decode_workspace_layout(batch, num_qo_heads, head_dim, max_seq_len, split_chunk):
    """(partial_o byte offset, partial_lse byte offset, max_chunks)."""
    o, l, c = _sz(), _sz(), _i32()
    st = load_library().k16v8_decode_workspace_layout(
        batch, num_qo_heads, head_dim, max_seq_len, split_chunk,
        ctypes.byref(o), ctypes.byref(l), ctypes.byref(c))
    _check("k16v8_decode_workspace_layout", st)
    return o.value, l.value, c.value


def workspace_views(workspace, batch, num_qo_heads, head_dim, max_seq_len, split_chunk):
    """fp32 views (partial_o [B,Hq,C,D], partial_lse [B,Hq,C]) of a workspace."""
    o_off, l_off, C = k16v8_decode_workspace_layout(batch, num_qo_heads, head_dim,
                                                    max_seq_len, split_chunk)
    n = batch * num_qo_heads * C
    po = workspace[o_off:o_off + n * head_dim * 4].view(torch.float32)
    pl = workspace[l_off:l_off + n * 4].view(torch.float32)
    return po.view(batch, num_qo_heads, C, head_dim), pl.view(batch, num_qo_heads, C)


def k16v8_paged_decode_split(q, k_cache, v_cache, v_scale, block_table, seq_lens, max_seq_len,
                             sm_scale, split_chunk, workspace, dev_error=None, stream=None):
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_split(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), int(max_seq_len), B, hq, k_cache.shape[1], d,
        k_cache.shape[0], float(sm_scale), int(split_chunk), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_decode_split", st)


def k16v8_paged_decode_split_wait_test(q, k_cache, v_cache, v_scale, block_table, seq_lens,
                                       max_seq_len, sm_scale, split_chunk, workspace,
                                       dev_error=None, stream=None):
    """Test hook: k16v8_paged_decode_split with one page copy of the first CTA
    withheld, so that CTA's bounded wait expires (K16V8_DEVERR_TIMEOUT)."""
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_split_wait_test(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), int(max_seq_len), B, hq, k_cache.shape[1], d,
        k_cache.shape[0], float(sm_scale), int(split_chunk), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_decode_split_wait_test", st)


def k16v8_merge_states(partial_o, partial_lse, seq_lens, split_chunk, out, lse=None,
                       stream=None):
    B, hq, C, d = partial_o.shape
    st = load_library().k16v8_merge_states(
        _ptr(partial_o), _ptr(partial_lse), B, hq, C, d, _ptr(seq_lens), int(split_chunk),
        _ptr(out), _ptr(lse), _stream(stream))
    _check("k16v8_merge_states", st)


def k16v8_paged_decode_attention(q, k_cache, v_cache, v_scale, block_table, seq_lens,
                                 max_seq_len, sm_scale, split_chunk, workspace, out, lse=None,
                                 dev_error=None, stream=None):
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), int(max_seq_len), B, hq, k_cache.shape[1], d,
        k_cache.shape[0], float(sm_scale), int(split_chunk), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _ptr(dev_error),
        _stream(stream))
    _check("k16v8_paged_decode_attention", st)


def k16v8_paged_decode_append_split(q, k_new, v_new, k_cache, v_cache, v_scale, block_table,
                                    seq_lens, max_seq_len, sm_scale, split_chunk, workspace,
                                    dev_error=None, stream=None):
    """Decode split with each sequence's new token (k_new / v_new fp16
    [B, Hkv, D]) written at position seq_lens[b] - 1 by the same kernel."""
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_append_split(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), int(max_seq_len), B, hq,
        k_cache.shape[1], d, k_cache.shape[0], float(sm_scale), int(split_chunk),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_error),
        _stream(stream))
    _check("k16v8_paged_decode_append_split", st)


def k16v8_paged_decode_append_attention(q, k_new, v_new, k_cache, v_cache, v_scale, block_table,
                                        seq_lens, max_seq_len, sm_scale, split_chunk, workspace,
                                        out, lse=None, dev_error=None, stream=None):
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_append_attention(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), int(max_seq_len), B, hq,
        k_cache.shape[1], d, k_cache.shape[0], float(sm_scale), int(split_chunk),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
        _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_decode_append_attention", st)


def k16v8_kv_append_v16(k, v, slot_mapping, k_cache, v_cache16, dev_error=None, stream=None):
    """FP16-KV control cache write (values copied as fp16)."""
    T, hkv, d = k.shape
    st = load_library().k16v8_kv_append_v16(
        _ptr(k), _row_stride(k, "k"), _ptr(v), _row_stride(v, "v"), _ptr(slot_mapping), T,
        _ptr(k_cache), _ptr(v_cache16), k_cache.shape[0], hkv, d, _ptr(dev_error),
        _stream(stream))
    _check("k16v8_kv_append_v16", st)


def k16v8_paged_decode_split_v16(q, k_cache, v_cache16, block_table, seq_lens, max_seq_len,
                                 sm_scale, split_chunk, workspace, dev_error=None, stream=None):
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_split_v16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache16), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), int(max_seq_len), B, hq, k_cache.shape[1], d, k_cache.shape[0],
        float(sm_scale), int(split_chunk), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_decode_split_v16", st)


def k16v8_paged_decode_attention_v16(q, k_cache, v_cache16, block_table, seq_lens, max_seq_len,
                                     sm_scale, split_chunk, workspace, out, lse=None,
                                     dev_error=None, stream=None):
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_attention_v16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache16), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), int(max_seq_len), B, hq, k_cache.shape[1], d, k_cache.shape[0],
        float(sm_scale), int(split_chunk), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _ptr(dev_error),
        _stream(stream))
    _check("k16v8_paged_decode_attention_v16", st)


def k16v8_paged_prefill_attention(q, qo_indptr, max_qlen, k_cache, v_cache, v_scale,
                                  block_table, seq_lens, sm_scale, out, lse=None, dev_error=None,
                                  stream=None):
    """Causal attention of q [total_q, Hq, D] (ragged by qo_indptr [B+1])
    against the paged cache, whose seq_lens include these new tokens."""
    total_q, hq, d = q.shape
    st = load_library().k16v8_paged_prefill_attention(
        _ptr(q), _ptr(qo_indptr), total_q, int(max_qlen), _ptr(k_cache), _ptr(v_cache),
        _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        seq_lens.shape[0], hq, k_cache.shape[1], d, k_cache.shape[0], float(sm_scale), _ptr(out),
        _ptr(lse), _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_prefill_attention", st)


def k16v8_paged_prefill_attention_wait_test(q, qo_indptr, max_qlen, k_cache, v_cache, v_scale,
                                            block_table, seq_lens, sm_scale, out, lse=None,
                                            dev_error=None, stream=None):
    """Test hook: k16v8_paged_prefill_attention with the first KV tile of the
    first CTA withheld, so that CTA's bounded wait expires
    (K16V8_DEVERR_TIMEOUT)."""
    total_q, hq, d = q.shape
    st = load_library().k16v8_paged_prefill_attention_wait_test(
        _ptr(q), _ptr(qo_indptr), total_q, int(max_qlen), _ptr(k_cache), _ptr(v_cache),
        _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        seq_lens.shape[0], hq, k_cache.shape[1], d, k_cache.shape[0], float(sm_scale), _ptr(out),
        _ptr(lse), _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_prefill_attention_wait_test", st)


def k16v8_prefill_workspace_size(max_qlen, batch, num_qo_heads, num_kv_heads, head_dim,
                                 kv_splits=0, max_seq_len=0) -> int:
    """Bytes of workspace k16v8_paged_prefill_attention_split needs (0: the
    call will not split, no workspace needed)."""
    return int(load_library().k16v8_prefill_workspace_size(max_qlen, batch, num_qo_heads,
                                                            num_kv_heads, head_dim, kv_splits,
                                                            max_seq_len))


def k16v8_paged_prefill_attention_split(q, qo_indptr, max_qlen, k_cache, v_cache, v_scale,
                                        block_table, seq_lens, sm_scale, workspace, out,
                                        lse=None, dev_error=None, stream=None, kv_splits=0,
                                        max_seq_len=0):
    """Prefill attention with the KV range of each query-tile pair cut into
    up to 4 parts (merged in the kernel) when the call has too few pairs to
    fill the GPU; `workspace` zero-filled before its first use."""
    total_q, hq, d = q.shape
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().k16v8_paged_prefill_attention_split(
        _ptr(q), _ptr(qo_indptr), total_q, int(max_qlen), _ptr(k_cache), _ptr(v_cache),
        _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        seq_lens.shape[0], hq, k_cache.shape[1], d, k_cache.shape[0], float(sm_scale),
        int(kv_splits), int(max_seq_len), _ptr(workspace), nbytes, _ptr(out), _ptr(lse),
        _ptr(dev_error),
        _stream(stream))
    _check("k16v8_paged_prefill_attention_split", st)


def k16v8_paged_decode_attention_static(q, k_cache, v_cache, v_scale, block_table, seq_lens,
                                        max_seq_len, sm_scale, split_chunk, out, lse=None,
                                        dev_error=None, stream=None):
    """Decode attention with the partials in the library's built-in device
    scratch: for callers that cannot allocate device memory.  Calls that
    overlap on the GPU race on that scratch; the first call on a device
    should come before any stream capture."""
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_attention_static(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), int(max_seq_len), B, hq, k_cache.shape[1], d,
        k_cache.shape[0], float(sm_scale), int(split_chunk), _ptr(out), _ptr(lse),
        _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_decode_attention_static", st)


def k16v8_decode_balanced_workspace_size(batch, num_qo_heads, head_dim) -> int:
    """Bytes of workspace k16v8_paged_decode_attention_balanced needs on the
    current device (0 for an unsupported shape)."""
    return int(load_library().k16v8_decode_balanced_workspace_size(batch, num_qo_heads, head_dim))


def k16v8_paged_decode_attention_balanced(q, k_cache, v_cache, v_scale, block_table, seq_lens,
                                          sm_scale, workspace, out, lse=None, dev_error=None,
                                          stream=None, flags=0):
    """Decode attention with every CTA given the same number of KV tiles."""
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_attention_balanced(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, hq, k_cache.shape[1], d, k_cache.shape[0],
        float(sm_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out), _ptr(lse), int(flags), _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_decode_attention_balanced", st)


def k16v8_paged_decode_balanced_split(q, k_cache, v_cache, v_scale, block_table, seq_lens,
                                      sm_scale, workspace, out, lse=None, dev_error=None,
                                      stream=None, flags=0):
    B, hq, d = q.shape
    st = load_library().k16v8_paged_decode_balanced_split(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, hq, k_cache.shape[1], d, k_cache.shape[0],
        float(sm_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out), _ptr(lse), int(flags), _ptr(dev_error), _stream(stream))
    _check("k16v8_paged_decode_balanced_split", st)


def k16v8_merge_balanced(workspace, num_kv_heads, out, lse=None, stream=None):
    B, hq, d = out.shape
    st = load_library().k16v8_merge_balanced(
        _ptr(workspace), workspace.numel() * workspace.element_size(), B, hq, int(num_kv_heads),
        d, _ptr(out), _ptr(lse), _stream(stream))
    _check("k16v8_merge_balanced", st)


def _append_balanced(name, q, k_new, v_new, k_cache, v_cache, v_scale, block_table, seq_lens,
                     sm_scale, workspace, out, lse, dev_error, stream, flags):
    B, hq, d = q.shape
    st = getattr(load_library(), name)(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, hq, k_cache.shape[1], d,
        k_cache.shape[0], float(sm_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), int(flags),
        _ptr(dev_error), _stream(stream))
    _check(name, st)


def k16v8_paged_decode_append_balanced_split(q, k_new, v_new, k_cache, v_cache, v_scale,
                                             block_table, seq_lens, sm_scale, workspace, out,
                                             lse=None, dev_error=None, stream=None, flags=0):
    """Load-balanced decode split with each sequence's new token (k_new,
    v_new [B, Hkv, D] fp16) written into the cache by the same kernel."""
    _append_balanced("k16v8_paged_decode_append_balanced_split", q, k_new, v_new, k_cache,
                     v_cache, v_scale, block_table, seq_lens, sm_scale, workspace, out, lse,
                     dev_error, stream, flags)


def k16v8_paged_decode_append_attention_balanced(q, k_new, v_new, k_cache, v_cache, v_scale,
                                                 block_table, seq_lens, sm_scale, workspace, out,
                                                 lse=None, dev_error=None, stream=None, flags=0):
    """k16v8_paged_decode_append_balanced_split followed by the merge."""
    _append_balanced("k16v8_paged_decode_append_attention_balanced", q, k_new, v_new, k_cache,
                     v_cache, v_scale, block_table, seq_lens, sm_scale, workspace, out, lse,
                     dev_error, stream, flags)


def k16v8_read_device_error(dev_error, stream=None) -> int:
    """Synchronise the stream and return the device error word."""
    v = _i32()
    st = load_library().k16v8_read_device_error(_ptr(dev_error), _stream(stream),
                                                ctypes.byref(v))
    if st not in (K16V8_OK, K16V8_ERR_DEVICE_BOUNDS):
        _check("k16v8_read_device_error", st)
    return int(v.value)
