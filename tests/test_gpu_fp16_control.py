"""FP16-KV control (values stored as fp16, the native format the subject
page compares against) on the same decode kernels, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import check_close, dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from fp8_paged_kv_append_gb300 import k16v8
    k16v8.load_library()
    return k16v8


@pytest.mark.parametrize("maker,chunk", [(workloads.tiny_decode, 64),
                                         (workloads.decode_1k_b32, 384),
                                         (workloads.decode_8k_b16, 512)])
def test_fp16_control_cache_and_decode(K, maker, chunk):
    w = maker()
    v16 = w.v_tok.astype(np.float16)
    P, hkv, d = w.num_pages, w.num_kv_heads, w.head_dim
    poison = int(np.uint16(0x7E00).view(np.int16))
    kc = torch.full((P, hkv, 16, d), poison, dtype=torch.int16, device=dev()).view(torch.float16)
    vc = torch.full((P, hkv, 16, d), poison, dtype=torch.int16, device=dev()).view(torch.float16)
    K.k16v8_kv_append_v16(to_dev(w.k_tok), to_dev(v16), to_dev(w.slot_mapping), kc, vc)
    okc = np.full((P, hkv, 16, d), 0x7E00, np.uint16).view(np.float16)
    ovc = np.full((P, hkv, 16, d), 0x7E00, np.uint16).view(np.float16)
    oracle.kv_append_v16(w.k_tok, v16, w.slot_mapping, okc, ovc)
    assert np.array_equal(kc.view(torch.int16).cpu().numpy().view(np.uint16), okc.view(np.uint16))
    assert np.array_equal(vc.view(torch.int16).cpu().numpy().view(np.uint16), ovc.view(np.uint16))
    B, hq, _ = w.q.shape
    L = int(w.seq_lens.max())
    ws = torch.empty(K.k16v8_decode_workspace_size(B, hq, d, L, chunk), dtype=torch.uint8,
                     device=dev())
    out = torch.empty((B, hq, d), dtype=torch.float16, device=dev())
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    K.k16v8_paged_decode_attention_v16(to_dev(w.q), kc, vc, to_dev(w.block_table),
                                       to_dev(w.seq_lens), L, w.sm_scale, chunk, ws, out, lse, err)
    assert K.k16v8_read_device_error(err) == 0
    ro, rl = oracle.paged_decode_v16(w.q, okc, ovc, w.block_table, w.seq_lens, w.sm_scale)
    check_close(out.float().cpu().numpy(), ro, lse.cpu().numpy(), rl)
