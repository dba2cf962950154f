"""Seeded synthetic inputs for the K16/V8 paged-attention path.

This module only draws inputs: random queries, keys and values with the
shapes and distributions of the Phi-4-shaped workloads, page tables and slot
mappings, and the per-KV-head value scales a calibration pass would supply.
It holds none of the path's arithmetic (no quantisation, no attention), so
both the CUDA path and the oracle can be fed from it.

Geometry from "Phi-4: quality transfer and interrupted throughput studies"
(intro): 40 query heads, 10 KV heads, head dimension 128, 40 layers, a 32 GiB
KV budget.  Pages hold 16 tokens.  The value scale of a KV head is the
calibration amax / 448 computed in fp32 (448 = largest finite E4M3FN value),
1.0 for an all-zero head.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE_SIZE = 16
E4M3_MAX = 448.0

PHI4_Q_HEADS = 40
PHI4_KV_HEADS = 10
PHI4_HEAD_DIM = 128
PHI4_LAYERS = 40
KV_BUDGET_BYTES = 32 * 2**30


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def default_sm_scale(head_dim: int) -> float:
    """1/sqrt(head_dim) held as the fp32 value the kernels receive."""
    return float(np.float32(1.0 / math.sqrt(head_dim)))


def calibrate_v_scale(v: np.ndarray) -> np.ndarray:
    """Per-KV-head fp32 scale amax/448 over values v [..., Hkv, D]."""
    hk = v.shape[-2]
    a = np.abs(v.reshape(-1, hk, v.shape[-1]).astype(np.float32)).max(axis=(0, 2))
    s = (a.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
    s[a == 0] = np.float32(1.0)
    return s


@dataclass
class DecodeInputs:
    """One decode layer-step: a paged cache described by token arrays.

    k_tok / v_tok hold every cached token of every sequence (sequence-major,
    position order); slot_mapping places token r at slot
    block_table[b, pos // 16] * 16 + pos % 16.  new_rows indexes the last
    token of each sequence, the one a decode step appends."""
    name: str
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    num_pages: int
    seq_lens: np.ndarray
    block_table: np.ndarray
    q: np.ndarray
    k_tok: np.ndarray
    v_tok: np.ndarray
    slot_mapping: np.ndarray
    v_scale: np.ndarray
    sm_scale: float
    new_rows: np.ndarray
    page_size: int = PAGE_SIZE
    notes: dict = field(default_factory=dict)

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())


def _slots_for(seq_lens, block_table, page_size):
    rows = []
    for b, L in enumerate(seq_lens.tolist()):
        pos = np.arange(L, dtype=np.int64)
        rows.append(block_table[b, pos // page_size].astype(np.int64) * page_size
                    + pos % page_size)
    return np.concatenate(rows) if rows else np.zeros(0, np.int64)


def assign_pages(rng, seq_lens, num_pages=None, page_size=PAGE_SIZE):
    """Distinct pages for every sequence, drawn from a seeded permutation of
    a pool of num_pages pages (default: exactly the pages needed)."""
    need = [-(-int(L) // page_size) for L in seq_lens]
    total = sum(need)
    if num_pages is None:
        num_pages = max(total, 1)
    if total > num_pages:
        raise ValueError(f"{total} pages needed, pool has {num_pages}")
    perm = rng.permutation(num_pages).astype(np.int32)
    width = max(max(need, default=1), 1)
    bt = np.full((len(seq_lens), width), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    return bt, num_pages


def make_decode(name, seed, seq_lens, num_qo_heads=PHI4_Q_HEADS,
                num_kv_heads=PHI4_KV_HEADS, head_dim=PHI4_HEAD_DIM,
                num_pages=None, v_dtype=np.float16, k_boost_heads=(),
                k_boost=4.0, page_size=PAGE_SIZE) -> DecodeInputs:
    rng = rng_for(seed)
    seq_lens = np.asarray(seq_lens, np.int32)
    B = len(seq_lens)
    bt, num_pages = assign_pages(rng, seq_lens, num_pages, page_size)
    N = int(seq_lens.astype(np.int64).sum())
    q = rng.standard_normal((B, num_qo_heads, head_dim), dtype=np.float32)
    k = rng.standard_normal((N, num_kv_heads, head_dim), dtype=np.float32)
    for h in k_boost_heads:
        k[:, h, :] *= np.float32(k_boost)
    v = rng.standard_normal((N, num_kv_heads, head_dim), dtype=np.float32)
    q = q.astype(np.float16)
    k = k.astype(np.float16)
    v = v.astype(v_dtype)
    ends = np.cumsum(seq_lens.astype(np.int64))
    return DecodeInputs(
        name=name, batch=B, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, num_pages=num_pages, seq_lens=seq_lens, block_table=bt,
        q=q, k_tok=k, v_tok=v, slot_mapping=_slots_for(seq_lens, bt, page_size),
        v_scale=calibrate_v_scale(v), sm_scale=default_sm_scale(head_dim),
        new_rows=np.where(seq_lens > 0, ends - 1, -1).astype(np.int64),
        page_size=page_size)


def tiny_decode(seed: int = 0) -> DecodeInputs:
    """Single-layer decode: batch 2, 8 q heads / 2 KV heads, d 128,
    seq_lens {37, 200}, pages drawn from a permuted 32-page pool, fp32 V."""
    return make_decode("tiny: B=2 Hq=8 Hkv=2 L={37,200}", seed, [37, 200],
                       num_qo_heads=8, num_kv_heads=2, num_pages=32,
                       v_dtype=np.float32)


def decode_lens(seed: int, batch: int, base: int, extra: int = 128) -> np.ndarray:
    """base + uniform[0, extra) cached tokens per sequence (the prompt plus
    the already generated part of 128 forced output tokens)."""
    return (base + rng_for(seed ^ 0x5EED).integers(0, extra, batch)).astype(np.int32)


def decode_1k_b32(seed: int = 1) -> DecodeInputs:
    """Phi-4-shaped decode at 1K / batch 32 (one layer)."""
    return make_decode("decode 1K/b32: Hq=40 Hkv=10 d=128 L=1024+U[0,128)", seed,
                       decode_lens(seed, 32, 1024))


def decode_8k_b16(seed: int = 2) -> DecodeInputs:
    """Phi-4-shaped decode at 8K / batch 16; keys of the even KV heads are
    drawn x4 to stretch the softmax range."""
    return make_decode("decode 8K/b16: Hq=40 Hkv=10 d=128 L=8192+U[0,128), K x4 on even heads",
                       seed, decode_lens(seed, 16, 8192), k_boost_heads=(0, 2, 4, 6, 8))


# ---- full-pool ragged decode across 40 layers -----------------------------

def pool_pages_per_layer(budget=KV_BUDGET_BYTES, layers=PHI4_LAYERS,
                         kv_heads=PHI4_KV_HEADS, head_dim=PHI4_HEAD_DIM,
                         k_bytes=2, v_bytes=1, page_size=PAGE_SIZE) -> int:
    """Whole pages of one layer's share of the budget (input sizing only)."""
    per_tok = kv_heads * head_dim * (k_bytes + v_bytes)
    return int((budget // layers) // (per_tok * page_size))


def fullpool_lens(seed: int = 4, batch: int = 64, max_len: int = 8192,
                  pool_pages: int | None = None, page_size: int = PAGE_SIZE):
    """seq_lens ~ U[1, max_len], redrawn as a whole until the batch fits the
    pool; returns (seq_lens, draws)."""
    if pool_pages is None:
        pool_pages = pool_pages_per_layer()
    rng = rng_for(seed)
    draws = 0
    while True:
        draws += 1
        L = rng.integers(1, max_len + 1, batch).astype(np.int32)
        if int(np.sum(-(-L.astype(np.int64) // page_size))) <= pool_pages:
            return L, draws


@dataclass
class FullPoolLayout:
    seq_lens: np.ndarray
    block_table: np.ndarray
    num_pages: int
    draws: int


def fullpool_layout(seed: int = 4, batch: int = 64) -> FullPoolLayout:
    P = pool_pages_per_layer()
    L, draws = fullpool_lens(seed, batch, pool_pages=P)
    bt, _ = assign_pages(rng_for(seed + 1), L, P)
    return FullPoolLayout(L, bt, P, draws)


def device_layer_pool(layer_seed: int, num_pages: int, device, kv_heads=PHI4_KV_HEADS,
                      head_dim=PHI4_HEAD_DIM, page_size=PAGE_SIZE):
    """One layer's cache drawn directly on a torch device: K fp16 ~ N(0,1);
    V ~ N(0,1) calibrated per head (amax/448) and cast to float8_e4m3fn by
    torch's own conversion.  Returns (k_cache, v_cache uint8, v_scale fp32)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(layer_seed)
    shape = (num_pages, kv_heads, page_size, head_dim)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    amax = v.abs().amax(dim=(0, 2, 3)).float()
    scale = (amax / E4M3_MAX).to(torch.float32)
    scale = torch.where(amax == 0, torch.ones_like(scale), scale)
    codes = torch.empty(shape, dtype=torch.uint8, device=device)
    for h in range(kv_heads):
        codes[:, h] = (v[:, h].float() / scale[h]).to(torch.float8_e4m3fn).view(torch.uint8)
    del v
    return k, codes, scale


# ---- chunked causal prefill ------------------------------------------------

@dataclass
class PrefillCall:
    """One prefill launch: new tokens of several sequences (ragged)."""
    seqs: np.ndarray        # sequence ids in this call
    starts: np.ndarray      # first new position per sequence
    qlens: np.ndarray       # new tokens per sequence
    qo_indptr: np.ndarray   # int32 [n+1]
    seq_lens: np.ndarray    # int32 [n] cached length after the append
    block_table: np.ndarray  # int32 [n, max_pages] rows of the sequences
    rows: np.ndarray        # int64 [total_q] token rows into PrefillInputs arrays


@dataclass
class PrefillInputs:
    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    num_pages: int
    prompt_lens: np.ndarray
    block_table: np.ndarray
    q: np.ndarray       # fp16 [N, Hq, D] all prompt tokens, sequence-major
    k_tok: np.ndarray   # fp16 [N, Hkv, D]
    v_tok: np.ndarray   # fp16 [N, Hkv, D]
    slot_mapping: np.ndarray  # int64 [N]
    v_scale: np.ndarray
    sm_scale: float
    chunk: int
    calls: list
    page_size: int = PAGE_SIZE


def make_prefill(name, seed, prompt_lens, chunk=1024, num_qo_heads=PHI4_Q_HEADS,
                 num_kv_heads=PHI4_KV_HEADS, head_dim=PHI4_HEAD_DIM,
                 page_size=PAGE_SIZE, num_pages=None) -> PrefillInputs:
    """Prompts split into chunks of at most `chunk` new tokens per sequence;
    call j carries chunk j of every prompt that still has one."""
    rng = rng_for(seed)
    lens = np.asarray(prompt_lens, np.int32)
    bt, num_pages = assign_pages(rng, lens, num_pages, page_size)
    N = int(lens.astype(np.int64).sum())
    q = rng.standard_normal((N, num_qo_heads, head_dim), dtype=np.float32).astype(np.float16)
    k = rng.standard_normal((N, num_kv_heads, head_dim), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((N, num_kv_heads, head_dim), dtype=np.float32).astype(np.float16)
    offs = np.concatenate([[0], np.cumsum(lens.astype(np.int64))])
    calls = []
    n_calls = max(-(-int(L) // chunk) for L in lens) if len(lens) else 0
    for j in range(n_calls):
        seqs, starts, qlens = [], [], []
        for b, L in enumerate(lens.tolist()):
            s = j * chunk
            if s < L:
                seqs.append(b)
                starts.append(s)
                qlens.append(min(chunk, L - s))
        seqs = np.asarray(seqs, np.int64)
        starts = np.asarray(starts, np.int64)
        qlens = np.asarray(qlens, np.int64)
        indptr = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
        rows = np.concatenate([offs[b] + s + np.arange(n, dtype=np.int64)
                               for b, s, n in zip(seqs, starts, qlens)])
        calls.append(PrefillCall(seqs=seqs, starts=starts, qlens=qlens,
                                 qo_indptr=indptr,
                                 seq_lens=(starts + qlens).astype(np.int32),
                                 block_table=np.ascontiguousarray(bt[seqs]), rows=rows))
    return PrefillInputs(name=name, num_qo_heads=num_qo_heads,
                         num_kv_heads=num_kv_heads, head_dim=head_dim,
                         num_pages=num_pages, prompt_lens=lens, block_table=bt,
                         q=q, k_tok=k, v_tok=v,
                         slot_mapping=_slots_for(lens, bt, page_size),
                         v_scale=calibrate_v_scale(v),
                         sm_scale=default_sm_scale(head_dim), chunk=chunk,
                         calls=calls, page_size=page_size)


def prefill_8x1k(seed: int = 5) -> PrefillInputs:
    return make_prefill("prefill 8x1024 prompts, one chunk each", seed, [1024] * 8)


def prefill_1x8k(seed: int = 6) -> PrefillInputs:
    return make_prefill("prefill 1x8192 prompt in 8 chunks of 1024", seed, [8192])
