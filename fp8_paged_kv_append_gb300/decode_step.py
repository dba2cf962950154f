"""A whole-model decode step: kv_append + split-KV attention + LSE merge for
every layer, replayed as one CUDA graph.

The per-layer pools, scales and workspaces stay resident; a step takes each
layer's new-token K/V and query and writes each layer's attention output.
The value scales are checked on the host before the graph is captured (the
subject page's production checks verify calibrated scales inside the engine
before graph capture: "Phi-4: quality transfer and interrupted throughput
studies", intro).  All computation runs in libk16v8's kernels; this module
only sequences the calls and owns the graph.
"""
from __future__ import annotations

import math

import torch

from . import k16v8 as K


class ScaleError(ValueError):
    pass


def validate_scales(v_scales) -> None:
    """Every per-(layer, KV head) value scale must be finite and > 0."""
    for li, s in enumerate(v_scales):
        host = s.detach().float().cpu()
        bad = ~(torch.isfinite(host) & (host > 0))
        if bool(bad.any()):
            idx = bad.nonzero().flatten().tolist()
            raise ScaleError(f"layer {li}: value scale not finite and positive at KV heads {idx}")


# Tiles per CTA of the load-balanced split (one full wave of SMs x 4 CTAs)
# above which the chunked split takes over.  Measured on GB300 (per
# layer-step, append folded in): 37 tiles per CTA (decode 1K/b32) balanced
# 26.1 us against chunked 29.1 us; 136 (8K/b16) 80.7 against 81.6 us; 225
# (64 ragged sequences over a 32 GiB pool) 138.5 against 126.3 us.  The
# balanced split removes the chunked split's partial last wave, which costs
# most when there are few waves; with long ranges per CTA the CTAs of one SM
# drift apart and the chunked split's many short CTAs even out better.
BALANCED_MAX_TILES_PER_CTA = 160


def choose_schedule(seq_lens_host, num_kv_heads: int, num_sms: int) -> str:
    """"balanced_fused" or "fused" (both with the append folded in) for a
    batch with these lengths, by the rule above."""
    pages = sum((int(L) + 15) // 16 for L in seq_lens_host if int(L) > 0)
    tiles = pages * int(num_kv_heads)
    per_cta = -(-tiles // (int(num_sms) * 4)) if tiles else 0
    return "balanced_fused" if per_cta <= BALANCED_MAX_TILES_PER_CTA else "fused"


class MultiLayerDecode:
    """Decode step over `len(k_caches)` layers that share one page table.

    k_caches[l] fp16 [P,Hkv,16,D], v_caches[l] uint8 [P,Hkv,16,D], v_scales[l]
    fp32 [Hkv]; block_table int32 [B, max_pages]; seq_lens int32 [B] (the
    lengths after this step's append); slots int64 [B] (where the new token
    of each sequence goes).

    schedule "chunked": split-KV with a fixed split_chunk, then the merge;
    "fused": the same with each layer's append done by the split kernel;
    "balanced": the load-balanced split (one full wave of equal tile ranges)
    and its merge; "balanced_fused": the same with each layer's append done
    by the split kernel itself (2 launches per layer instead of 3; the slot
    of the new token is then the one the block table gives for position
    seq_len - 1, which `slots` must agree with); "whole": one CTA per
    (sequence, KV head) over the whole sequence with the append folded in,
    the output written by that kernel (1 launch per layer, no merge; needs
    max_seq_len <= 8192).  The block table and lengths
    are written only by host copies, never by the kernel before the
    attention, so the balanced split may read them ahead of its wait on that
    kernel.  "auto" picks "balanced_fused" or "fused" by choose_schedule
    from the lengths (copied to the host once, at construction)."""

    def __init__(self, k_caches, v_caches, v_scales, block_table, seq_lens, slots, max_seq_len,
                 num_qo_heads, sm_scale=None, split_chunk=512, validate=True,
                 schedule="chunked"):
        if validate:
            validate_scales(v_scales)
        self.k_caches, self.v_caches, self.v_scales = k_caches, v_caches, v_scales
        self.block_table, self.seq_lens, self.slots = block_table, seq_lens, slots
        self.max_seq_len = int(max_seq_len)
        self.layers = len(k_caches)
        dev = k_caches[0].device
        self.batch = int(block_table.shape[0])
        self.hq = int(num_qo_heads)
        self.hkv = int(k_caches[0].shape[1])
        self.d = int(k_caches[0].shape[3])
        self.sm_scale = float(sm_scale if sm_scale is not None else 1.0 / math.sqrt(self.d))
        self.chunk = int(split_chunk)
        if schedule == "auto":  # by the lengths of this batch (read once, here)
            schedule = choose_schedule(seq_lens.detach().cpu().tolist(), k_caches[0].shape[1],
                                       torch.cuda.get_device_properties(dev).multi_processor_count)
        if schedule not in ("chunked", "fused", "balanced", "balanced_fused", "whole"):
            raise ValueError(f"unknown schedule {schedule!r}")
        if schedule == "whole":  # one chunk covering the longest sequence
            self.chunk = max(16, -(-self.max_seq_len // 16) * 16)
            if self.chunk > K.MAX_SPLIT_CHUNK:
                raise ValueError(f"schedule 'whole' needs max_seq_len <= {K.MAX_SPLIT_CHUNK}")
        self.schedule = schedule
        if schedule in ("balanced", "balanced_fused"):
            n = K.k16v8_decode_balanced_workspace_size(self.batch, self.hq, self.d)
        else:
            n = K.k16v8_decode_workspace_size(self.batch, self.hq, self.d, self.max_seq_len,
                                              self.chunk)
        if n == 0:
            raise ValueError("invalid decode workspace shape")
        self.workspace = torch.empty(n, dtype=torch.uint8, device=dev)
        if schedule in ("chunked", "fused"):
            self.partial_o, self.partial_lse = K.workspace_views(
                self.workspace, self.batch, self.hq, self.d, self.max_seq_len, self.chunk)
        self.dev_error = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None

    def layer(self, li, q, k_new, v_new, out, lse=None):
        self.split(li, q, k_new, v_new, out, lse)
        self.merge(li, out, lse)

    def split(self, li, q, k_new, v_new, out, lse=None, append=True):
        """Layer li's launches up to the attention split (the separate append
        first, unless the split kernel does it or append is False)."""
        if self.schedule == "whole":
            K.k16v8_paged_decode_append_attention(
                q, k_new, v_new, self.k_caches[li], self.v_caches[li], self.v_scales[li],
                self.block_table, self.seq_lens, self.max_seq_len, self.sm_scale, self.chunk,
                self.workspace, out, lse, self.dev_error)
        elif self.schedule == "balanced_fused":
            K.k16v8_paged_decode_append_balanced_split(
                q, k_new, v_new, self.k_caches[li], self.v_caches[li], self.v_scales[li],
                self.block_table, self.seq_lens, self.sm_scale, self.workspace, out, lse,
                self.dev_error, flags=K.DECODE_METADATA_READY)
        elif self.schedule == "fused":
            K.k16v8_paged_decode_append_split(
                q, k_new, v_new, self.k_caches[li], self.v_caches[li], self.v_scales[li],
                self.block_table, self.seq_lens, self.max_seq_len, self.sm_scale, self.chunk,
                self.workspace, self.dev_error)
        else:
            if append:
                K.k16v8_kv_append(k_new, v_new, self.slots, self.v_scales[li],
                                  self.k_caches[li], self.v_caches[li], self.dev_error)
            if self.schedule == "balanced":
                K.k16v8_paged_decode_balanced_split(q, self.k_caches[li], self.v_caches[li],
                                                    self.v_scales[li], self.block_table,
                                                    self.seq_lens, self.sm_scale, self.workspace,
                                                    out, lse, self.dev_error,
                                                    flags=K.DECODE_METADATA_READY)
            else:
                K.k16v8_paged_decode_split(q, self.k_caches[li], self.v_caches[li],
                                           self.v_scales[li], self.block_table, self.seq_lens,
                                           self.max_seq_len, self.sm_scale, self.chunk,
                                           self.workspace, self.dev_error)

    def merge(self, li, out, lse=None):
        """Layer li's merge of the split partials into out / lse (none for
        "whole", whose split kernel writes them)."""
        if self.schedule == "whole":
            return
        if self.schedule in ("balanced", "balanced_fused"):
            K.k16v8_merge_balanced(self.workspace, self.hkv, out, lse)
        else:
            K.k16v8_merge_states(self.partial_o, self.partial_lse, self.seq_lens, self.chunk,
                                 out, lse)

    def launches_per_layer(self) -> int:
        """Launches per layer: 2 when the append runs inside the split, 1 when
        the split also writes the output."""
        if self.schedule == "whole":
            return 1
        return 2 if self.schedule in ("fused", "balanced_fused") else 3

    def step(self, qs, k_news, v_news, outs, lses=None):
        for li in range(self.layers):
            self.layer(li, qs[li], k_news[li], v_news[li], outs[li],
                       None if lses is None else lses[li])

    def capture(self, qs, k_news, v_news, outs, lses=None):
        """Capture one whole step into a CUDA graph over these buffers (the
        caller refills qs / k_news / v_news in place between replays)."""
        self.step(qs, k_news, v_news, outs, lses)  # eager run configures the kernels
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream(), capture_error_mode="thread_local"):
            self.step(qs, k_news, v_news, outs, lses)
        self.graph = g
        return g

    def replay(self):
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()

    def check(self) -> int:
        """Synchronise and return the device error word (0 = clean)."""
        return K.k16v8_read_device_error(self.dev_error)
