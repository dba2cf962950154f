#!/usr/bin/env python3
"""K16/V8 paged decode benchmark (one JSON line on stdout).

The headline is a whole decode step through the 40 layers of the full KV
pool: per layer a pool of 223,696 token slots (FP16 K + E4M3 V, 32 GiB over
all layers), batch 64 with ragged lengths in [1, 8192], the Phi-4 geometry
(40 query / 10 KV heads, d 128, 16-token pages).  Per layer the step appends
each sequence's new token, runs paged decode attention split over the KV
sequence and merges the partials (the automatic schedule folds the append
into the split kernel: 2 launches per layer); the 40 layers are one CUDA
graph.  `value` is KV GB/s (3,840 B per cached token per layer), with
`us_per_layer_step` beside it; `roofline` is the attention split kernel's;
`e2e` runs the same step from pinned host buffers; `cpu_baseline` is the
oracle on a bounded host sample of the same workload.  Extra lines: decode
1K/batch 32, prefill with its cache write, the FP16-KV control, and decode
8K/batch 16 (last).  `--workload 1k|8k` puts a one-layer workload on the main
line instead; `--workload prefill` prints prefill alone.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the
workload (the path has no exchange step); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "K16/V8 paged decode attention: KV GB/s vs HBM peak; µs per layer-step"
L2_BYTES = 129 * 10 ** 6


# ---- multi-process plumbing (replicas only) ---------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(local_ms: float, local_units: float, group=None):
    """Max step time and summed units over ranks (plain values at N = 1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_ms, local_units
    backend = dist.get_backend(group)
    devc = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=devc)
    u = torch.tensor([local_units], dtype=torch.float64, device=devc)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---- environment records ----------------------------------------------------------

def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms while running; start()
    returns once the first sample is in, so the samples cover the timed
    region that follows."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 5.0 and self.proc.poll() is None:
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.02)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)  # one more sample period
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v
                          and "Not" not in v})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


MODES = ("chunked", "fused", "balanced", "balanced_fused", "whole")
DEFAULT_DECODE = "balanced_fused"  # schedule of a one-layer decode line
SUFFIX = {"chunked": "chunked", "fused": "fused_append", "balanced": "balanced",
          "balanced_fused": "balanced_fused_append", "whole": "whole_sequence"}

_DECODE_SRC = ["decode.cu", "decode_page.cuh", "k16v8_device.cuh"]
_BALANCED_SRC = ["decode_balanced.cu", "decode_page.cuh", "k16v8_device.cuh"]
# (workload, schedule) -> committed ncu summary of its attention kernel and
# the sources that kernel is built from
KERNEL_PROFILES = {
    ("1k", "chunked"): ("decode_split_1k_b32.md", _DECODE_SRC),
    ("1k", "balanced"): ("decode_balanced_1k_b32.md", _BALANCED_SRC),
    ("1k", "balanced_fused"): ("decode_balanced_append_1k_b32.md", _BALANCED_SRC),
    ("8k", "chunked"): ("decode_split_8k_b16.md", _DECODE_SRC),
    ("8k", "balanced_fused"): ("decode_balanced_append_8k_b16.md", _BALANCED_SRC),
    ("fullpool", "fused"): ("decode_split_append_fullpool_layer.md", _DECODE_SRC),
    ("prefill_8x1024", "kv_append"): ("kv_append_8x1024.md", ["kv_append.cu", "k16v8_device.cuh"]),
}


def sources_sha256(names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "fp8_paged_kv_append_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_from_profiles(workload: str, mode: str):
    """DRAM bytes per launch of the attention kernel of (workload, mode) from
    the committed ncu summary, or None when there is none or its sources
    changed since that capture."""
    if (workload, mode) not in KERNEL_PROFILES:
        return None
    prof, srcs = KERNEL_PROFILES[(workload, mode)]
    path = os.path.join(ROOT, "profiles", prof)
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_src = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    m_tr = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", txt)
    if not m_src or not m_tr:
        return None
    return float(m_tr.group(1)) if sources_sha256(srcs) == m_src.group(1) else None


# ---- the decode workload on the GPU ---------------------------------------------

def kv_bytes(w) -> int:
    return int(w.seq_lens.astype(np.int64).sum()) * w.num_kv_heads * w.head_dim * 3


def replicas_for(w) -> int:
    """Pool copies rotated between steps so that every step reads HBM (>= 4x L2)."""
    pool_bytes = w.num_pages * w.num_kv_heads * 16 * w.head_dim * 3
    return max(1, -(-4 * L2_BYTES // pool_bytes))


class DecodeBench:
    """Device state for timed decode steps over `replicas` copies of the pool."""

    def __init__(self, w, device, split_chunk=512, replicas=None, mode="chunked"):
        """mode: "chunked" (append, split, merge), "fused" (append fused into
        the split kernel, merge), "balanced" (append, load-balanced split,
        its merge), "balanced_fused" (append fused into the load-balanced
        split, its merge) or "whole" (one CTA per (sequence, KV head) over the
        whole sequence, append folded in, the output written by that kernel:
        one launch)."""
        import torch
        from fp8_paged_kv_append_gb300 import k16v8 as K
        assert mode in MODES
        self.K, self.torch, self.w, self.dev = K, torch, w, device
        self.chunk = split_chunk
        self.mode = mode
        self.fused = mode in ("fused", "balanced_fused", "whole")
        self.balanced = mode in ("balanced", "balanced_fused")
        self.R = replicas or replicas_for(w)
        P = w.num_pages
        self.P = P
        B, hq, d = w.q.shape
        td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.kc = torch.empty((self.R * P, w.num_kv_heads, 16, d), dtype=torch.float16,
                              device=device)
        self.vc = torch.empty((self.R * P, w.num_kv_heads, 16, d), dtype=torch.uint8,
                              device=device)
        self.v_scale = td(w.v_scale)
        k_all, v_all = td(w.k_tok), td(w.v_tok)
        self.bt, self.slots_new = [], []
        for r in range(self.R):
            K.k16v8_kv_append(k_all, v_all, td(w.slot_mapping + r * P * 16), self.v_scale,
                              self.kc, self.vc)
            self.bt.append(td(w.block_table + r * P))
            self.slots_new.append(td(w.slot_mapping[w.new_rows] + r * P * 16))
        del k_all, v_all
        self.k_new = td(w.k_tok[w.new_rows])
        self.v_new = td(w.v_tok[w.new_rows])
        self.k_new16 = self.k_new.contiguous()
        self.v_new16 = self.v_new.to(torch.float16).contiguous()
        self.q = td(w.q)
        self.seq_lens = td(w.seq_lens)
        self.max_len = int(w.seq_lens.max())
        if mode == "whole":  # one chunk covering the longest sequence
            self.chunk = max(16, -(-self.max_len // 16) * 16)
        if self.balanced:
            self.ws = torch.empty(K.k16v8_decode_balanced_workspace_size(B, hq, d),
                                  dtype=torch.uint8, device=device)
        else:
            self.ws = torch.empty(K.k16v8_decode_workspace_size(B, hq, d, self.max_len,
                                                                self.chunk),
                                  dtype=torch.uint8, device=device)
            self.po, self.pl = K.workspace_views(self.ws, B, hq, d, self.max_len, self.chunk)
        self.out = torch.empty((B, hq, d), dtype=torch.float16, device=device)
        self.lse = torch.empty((B, hq), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize(device)

    def step(self, i, ev=None):
        K, r = self.K, i % self.R
        if ev:
            ev[0].record()
        if not self.fused:
            K.k16v8_kv_append(self.k_new, self.v_new, self.slots_new[r], self.v_scale, self.kc,
                              self.vc, self.err)
        if ev:
            ev[1].record()
        self.split(i)
        if ev:
            ev[2].record()
        self.merge()
        if ev:
            ev[3].record()

    def split(self, i):
        K, r = self.K, i % self.R
        if self.mode == "whole":
            K.k16v8_paged_decode_append_attention(
                self.q, self.k_new16, self.v_new16, self.kc, self.vc, self.v_scale, self.bt[r],
                self.seq_lens, self.max_len, self.w.sm_scale, self.chunk, self.ws, self.out,
                self.lse, self.err)
        elif self.mode == "fused":
            K.k16v8_paged_decode_append_split(self.q, self.k_new16, self.v_new16, self.kc, self.vc,
                                              self.v_scale, self.bt[r], self.seq_lens,
                                              self.max_len, self.w.sm_scale, self.chunk, self.ws,
                                              self.err)
        elif self.mode == "balanced_fused":
            # block table and lengths are never written by the preceding kernel
            K.k16v8_paged_decode_append_balanced_split(
                self.q, self.k_new16, self.v_new16, self.kc, self.vc, self.v_scale, self.bt[r],
                self.seq_lens, self.w.sm_scale, self.ws, self.out, self.lse, self.err,
                flags=K.DECODE_METADATA_READY)
        elif self.mode == "balanced":
            # block table and lengths are never written by the preceding kernel
            K.k16v8_paged_decode_balanced_split(self.q, self.kc, self.vc, self.v_scale,
                                                self.bt[r], self.seq_lens, self.w.sm_scale,
                                                self.ws, self.out, self.lse, self.err,
                                                flags=K.DECODE_METADATA_READY)
        else:
            K.k16v8_paged_decode_split(self.q, self.kc, self.vc, self.v_scale, self.bt[r],
                                       self.seq_lens, self.max_len, self.w.sm_scale, self.chunk,
                                       self.ws, self.err)

    def merge(self):
        K = self.K
        if self.mode == "whole":  # the split kernel wrote out / lse
            return
        if self.balanced:
            K.k16v8_merge_balanced(self.ws, self.w.num_kv_heads, self.out, self.lse)
        else:
            K.k16v8_merge_states(self.po, self.pl, self.seq_lens, self.chunk, self.out, self.lse)

    def capture(self, steps, with_events=False):
        """One CUDA graph per step, so the timed region replays pre-built
        launches without host overhead."""
        torch = self.torch
        side = torch.cuda.Stream(self.dev)
        graphs, evs = [], []
        for i in range(steps):
            g = torch.cuda.CUDAGraph()
            e = None
            with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
                self.step(i, e)
            graphs.append(g)
            evs.append(e)
        torch.cuda.synchronize(self.dev)
        return graphs, evs

    def run(self, steps, warmup):
        """Time `steps` decode steps captured back to back into one CUDA graph
        (no timing nodes inside, so the programmatic launch edges between all
        the kernels stay intact, as in a whole-model decode graph), then the
        average duration of each kernel from a graph of `steps` launches of
        that kernel alone over the same state."""
        torch = self.torch
        for i in range(warmup):  # eager warm-up also configures kernel attributes
            self.step(i)
        torch.cuda.synchronize(self.dev)
        side = torch.cuda.Stream(self.dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
            for i in range(steps):
                self.step(i)
        for _ in range(-(-warmup // steps)):
            graph.replay()
        torch.cuda.synchronize(self.dev)
        barrier()
        torch.cuda.synchronize(self.dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        graph.replay()
        t1.record()
        torch.cuda.synchronize(self.dev)
        barrier()
        total_ms = t0.elapsed_time(t1)
        seg = self.per_kernel(steps)
        if self.K.k16v8_read_device_error(self.err) != 0:
            raise RuntimeError("device error flag raised during the benchmark")
        return total_ms / steps, seg

    def per_kernel(self, steps):
        """Average launch duration per kernel: one graph per kernel kind with
        `steps` launches (rotating over the pool replicas), timed as a block."""
        torch, K = self.torch, self.K
        outs = []
        kinds = [
            (lambda i: None) if self.fused else (
                lambda i: K.k16v8_kv_append(self.k_new, self.v_new, self.slots_new[i % self.R],
                                            self.v_scale, self.kc, self.vc, self.err)),
            self.split,
            lambda i: self.merge()]
        side = torch.cuda.Stream(self.dev)
        for ki, fn in enumerate(kinds):
            if (ki == 0 and self.fused) or (ki == 2 and self.mode == "whole"):
                outs.append(0.0)
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
                for i in range(steps):
                    fn(i)
            g.replay()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            g.replay()
            t1.record()
            torch.cuda.synchronize(self.dev)
            outs.append(t0.elapsed_time(t1) / steps)
        return np.array([outs])

    def run_e2e(self, steps, warmup, nbuf=3):
        """Same steps through host buffers.  Every step copies its inputs (q,
        the new K/V rows, lengths, block table, slots) from one pinned host
        buffer to the device in one copy, runs the launches, and reads out +
        lse back into a pinned host buffer in one copy, all inside the timed
        region (host wall clock).  The copies are pipelined as a serving loop
        would: later steps' inputs go up (copy stream) and earlier steps'
        results come down (a second copy stream) while step i computes, with
        `nbuf` device buffers each way; every step still moves all of its
        bytes.
        The steps are captured back to back in one CUDA graph."""
        torch, K, w = self.torch, self.K, self.w
        align = lambda n: (n + 255) // 256 * 256
        parts = [("q", self.q), ("k_new", self.k_new), ("v_new", self.v_new),
                 ("seq_lens", self.seq_lens), ("bt", self.bt[0]), ("slots", self.slots_new[0])]
        offs, total = {}, 0
        for name, t in parts:
            offs[name] = total
            total += align(t.numel() * t.element_size())
        h_in = []
        for r in range(self.R):  # one pinned input image per pool replica
            buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
            for name, t in parts:
                src = {"bt": self.bt[r], "slots": self.slots_new[r]}.get(name, t)
                nb = src.numel() * src.element_size()
                buf[offs[name]:offs[name] + nb].copy_(src.cpu().contiguous().view(-1)
                                                      .view(torch.uint8))
            h_in.append(buf)
        o_bytes = self.out.numel() * 2
        out_total = align(o_bytes) + self.lse.numel() * 4
        d_in = [torch.empty(total, dtype=torch.uint8, device=self.dev) for _ in range(nbuf)]
        d_out = [torch.empty(out_total, dtype=torch.uint8, device=self.dev) for _ in range(nbuf)]
        h_out = [torch.empty(out_total, dtype=torch.uint8).pin_memory() for _ in range(nbuf)]

        def views(k):
            v = lambda name, t: d_in[k][offs[name]:offs[name] + t.numel() * t.element_size()] \
                .view(t.dtype).view(t.shape)
            d = {name: v(name, t) for name, t in parts}
            d["out"] = d_out[k][:o_bytes].view(torch.float16).view(self.out.shape)
            d["lse"] = d_out[k][align(o_bytes):].view(torch.float32).view(self.lse.shape)
            return d

        dv = [views(k) for k in range(nbuf)]
        h2d = sum(t.numel() * t.element_size() for _, t in parts)
        d2h = o_bytes + self.lse.numel() * 4

        def split_launches(d):  # the step's launches up to the attention split
            if self.mode == "whole":
                K.k16v8_paged_decode_append_attention(
                    d["q"], d["k_new"], d["v_new"], self.kc, self.vc, self.v_scale, d["bt"],
                    d["seq_lens"], self.max_len, w.sm_scale, self.chunk, self.ws, d["out"],
                    d["lse"], self.err)
            elif self.mode == "balanced_fused":
                K.k16v8_paged_decode_append_balanced_split(
                    d["q"], d["k_new"], d["v_new"], self.kc, self.vc, self.v_scale, d["bt"],
                    d["seq_lens"], w.sm_scale, self.ws, d["out"], d["lse"], self.err,
                    flags=K.DECODE_METADATA_READY)
            elif self.mode == "fused":
                K.k16v8_paged_decode_append_split(
                    d["q"], d["k_new"], d["v_new"], self.kc, self.vc, self.v_scale, d["bt"],
                    d["seq_lens"], self.max_len, w.sm_scale, self.chunk, self.ws, self.err)
            else:
                K.k16v8_kv_append(d["k_new"], d["v_new"], d["slots"], self.v_scale, self.kc,
                                  self.vc, self.err)
                if self.mode == "balanced":
                    K.k16v8_paged_decode_balanced_split(
                        d["q"], self.kc, self.vc, self.v_scale, d["bt"], d["seq_lens"],
                        w.sm_scale, self.ws, d["out"], d["lse"], self.err,
                        flags=K.DECODE_METADATA_READY)
                else:
                    K.k16v8_paged_decode_split(d["q"], self.kc, self.vc, self.v_scale, d["bt"],
                                               d["seq_lens"], self.max_len, w.sm_scale,
                                               self.chunk, self.ws, self.err)

        def merge_launch(d):
            if self.mode == "whole":
                return
            if self.balanced:
                K.k16v8_merge_balanced(self.ws, w.num_kv_heads, d["out"], d["lse"])
            else:
                K.k16v8_merge_states(self.po, self.pl, d["seq_lens"], self.chunk, d["out"],
                                     d["lse"])

        up = torch.cuda.Stream(self.dev)
        down = torch.cuda.Stream(self.dev)

        def run(n, first):
            """n pipelined steps on the current stream (step indices first..)."""
            main = torch.cuda.current_stream(self.dev)
            ev = lambda: torch.cuda.Event()
            in_ready, done, read = [None] * n, [None] * n, [None] * n
            up.wait_stream(main)
            down.wait_stream(main)

            def upload(i):  # step i's inputs into buffer i % nbuf
                with torch.cuda.stream(up):
                    if i >= nbuf:
                        up.wait_event(done[i - nbuf])  # that buffer's last reader is done
                    d_in[i % nbuf].copy_(h_in[(first + i) % self.R], non_blocking=True)
                    in_ready[i] = ev()
                    in_ready[i].record(up)

            for i in range(min(nbuf - 1, n)):
                upload(i)
            # A step's waits (its inputs uploaded, its output buffer read back)
            # go in before the previous step's merge, so that the launches of
            # consecutive kernels stay adjacent and keep their programmatic
            # overlap; the order still holds through that merge.
            main.wait_event(in_ready[0])
            for i in range(n):
                k = i % nbuf
                if i + nbuf - 1 < n:
                    upload(i + nbuf - 1)
                split_launches(dv[k])
                if i + 1 < n:
                    main.wait_event(in_ready[i + 1])
                    if i + 1 >= nbuf:
                        main.wait_event(read[i + 1 - nbuf])
                merge_launch(dv[k])
                done[i] = ev()
                done[i].record(main)
                with torch.cuda.stream(down):
                    down.wait_event(done[i])
                    h_out[k].copy_(d_out[k], non_blocking=True)
                    read[i] = ev()
                    read[i].record(down)
            main.wait_stream(up)
            main.wait_stream(down)

        run(max(warmup, 2), 0)
        torch.cuda.synchronize(self.dev)
        side = torch.cuda.Stream(self.dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
            run(steps, 0)
        graph.replay()
        torch.cuda.synchronize(self.dev)
        barrier()
        t0 = time.perf_counter()
        graph.replay()
        torch.cuda.synchronize(self.dev)
        dt = (time.perf_counter() - t0) * 1e3 / steps
        barrier()
        last = dv[(steps - 1) % nbuf]
        if not torch.equal(last["out"], self.out):
            raise RuntimeError("end-to-end step disagrees with the device-resident step")
        host = h_out[(steps - 1) % nbuf][:o_bytes].view(torch.float16).view(self.out.shape)
        if not torch.equal(host, self.out.cpu()):
            raise RuntimeError("end-to-end result read back to the host disagrees")
        return dt, h2d, d2h


# ---- the FP16-KV control on the same kernels ---------------------------------------

def fp16_control_line(w, device, chunk, steps, warmup, hbm_peak):
    """Decode step (append + split + merge) over a pool whose values are fp16
    (5,120 B per token per layer), same workload and launch shape."""
    import torch
    from fp8_paged_kv_append_gb300 import k16v8 as K
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    B, hq, d = w.q.shape
    P = w.num_pages
    R = max(1, -(-4 * L2_BYTES // (P * w.num_kv_heads * 16 * d * 4)))
    kc = torch.empty((R * P, w.num_kv_heads, 16, d), dtype=torch.float16, device=device)
    vc = torch.empty_like(kc)
    k_all, v_all = td(w.k_tok), td(w.v_tok.astype(np.float16))
    bts, slots = [], []
    for r in range(R):
        K.k16v8_kv_append_v16(k_all, v_all, td(w.slot_mapping + r * P * 16), kc, vc)
        bts.append(td(w.block_table + r * P))
        slots.append(td(w.slot_mapping[w.new_rows] + r * P * 16))
    del k_all, v_all
    k_new, v_new = td(w.k_tok[w.new_rows]), td(w.v_tok[w.new_rows].astype(np.float16))
    q, lens = td(w.q), td(w.seq_lens)
    L = int(w.seq_lens.max())
    ws = torch.empty(K.k16v8_decode_workspace_size(B, hq, d, L, chunk), dtype=torch.uint8,
                     device=device)
    po, pl = K.workspace_views(ws, B, hq, d, L, chunk)
    out = torch.empty((B, hq, d), dtype=torch.float16, device=device)
    lse = torch.empty((B, hq), dtype=torch.float32, device=device)

    def split(i):
        K.k16v8_paged_decode_split_v16(q, kc, vc, bts[i % R], lens, L, w.sm_scale, chunk, ws)

    def step(i):
        K.k16v8_kv_append_v16(k_new, v_new, slots[i % R], kc, vc)
        split(i)
        K.k16v8_merge_states(po, pl, lens, chunk, out, lse)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(device)
    side = torch.cuda.Stream(device)
    times = []
    for fn in (step, split):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
            for i in range(steps):
                fn(i)
        g.replay()
        torch.cuda.synchronize(device)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        g.replay()
        t1.record()
        torch.cuda.synchronize(device)
        times.append(t0.elapsed_time(t1) / steps)
    kvb = int(w.seq_lens.astype(np.int64).sum()) * w.num_kv_heads * d * 4
    split_bytes = kvb + B * hq * d * 2
    return {"us_per_layer_step": round(times[0] * 1e3, 2),
            "split_us": round(times[1] * 1e3, 2),
            "kv_bytes_per_step": kvb, "value": round(kvb / (times[0] * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "split_frac_of_hbm_peak": round(split_bytes / (times[1] * 1e-3) / 1e9 / hbm_peak, 4),
            "split_frac_of_nominal": round(split_bytes / (times[1] * 1e-3) / 1e9
                                           / NOMINAL_HBM_GBS, 4)}


# ---- chunked prefill on the GPU --------------------------------------------------

def prefill_flops(p) -> float:
    """Algorithmic flops of a prefill workload: 4 * D * Hq per visible
    (query, key) pair (Q.K^T and P.V over the causal prefix)."""
    pairs = 0
    for call in p.calls:
        for st, ql in zip(call.starts.tolist(), call.qlens.tolist()):
            pairs += sum(st + i + 1 for i in range(ql))
    return 4.0 * p.head_dim * p.num_qo_heads * pairs


class PrefillBench:
    """All calls of a chunked-prefill workload (per call: kv_append of the
    chunk, then prefill attention), replayed from CUDA graphs."""

    def __init__(self, p, device, split=True):
        """split: the KV-split call (parts chosen by the library; one
        zero-filled workspace for all calls) instead of the plain call."""
        import torch
        from fp8_paged_kv_append_gb300 import k16v8 as K
        self.K, self.torch, self.p, self.dev = K, torch, p, device
        self.split = split
        td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.kc = torch.zeros((p.num_pages, p.num_kv_heads, 16, p.head_dim), dtype=torch.float16,
                              device=device)
        self.vc = torch.zeros((p.num_pages, p.num_kv_heads, 16, p.head_dim), dtype=torch.uint8,
                              device=device)
        self.vs = td(p.v_scale)
        self.calls = []
        for call in p.calls:
            rows = call.rows
            q = td(p.q[rows])
            self.calls.append(dict(
                k=td(p.k_tok[rows]), v=td(p.v_tok[rows]), slots=td(p.slot_mapping[rows]), q=q,
                indptr=td(call.qo_indptr), bt=td(call.block_table), lens=td(call.seq_lens),
                max_qlen=int(call.qlens.max()),
                out=torch.empty(q.shape, dtype=torch.float16, device=device),
                lse=torch.empty(q.shape[:2], dtype=torch.float32, device=device)))
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        for c, pc in zip(self.calls, p.calls):
            c["max_len"] = int(pc.seq_lens.max())  # the scheduler knows its lengths
        n = max(K.k16v8_prefill_workspace_size(c["max_qlen"], len(pc.seq_lens), p.num_qo_heads,
                                               p.num_kv_heads, p.head_dim, 0, c["max_len"])
                for c, pc in zip(self.calls, p.calls))
        self.ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=device)
        self.ws_bytes = n

    def append(self, c):
        self.K.k16v8_kv_append(c["k"], c["v"], c["slots"], self.vs, self.kc, self.vc, self.err)

    def attend(self, c):
        if self.split:
            self.K.k16v8_paged_prefill_attention_split(
                c["q"], c["indptr"], c["max_qlen"], self.kc, self.vc, self.vs, c["bt"], c["lens"],
                self.p.sm_scale, self.ws, c["out"], c["lse"], self.err, max_seq_len=c["max_len"])
        else:
            self.K.k16v8_paged_prefill_attention(c["q"], c["indptr"], c["max_qlen"], self.kc,
                                                 self.vc, self.vs, c["bt"], c["lens"],
                                                 self.p.sm_scale, c["out"], c["lse"], self.err)

    def step(self):
        for c in self.calls:
            self.append(c)
            self.attend(c)

    def _graph(self, fn, reps):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream(self.dev),
                              capture_error_mode="thread_local"):
            for _ in range(reps):
                fn()
        return g

    def _time(self, g, reps_inside):
        torch = self.torch
        g.replay()
        torch.cuda.synchronize(self.dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        g.replay()
        t1.record()
        torch.cuda.synchronize(self.dev)
        return t0.elapsed_time(t1) / reps_inside

    def run(self, steps, warmup):
        torch = self.torch
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize(self.dev)
        step_ms = self._time(self._graph(self.step, steps), steps)
        attn_ms = self._time(self._graph(lambda: [self.attend(c) for c in self.calls], steps), steps)
        app_ms = self._time(self._graph(lambda: [self.append(c) for c in self.calls], steps), steps)
        if self.K.k16v8_read_device_error(self.err) != 0:
            raise RuntimeError("device error flag raised during the prefill benchmark")
        return step_ms, attn_ms, app_ms


def kv_append_bytes(p) -> int:
    """Algorithmic bytes of writing every prompt token to the cache: per token
    and KV head the fp16 K and V rows read (2 + 2 B per element), the fp16 K
    row and the E4M3 V row written (2 + 1 B per element)."""
    return int(p.q.shape[0]) * p.num_kv_heads * p.head_dim * (2 + 2 + 2 + 1)


def prefill_line(p, device, steps, warmup, tensor_peak, hbm_peak, workload=None):
    """The prefill calls through the KV-split entry point (the library picks
    the parts; 1 when the items fill the GPU), and the plain call beside it
    when the split one split anything.  The cache write of the prompts
    (kv_append, HBM-bound) gets its own roofline."""
    pb = PrefillBench(p, device, split=True)
    step_ms, attn_ms, app_ms = pb.run(steps, warmup)
    fl = prefill_flops(p)
    ab = kv_append_bytes(p)
    line = {"workload": p.name, "calls": len(p.calls), "query_tokens": int(p.q.shape[0]),
            "ms_per_prompt_batch": round(step_ms, 4),
            "prefill_attention_ms": round(attn_ms, 4), "kv_append_ms": round(app_ms, 4),
            "algorithmic_tflop": round(fl / 1e12, 4),
            "prefill_tflops": round(fl / (attn_ms * 1e-3) / 1e12, 1),
            "frac_of_fp16_tensor_peak": round(fl / (attn_ms * 1e-3) / 1e12 / tensor_peak, 4),
            "kv_split_workspace_bytes": pb.ws_bytes,
            "kv_append_roofline": {
                "bound": "hbm", "kernel": "kv_append_kernel", "launches": len(p.calls),
                "algorithmic_bytes": ab,
                "achieved": round(ab / (app_ms * 1e-3) / 1e9, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(ab / (app_ms * 1e-3) / 1e9 / hbm_peak, 4),
                "frac_of_nominal": round(ab / (app_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
                "traffic": traffic_from_profiles(workload, "kv_append") if workload else None}}
    if pb.ws_bytes:
        del pb
        plain = PrefillBench(p, device, split=False)
        _, attn0, _ = plain.run(steps, warmup)
        line["unsplit_prefill_attention_ms"] = round(attn0, 4)
        line["unsplit_prefill_tflops"] = round(fl / (attn0 * 1e-3) / 1e12, 1)
    return line


# ---- full-pool ragged decode across 40 layers (the headline workload) ---------------

FULLPOOL_SEED = 4
NOMINAL_HBM_GBS = 8000.0  # nominal GB300 HBM3e bandwidth, for the second fraction

SCHEDULE_TEXT = {
    "auto": "automatic per batch: the load-balanced split when it gives at most 160 "
            "(sequence, KV head, page) tiles per CTA, else split-KV chunks of 512 tokens; the "
            "new token's cache append folded into the split kernel either way; LSE merge",
    "chunked": "split-KV chunks of 512 tokens (separate append), LSE merge",
    "fused": "split-KV chunks of 512 tokens with the new token's cache append folded in, "
             "LSE merge",
    "balanced": "load-balanced split (one full wave of SMs x 4 CTAs over equal tile ranges, "
                "separate append), LSE merge of cut segments",
    "balanced_fused": "load-balanced split with the new token's cache append folded in, LSE "
                      "merge of cut segments",
    "whole": "one CTA per (sequence, KV head) over the whole sequence with the new token's "
             "cache append folded in; the output written by that kernel (no merge)",
}


def fullpool_config(lay, layers, schedule):
    """The full-pool workload's config (host-side facts only, so the
    reference arm reports the same one)."""
    P = lay.num_pages
    L = lay.seq_lens.astype(np.int64)
    gib = layers * P * 10 * 16 * 128 * 3 / 2 ** 30
    return {"workload": f"full-pool ragged decode step through {layers} layers: per layer a pool "
                        f"of {P * 16:,} slots ({P:,} pages of 16 tokens; {gib:.1f} GiB of FP16 K + "
                        f"E4M3 V over all layers), batch {len(L)}, seq_lens uniform in [1, 8192] "
                        f"redrawn until the batch fits the pool, 40 q / 10 KV heads, head_dim 128",
            "layers": layers, "batch": int(len(L)),
            "seq_lens": f"{int(L.min())}..{int(L.max())}",
            "cached_tokens_per_layer": int(L.sum()),
            "schedule": SCHEDULE_TEXT[schedule],
            "l2": "inputs larger than L2: every step streams the distinct pools of all layers "
                  f"({layers * int(L.sum()) * 3840 / 1e9:.1f} GB of KV) through the 129 MB L2"}


class FullPoolBench:
    """The decode step through every layer of the 32 GiB pool (per layer: the
    new token's append, split-KV attention, merge), captured as one CUDA
    graph per step by MultiLayerDecode."""

    def __init__(self, device, layers=40, schedule="auto", split_chunk=512):
        import torch
        from fp8_paged_kv_append_gb300 import k16v8 as K
        from fp8_paged_kv_append_gb300 import workloads
        from fp8_paged_kv_append_gb300.decode_step import MultiLayerDecode
        self.torch, self.K, self.dev, self.layers = torch, K, device, layers
        self.split_chunk = split_chunk
        self.MLD = MultiLayerDecode
        self.lay = lay = workloads.fullpool_layout(seed=FULLPOOL_SEED)
        P, B = lay.num_pages, len(lay.seq_lens)
        self.B = B
        self.pools = [workloads.device_layer_pool(1000 + l, P, device) for l in range(layers)]
        g = torch.Generator(device=device)
        g.manual_seed(44)
        rnd = lambda shape: torch.randn(shape, generator=g, device=device, dtype=torch.float16)
        self.qs = [rnd((B, 40, 128)) for _ in range(layers)]
        self.kn = [rnd((B, 10, 128)) for _ in range(layers)]
        self.vn = [rnd((B, 10, 128)) for _ in range(layers)]
        L = lay.seq_lens.astype(np.int64)
        self.L = L
        self.slots = (lay.block_table[np.arange(B), (L - 1) // 16].astype(np.int64) * 16
                      + (L - 1) % 16)
        td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.step = self.make_step(td(lay.block_table), td(lay.seq_lens), td(self.slots),
                                   schedule)
        self.schedule = self.step.schedule
        self.outs = [torch.empty((B, 40, 128), dtype=torch.float16, device=device)
                     for _ in range(layers)]
        self.lses = [torch.empty((B, 40), dtype=torch.float32, device=device)
                     for _ in range(layers)]
        self.step.capture(self.qs, self.kn, self.vn, self.outs, self.lses)
        torch.cuda.synchronize(device)

    def make_step(self, bt, lens, slots, schedule):
        return self.MLD([p[0] for p in self.pools], [p[1] for p in self.pools],
                        [p[2] for p in self.pools], bt, lens, slots, int(self.L.max()), 40,
                        split_chunk=self.split_chunk, schedule=schedule)

    @property
    def kv_bytes_per_layer(self) -> int:
        return int(self.L.sum()) * 10 * 128 * 3

    def run(self, steps, warmup):
        """ms per whole step: `steps` replays of the step graph between CUDA
        events on the launching stream, a barrier and a synchronise on both
        sides."""
        torch = self.torch
        for _ in range(warmup):
            self.step.replay()
        torch.cuda.synchronize(self.dev)
        barrier()
        torch.cuda.synchronize(self.dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            self.step.replay()
        t1.record()
        torch.cuda.synchronize(self.dev)
        barrier()
        if self.step.check() != 0:
            raise RuntimeError("device error flag raised during the full-pool benchmark")
        return t0.elapsed_time(t1) / steps

    def per_kernel(self, reps=2):
        """Average launch duration (ms) of the attention split and of the
        merge: one graph per kind holding that launch for every layer (a
        different pool each), replayed `reps` times between CUDA events on
        the launching stream."""
        torch, s = self.torch, self.step
        # The layers share one workspace, so back-to-back splits leave only the
        # last layer's partials for the merges: they write scratch outputs,
        # never the step's.
        so = [torch.empty_like(o) for o in self.outs]
        sl = [torch.empty_like(x) for x in self.lses]
        res = []
        for fn in (lambda li: s.split(li, self.qs[li], self.kn[li], self.vn[li], so[li], sl[li],
                                      append=False),
                   lambda li: s.merge(li, so[li], sl[li])):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=torch.cuda.Stream(self.dev),
                                  capture_error_mode="thread_local"):
                for li in range(self.layers):
                    fn(li)
            g.replay()
            torch.cuda.synchronize(self.dev)
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            for _ in range(reps):
                g.replay()
            t1.record()
            torch.cuda.synchronize(self.dev)
            res.append(t0.elapsed_time(t1) / (reps * self.layers))
        if s.check() != 0:
            raise RuntimeError("device error flag raised while timing the kernels")
        return res

    def run_e2e(self, steps, warmup, nbuf=2):
        """The same step through host buffers, as a serving loop drives it:
        every step copies all layers' queries and new K/V rows plus the
        lengths, block table and slots from pinned host memory to the device
        in one copy, replays the step graph over that buffer, and reads every
        layer's out + lse back into pinned host memory in one copy.  `nbuf`
        device buffers each way, so step i+1's inputs go up while step i
        computes.  Host wall clock over `steps` steps.  Returns (ms per step,
        H2D bytes per step, D2H bytes per step)."""
        torch = self.torch
        align = lambda n: (n + 255) // 256 * 256
        lay = self.lay
        meta = [("seq_lens", torch.from_numpy(lay.seq_lens.astype(np.int32))),
                ("bt", torch.from_numpy(np.ascontiguousarray(lay.block_table.astype(np.int32)))),
                ("slots", torch.from_numpy(self.slots.astype(np.int64)))]
        parts = list(meta)
        for li in range(self.layers):
            parts += [(f"q{li}", self.qs[li]), (f"k{li}", self.kn[li]), (f"v{li}", self.vn[li])]
        offs, total = {}, 0
        for name, t in parts:
            offs[name] = total
            total += align(t.numel() * t.element_size())
        h_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for name, t in parts:
            nb = t.numel() * t.element_size()
            h_in[offs[name]:offs[name] + nb].copy_(t.detach().cpu().contiguous().view(-1)
                                                  .view(torch.uint8))
        o_bytes = self.outs[0].numel() * 2
        l_bytes = self.lses[0].numel() * 4
        o_stride = align(o_bytes) + align(l_bytes)
        out_total = self.layers * o_stride
        d_in = [torch.empty(total, dtype=torch.uint8, device=self.dev) for _ in range(nbuf)]
        d_out = [torch.empty(out_total, dtype=torch.uint8, device=self.dev) for _ in range(nbuf)]
        h_out = [torch.empty(out_total, dtype=torch.uint8).pin_memory() for _ in range(nbuf)]

        def view(buf, name, like):
            nb = like.numel() * like.element_size()
            return buf[offs[name]:offs[name] + nb].view(like.dtype).view(like.shape)

        graphs, outs_k, lses_k = [], [], []
        for k in range(nbuf):
            d_in[k].copy_(h_in)
            sb = self.make_step(view(d_in[k], "bt", meta[1][1]),
                                view(d_in[k], "seq_lens", meta[0][1]),
                                view(d_in[k], "slots", meta[2][1]), self.schedule)
            qs = [view(d_in[k], f"q{li}", self.qs[li]) for li in range(self.layers)]
            kn = [view(d_in[k], f"k{li}", self.kn[li]) for li in range(self.layers)]
            vn = [view(d_in[k], f"v{li}", self.vn[li]) for li in range(self.layers)]
            outs = [d_out[k][li * o_stride:li * o_stride + o_bytes].view(torch.float16)
                    .view(self.outs[0].shape) for li in range(self.layers)]
            lses = [d_out[k][li * o_stride + align(o_bytes):li * o_stride + align(o_bytes)
                             + l_bytes].view(torch.float32).view(self.lses[0].shape)
                    for li in range(self.layers)]
            sb.capture(qs, kn, vn, outs, lses)
            graphs.append(sb)
            outs_k.append(outs)
            lses_k.append(lses)
        torch.cuda.synchronize(self.dev)
        up = torch.cuda.Stream(self.dev)
        down = torch.cuda.Stream(self.dev)

        def run(n):
            main = torch.cuda.current_stream(self.dev)
            ev = torch.cuda.Event
            in_ready, done, read = [None] * n, [None] * n, [None] * n
            up.wait_stream(main)
            down.wait_stream(main)

            def upload(i):
                with torch.cuda.stream(up):
                    if i >= nbuf:
                        up.wait_event(done[i - nbuf])  # that buffer's last step is done
                    d_in[i % nbuf].copy_(h_in, non_blocking=True)
                    in_ready[i] = ev()
                    in_ready[i].record(up)

            upload(0)
            for i in range(n):
                k = i % nbuf
                if i + 1 < n:
                    upload(i + 1)
                main.wait_event(in_ready[i])
                if i >= nbuf:
                    main.wait_event(read[i - nbuf])  # its output buffer was read back
                graphs[k].replay()
                done[i] = ev()
                done[i].record(main)
                with torch.cuda.stream(down):
                    down.wait_event(done[i])
                    h_out[k].copy_(d_out[k], non_blocking=True)
                    read[i] = ev()
                    read[i].record(down)
            main.wait_stream(up)
            main.wait_stream(down)

        run(max(warmup, 2))
        torch.cuda.synchronize(self.dev)
        barrier()
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        run(steps)
        torch.cuda.synchronize(self.dev)
        dt = (time.perf_counter() - t0) * 1e3 / steps
        barrier()
        for sb in graphs:
            if sb.check() != 0:
                raise RuntimeError("device error flag raised during the end-to-end steps")
        last = (steps - 1) % nbuf
        host = h_out[last]
        for li in range(self.layers):
            o = host[li * o_stride:li * o_stride + o_bytes].view(torch.float16) \
                .view(self.outs[0].shape)
            if not torch.equal(o, self.outs[li].cpu()):
                raise RuntimeError(f"end-to-end output of layer {li} read back to the host "
                                   "disagrees with the device-resident step")
        h2d = sum(t.numel() * t.element_size() for _, t in parts)
        d2h = self.layers * (o_bytes + l_bytes)
        del graphs, d_in, d_out
        return dt, h2d, d2h


def fullpool_cpu_sample(nseq=8):
    """A bounded host-side sample of the full-pool workload for the oracle:
    `nseq` of its 64 sequences spread over the length range (the shortest,
    the longest and evenly spaced ranks between), one layer, drawn on the
    host with the same distributions (K, V fp16 N(0,1), V scales amax/448)."""
    from fp8_paged_kv_append_gb300 import workloads
    lay = workloads.fullpool_layout(seed=FULLPOOL_SEED)
    order = np.argsort(lay.seq_lens, kind="stable")
    pick = order[np.unique(np.linspace(0, len(order) - 1, nseq).round().astype(int))]
    lens = lay.seq_lens[pick]
    w = workloads.make_decode("full-pool sample", 77, lens)
    desc = (f"one layer, {len(lens)} of the {len(lay.seq_lens)} sequences (lengths "
            f"{', '.join(str(int(x)) for x in sorted(lens))}; {int(lens.sum())} cached tokens)")
    return w, desc


# ---- CPU baseline: the oracle on the host cores -------------------------------------

def oracle_decode_pass(w, okc, ovc, chunk, sample_b, nthreads):
    """One oracle decode step over sequences sample_b: append the new tokens,
    split partials, merge.  Returns KV bytes processed."""
    import oracle
    rows = w.new_rows[sample_b]
    oracle.kv_append(w.k_tok[rows], w.v_tok[rows], w.slot_mapping[rows], w.v_scale, okc, ovc)
    r = oracle.paged_decode(w.q[sample_b], okc, ovc, w.v_scale, w.block_table[sample_b],
                            w.seq_lens[sample_b], w.sm_scale, split_chunk=chunk,
                            nthreads=nthreads, want_full=False)
    nc = -(-w.seq_lens[sample_b] // chunk)
    oracle.merge(r["partial_o"], r["partial_lse"], nc)
    return int(w.seq_lens[sample_b].astype(np.int64).sum()) * w.num_kv_heads * w.head_dim * 3


def oracle_cache_for(w):
    import oracle
    okc = np.zeros((w.num_pages, w.num_kv_heads, 16, w.head_dim), np.float16)
    ovc = np.zeros((w.num_pages, w.num_kv_heads, 16, w.head_dim), np.uint8)
    oracle.kv_append(w.k_tok, w.v_tok, w.slot_mapping, w.v_scale, okc, ovc)
    return okc, ovc


def run_cpu_baseline(w, chunk, sample, desc, budget_s=12.0, single_budget_s=None):
    """Time the oracle, as it stands, on a bounded sample of the workload:
    decode passes over sequences `sample` of w until `budget_s` has passed,
    on every host core; then (single_budget_s, default a quarter of that) the
    same passes on one thread."""
    ncores = os.cpu_count() or 1
    okc, ovc = oracle_cache_for(w)

    def timed(nthreads, budget):
        t0 = time.perf_counter()
        bytes_done = passes = 0
        while True:
            bytes_done += oracle_decode_pass(w, okc, ovc, chunk, sample, nthreads)
            passes += 1
            el = time.perf_counter() - t0
            if el >= budget or passes >= 5000:
                return bytes_done / el / 1e9, passes, el

    v, passes, el = timed(ncores, budget_s)
    v1, passes1, el1 = timed(1, budget_s / 4 if single_budget_s is None else single_budget_s)
    return {"value": round(v, 4), "unit": "GB/s", "cores": ncores, "kind": "oracle",
            "sample": f"{passes} oracle decode steps (append + split partials + merge) over "
                      f"{desc}, {el:.1f} s wall",
            "single_thread_value": round(v1, 4),
            "single_thread_sample": f"{passes1} of the same steps on one thread, {el1:.1f} s"}


def prefill_cpu_baseline(p, row_stride=64, budget_s=4.0):
    """The oracle's prefill attention and cache write, as they stand, on a
    bounded sample of a prefill workload: the cache write of every prompt
    token (GB/s against kv_append's 8,960 B per token), then the causal
    attention of every row_stride-th query row of the first call (TFLOP/s
    against 4 D Hq (position + 1) flops per row), repeated for about
    budget_s on all host cores and once on one thread."""
    import oracle
    ncores = os.cpu_count() or 1
    okc = np.zeros((p.num_pages, p.num_kv_heads, 16, p.head_dim), np.float16)
    ovc = np.zeros((p.num_pages, p.num_kv_heads, 16, p.head_dim), np.uint8)
    t0 = time.perf_counter()
    oracle.kv_append(p.k_tok, p.v_tok, p.slot_mapping, p.v_scale, okc, ovc)
    t_app = time.perf_counter() - t0
    call = p.calls[0]
    q = np.ascontiguousarray(p.q[call.rows])
    rows = np.arange(0, len(call.rows), row_stride, dtype=np.int64)
    # absolute position of each sampled query row
    seq_of = np.searchsorted(call.qo_indptr, rows, side="right") - 1
    pos = (call.seq_lens[seq_of].astype(np.int64) - (call.qo_indptr[seq_of + 1]
           - call.qo_indptr[seq_of]) + (rows - call.qo_indptr[seq_of]))

    def flops_of(r):
        return float(4 * p.head_dim * p.num_qo_heads * int((pos[r] + 1).sum()))

    def timed(sel, nthreads, budget):
        t0 = time.perf_counter()
        n = 0
        while True:
            oracle.paged_prefill(q, call.qo_indptr, okc, ovc, p.v_scale, call.block_table,
                                 call.seq_lens, p.sm_scale, rows=rows[sel], nthreads=nthreads)
            n += 1
            el = time.perf_counter() - t0
            if el >= budget or n >= 1000:
                return flops_of(sel) * n / el / 1e12, n, el

    every = np.arange(len(rows))
    v, n, el = timed(every, ncores, budget_s)
    one = every[::4]  # the single-thread pass takes a quarter of the rows
    v1, n1, el1 = timed(one, 1, 0.0)
    return {"value": round(v, 6), "unit": "TFLOP/s", "cores": ncores, "kind": "oracle",
            "sample": f"{n} oracle passes over every {row_stride}th query row of the first call "
                      f"({len(rows)} rows, {flops_of(every) / 1e9:.2f} GFLOP each), {el:.1f} s "
                      "wall",
            "single_thread_value": round(v1, 6),
            "single_thread_sample": f"{n1} pass over every {4 * row_stride}th row on one "
                                    f"thread, {el1:.1f} s",
            "kv_append": {"value": round(kv_append_bytes(p) / t_app / 1e9, 4), "unit": "GB/s",
                          "threads": 1,
                          "sample": f"the cache write of all {p.q.shape[0]} prompt tokens, "
                                    f"{t_app:.2f} s"}}


# ---- decode lines of one layer ------------------------------------------------------

def make_workload(name):
    from fp8_paged_kv_append_gb300 import workloads
    if name == "1k":
        return workloads.decode_1k_b32(), "decode 1K/batch 32", 384
    if name == "8k":
        return workloads.decode_8k_b16(), "decode 8K/batch 16", 512
    raise SystemExit(f"unknown workload {name}")


def config_of(w, label, chunk, replicas, mode="balanced"):
    if mode in ("balanced", "balanced_fused"):
        sched = ("load-balanced split: one full wave (SMs x 4 CTAs) of equal (sequence, KV "
                 "head, page) tile ranges, LSE merge of cut segments")
    elif mode == "whole":
        sched = ("one CTA per (sequence, KV head) over the whole sequence, the output written "
                 "by that kernel (no merge)")
    else:
        sched = f"split-KV chunks of {chunk} tokens, LSE merge"
    if mode in ("fused", "balanced_fused", "whole"):
        sched += "; the new token's cache append folded into the split kernel"
    return {"workload": f"Phi-4-shaped {label}: one layer, 40 q / 10 KV heads, head_dim 128, "
                        "16-token pages, FP16 K + E4M3 V",
            "batch": int(w.batch), "seq_lens": f"{int(w.seq_lens.min())}..{int(w.seq_lens.max())}",
            "cached_tokens": int(w.seq_lens.sum()), "schedule": sched,
            "l2": f"{replicas} rotating pool replicas (>= 4x L2) so every step reads HBM"}


KERNEL_NAMES = {
    "chunked": ("decode_split", "merge_states", "decode_split_kernel"),
    "balanced": ("decode_balanced", "merge_balanced", "decode_balanced_kernel"),
    "fused": ("decode_append_split", "merge_states", "decode_split_kernel<append>"),
    "balanced_fused": ("decode_append_balanced", "merge_balanced",
                       "decode_balanced_kernel<append>"),
    "whole": ("decode_append_whole", None, "decode_split_kernel<append>"),
}
# launches per one-layer decode step
LAUNCHES = {"chunked": 3, "balanced": 3, "fused": 2, "balanced_fused": 2, "whole": 1}


def kernel_us_of(mode, append_ms, split_ms, merge_ms):
    """Average launch duration (µs) of each kernel a step of this schedule
    launches (no separate append for the fused schedules, no merge for
    "whole")."""
    split_name, merge_name, _ = KERNEL_NAMES[mode]
    out = {}
    if mode not in ("fused", "balanced_fused", "whole"):
        out["kv_append"] = round(append_ms * 1e3, 2)
    out[split_name] = round(split_ms * 1e3, 2)
    if merge_name:
        out[merge_name] = round(merge_ms * 1e3, 2)
    return out


def roofline(algo_bytes, kernel_ms, hbm_peak, peak_kind, kernel, traffic):
    """The roofline object of an HBM-bound kernel: algorithmic bytes per
    launch over its average launch duration, against the measured copy
    bandwidth and, beside it, the nominal HBM3e peak."""
    achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
            "peak_kind": f"{peak_kind} (copy bandwidth)",
            "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "nominal_peak": NOMINAL_HBM_GBS, "kernel": kernel,
            "algorithmic_bytes_per_launch": int(algo_bytes),
            "kernel_us": round(kernel_ms * 1e3, 2)}


def decode_line(w, label, chunk, mode, device, steps, hbm_peak, peak_kind, workload):
    """One-layer decode line (one workload, one schedule) with the roofline of
    its attention kernel."""
    import torch
    b = DecodeBench(w, device, split_chunk=chunk, mode=mode)
    ms, seg = b.run(steps, 3)
    kernel = KERNEL_NAMES[mode][2]
    kvb = kv_bytes(w)
    s_ms = float(np.mean(seg[:, 1]))
    sb = kvb + w.batch * w.num_qo_heads * w.head_dim * 2
    out = {"value": round(kvb / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "us_per_layer_step": round(ms * 1e3, 2),
           "kernel_us": kernel_us_of(mode, float(np.mean(seg[:, 0])), s_ms,
                                     float(np.mean(seg[:, 2]))),
           "roofline": roofline(sb, s_ms, hbm_peak, peak_kind, kernel,
                                traffic_from_profiles(workload, mode)),
           "step_frac_of_hbm_peak": round(kvb / (ms * 1e-3) / 1e9 / hbm_peak, 4),
           "step_frac_of_nominal": round(kvb / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
           "config": config_of(w, label, chunk, b.R, mode)}
    if mode in ("fused", "balanced_fused"):
        out["step"] = "append fused into the split kernel, then merge (2 launches)"
    elif mode == "whole":
        out["step"] = "append and output in the split kernel (1 launch)"
    del b
    torch.cuda.empty_cache()
    return out


# ---- the measured arm ---------------------------------------------------------------

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="fullpool", choices=["fullpool", "1k", "8k", "prefill"])
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the secondary lines (1K/b32, 8K/b16, prefill, FP16-KV control)")
    ap.add_argument("--all-schedules", action="store_true",
                    help="also time every decode schedule on 1K/b32, 8K/b16 and the full pool")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--decode", default=None, choices=list(MODES) + ["auto"],
                    help="decode schedule of the main line (default: auto on the full pool, "
                         "balanced_fused on one layer)")
    ap.add_argument("--split-chunk", type=int, default=0,
                    help="tokens per split-KV chunk of the chunked schedules (0: the workload's "
                         "default)")
    ap.add_argument("--layers", type=int, default=40,
                    help="layers of the full-pool workload (fewer for profiling captures)")
    args = ap.parse_args(argv)
    if args.decode is None:
        args.decode = "auto" if args.workload == "fullpool" else DEFAULT_DECODE
    if args.decode == "auto" and args.workload != "fullpool":
        args.decode = DEFAULT_DECODE
    return args


def measure_fullpool(args, device, rank, world):
    """The headline: the 40-layer decode step over the 32 GiB pool."""
    import torch
    hbm_peak, _, peak_kind = load_peaks()
    fb = FullPoolBench(device, layers=args.layers, schedule=args.decode,
                       split_chunk=args.split_chunk or 512)
    warm = max(args.warmup, 3)
    clocks = ClockSampler(device.index or 0).start()
    ms = fb.run(args.steps, warm)
    clk = clocks.stop()
    split_ms, merge_ms = fb.per_kernel()
    e2e = None
    if not args.no_e2e:
        e2e = fb.run_e2e(max(5, args.steps // 2), 3)
    kernel = KERNEL_NAMES[fb.schedule][2]
    algo = fb.kv_bytes_per_layer + fb.B * 40 * 128 * 2
    units = fb.kv_bytes_per_layer * fb.layers
    per_layer = fb.step.launches_per_layer()
    res = {
        "ms": ms, "units": units, "e2e": e2e,
        "config": fullpool_config(fb.lay, fb.layers, args.decode),
        "fields": {
            "us_per_layer_step": round(ms * 1e3 / fb.layers, 2),
            "schedule_chosen": fb.schedule,
            "kernel_us": kernel_us_of(fb.schedule, 0.0, split_ms, merge_ms),
            "roofline": roofline(algo, split_ms, hbm_peak, peak_kind, kernel,
                                 traffic_from_profiles("fullpool", fb.schedule)),
            "step_frac_of_hbm_peak": round(units / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "step_frac_of_nominal": round(units / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
            "gpu_launches": per_layer * fb.layers * args.steps,
            "clocks": clk}}
    del fb
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu:
        w, desc = fullpool_cpu_sample()
        res["fields"]["cpu_baseline"] = run_cpu_baseline(w, 512, np.arange(w.batch), desc,
                                                         args.cpu_budget)
    return res


def measure_one_layer(args, device, rank, world):
    """A one-layer decode workload (1K/b32 or 8K/b16) as the main line."""
    hbm_peak, _, peak_kind = load_peaks()
    w, label, chunk = make_workload(args.workload)
    if args.split_chunk:
        chunk = args.split_chunk
    bench = DecodeBench(w, device, split_chunk=chunk, mode=args.decode)
    clocks = ClockSampler(device.index or 0).start()
    ms, seg = bench.run(args.steps, max(args.warmup, 3))
    clk = clocks.stop()
    e2e = None if args.no_e2e else bench.run_e2e(max(10, args.steps // 2), 3)
    kvb = kv_bytes(w)
    B, hq, d = w.q.shape
    split_ms = float(np.mean(seg[:, 1]))
    kernel = KERNEL_NAMES[args.decode][2]
    fields = {
        "us_per_layer_step": round(ms * 1e3, 2),
        "kernel_us": kernel_us_of(args.decode, float(np.mean(seg[:, 0])), split_ms,
                                  float(np.mean(seg[:, 2]))),
        "roofline": roofline(kvb + B * hq * d * 2, split_ms, hbm_peak, peak_kind, kernel,
                             traffic_from_profiles(args.workload, args.decode)),
        "gpu_launches": LAUNCHES[args.decode] * args.steps,
        "clocks": clk}
    res = {"ms": ms, "units": kvb, "e2e": e2e, "fields": fields,
           "config": config_of(w, label, chunk, bench.R, args.decode)}
    del bench
    if rank == 0 and world == 1 and not args.no_cpu:
        n = min(w.batch, 4)
        fields["cpu_baseline"] = run_cpu_baseline(
            w, chunk, np.arange(n), f"sequences 0..{n - 1} of the workload", args.cpu_budget)
    return res


def extra_lines(args, device):
    """Secondary lines: one-layer decode at 1K/b32, prefill with its cache
    write, the FP16-KV control, and 8K/b16 last (each with the roofline of
    its dominant kernel)."""
    import torch
    from fp8_paged_kv_append_gb300 import workloads
    hbm_peak, tpeak, peak_kind = load_peaks()
    n2 = max(10, args.steps // 2)
    extra = {}
    w1, l1, c1 = make_workload("1k")
    w8, l8, c8 = make_workload("8k")
    if args.workload != "1k":
        extra["decode_1k_b32"] = decode_line(w1, l1, c1, DEFAULT_DECODE, device, n2, hbm_peak,
                                             peak_kind, "1k")
    torch.cuda.empty_cache()
    extra["prefill"] = {
        "peak_tflops": tpeak,
        "peak_kind": f"{peak_kind} dense bf16 (fp16 has the same nominal rate)",
        "8x1024": prefill_line(workloads.prefill_8x1k(), device, 10, 3, tpeak, hbm_peak,
                               "prefill_8x1024"),
        "1x8192_in_8_chunks": prefill_line(workloads.prefill_1x8k(), device, 5, 2, tpeak,
                                           hbm_peak)}
    if not args.no_cpu:
        extra["prefill"]["8x1024"]["cpu_baseline"] = prefill_cpu_baseline(workloads.prefill_8x1k())
    for name, (wf, lf, cf) in (("decode_1k_b32", (w1, l1, c1)), ("decode_8k_b16", (w8, l8, c8))):
        torch.cuda.empty_cache()
        ctl = fp16_control_line(wf, device, cf, n2, 3, hbm_peak)
        ref = decode_line(wf, lf, cf, "chunked", device, n2, hbm_peak, peak_kind, name[7:9])
        ctl["k16v8_same_split_us_per_layer_step"] = ref["us_per_layer_step"]
        ctl["k16v8_speedup_over_fp16_kv"] = round(ctl["us_per_layer_step"] /
                                                  ref["us_per_layer_step"], 3)
        ctl["compared_with"] = "K16/V8 with the same chunked split (separate append)"
        extra[f"{name}_fp16_kv_control"] = ctl
    if args.all_schedules:
        for m in MODES:
            for name, (wf, lf, cf) in (("decode_1k_b32", (w1, l1, c1)),
                                       ("decode_8k_b16", (w8, l8, c8))):
                extra[f"{name}_{SUFFIX[m]}"] = decode_line(wf, lf, cf, m, device, n2, hbm_peak,
                                                           peak_kind, name[7:9])
            torch.cuda.empty_cache()
            fb = FullPoolBench(device, schedule=m)
            ms = fb.run(10, 3)
            extra[f"fullpool_40_layers_{SUFFIX[m]}"] = {
                "us_per_layer_step": round(ms * 1e3 / 40, 2),
                "value": round(fb.kv_bytes_per_layer * 40 / (ms * 1e-3) / 1e9, 1),
                "unit": "GB/s"}
            del fb
    if args.workload != "8k":
        torch.cuda.empty_cache()
        extra["decode_8k_b16"] = decode_line(w8, l8, c8, DEFAULT_DECODE, device, n2, hbm_peak,
                                             peak_kind, "8k")
    return extra


def measure_gpu(args, rank, world, local_rank):
    """Everything this rank measures on its GPU (replicas only: every rank
    runs the same seeded workload)."""
    import torch
    from fp8_paged_kv_append_gb300 import k16v8 as K
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    K.load_library()
    if args.workload == "fullpool":
        res = measure_fullpool(args, device, rank, world)
    else:
        res = measure_one_layer(args, device, rank, world)
    if not args.no_extra and rank == 0:
        res["fields"]["extra"] = extra_lines(args, device)
    return res


def same_config_on_all_ranks(config) -> None:
    """Replicas must run the same workload: compare every rank's config."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return
    mine = json.dumps(config, sort_keys=True)
    allc = [None] * dist.get_world_size()
    dist.all_gather_object(allc, mine)
    if any(c != mine for c in allc):
        raise RuntimeError("ranks ran different workloads")


def main(argv=None, backend=None, measure=None):
    """Parse the flags, set up the ranks (torchrun, replicas only), measure,
    aggregate (max time, summed units over ranks) and print one JSON line on
    rank 0.  `backend` / `measure` replace NCCL and the GPU section (tests)."""
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        return main_reference(args, rank, world)
    if args.workload == "prefill":
        return main_prefill(args)
    import torch.distributed as dist
    if world > 1:
        if backend is None:
            import torch
            torch.cuda.set_device(local_rank)
            backend = "nccl"
        dist.init_process_group(backend)
    res = (measure or measure_gpu)(args, rank, world, local_rank)
    same_config_on_all_ranks(res["config"])
    t_ms, units = aggregate(res["ms"], res["units"])
    line = {
        "metric": METRIC, "value": round(units / (t_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(t_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) Q/K/V, E4M3 V with per-head amax/448 scales)",
        "config": res["config"]}
    if res["e2e"] is not None:
        e_ms, h2d, d2h = res["e2e"]
        te_ms, _ = aggregate(e_ms, res["units"])
        line["e2e"] = {"value": round(units / (te_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                       "ms_per_step": round(te_ms, 4), "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h}
    line.update(res["fields"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return line


def main_prefill(args):
    """Prefill-only line (for profiling the tensor-core kernel)."""
    import torch
    from fp8_paged_kv_append_gb300 import k16v8 as K
    from fp8_paged_kv_append_gb300 import workloads
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    K.load_library()
    hbm_peak, tpeak, tkind = load_peaks()
    res = {"8x1024": prefill_line(workloads.prefill_8x1k(), device, args.steps,
                                  max(3, args.warmup), tpeak, hbm_peak, "prefill_8x1024")}
    if not args.no_extra:
        res["1x8192_in_8_chunks"] = prefill_line(workloads.prefill_1x8k(), device, args.steps,
                                                 max(3, args.warmup), tpeak, hbm_peak)
    print(json.dumps({"prefill": res, "peak_tflops": tpeak, "peak_kind": tkind}), flush=True)


def reference_workload(args):
    """(DecodeInputs, split chunk, sequences per step, sample text, config)
    of the reference arm, matching the measured arm's config."""
    if args.workload == "fullpool":
        from fp8_paged_kv_append_gb300 import workloads
        w, desc = fullpool_cpu_sample()
        lay = workloads.fullpool_layout(seed=FULLPOOL_SEED)
        return w, 512, np.arange(w.batch), desc, fullpool_config(lay, args.layers, args.decode)
    w, label, chunk = make_workload(args.workload)
    if args.split_chunk:
        chunk = args.split_chunk
    n = min(w.batch, 2)
    return (w, chunk, np.arange(n), f"sequences 0..{n - 1} of the workload",
            config_of(w, label, chunk, replicas_for(w), args.decode))


def main_reference(args, rank, world):
    """The reference arm: the oracle, as it stands, on the host cores, on a
    bounded sample of the same workload (rank 0 only)."""
    if rank != 0:
        return
    w, chunk, sample, desc, config = reference_workload(args)
    okc, ovc = oracle_cache_for(w)
    ncores = os.cpu_count() or 1
    for _ in range(max(args.warmup, 1)):
        oracle_decode_pass(w, okc, ovc, chunk, sample, ncores)
    t0 = time.perf_counter()
    done = 0
    for _ in range(args.steps):
        done += oracle_decode_pass(w, okc, ovc, chunk, sample, ncores)
    el = time.perf_counter() - t0
    val = round(done / el / 1e9, 4)
    line = {"metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": config,
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": ncores, "kind": "oracle",
                             "sample": f"each step: one oracle decode step (append + split "
                                       f"partials + merge) over {desc}"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return line


if __name__ == "__main__":
    main()
