#!/usr/bin/env python3
"""K16/V8 paged decode benchmark (one JSON line on stdout).

A step is one decode layer-step of the whole hot path: the append of each
sequence's new token (FP16 K + E4M3 V), paged decode attention split over
the KV sequence, and the LSE merge, on the Phi-4-shaped workload (40 query /
10 KV heads, d 128, 16-token pages).  The headline schedule folds the append
into the load-balanced split kernel (2 launches per step); the other
schedules, the FP16-KV control, the 40-layer full pool and prefill run as
extra lines.  Default workload: decode 1K/batch 32; `--workload 8k` selects
8K/batch 16.  The KV pool is replicated so that consecutive steps read
different copies (the rotation spans >= 4x the L2 size), which keeps the
timed reads coming from HBM.

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
    """nvidia-smi clock / throttle samples every 200 ms while running."""
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
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
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


MODES = ("chunked", "fused", "balanced", "balanced_fused")
DEFAULT_DECODE = "balanced_fused"  # schedule of the headline line
SUFFIX = {"chunked": "chunked", "fused": "fused_append", "balanced": "balanced",
          "balanced_fused": "balanced_fused_append"}

KERNEL_SOURCES = {
    "chunked": ("decode_split_1k_b32.md", ["decode.cu", "decode_page.cuh", "k16v8_device.cuh"]),
    "balanced": ("decode_balanced_1k_b32.md",
                 ["decode_balanced.cu", "decode_page.cuh", "k16v8_device.cuh"]),
    "balanced_fused": ("decode_balanced_append_1k_b32.md",
                       ["decode_balanced.cu", "decode_page.cuh", "k16v8_device.cuh"]),
    "fused": ("decode_split_append_1k_b32.md", ["decode.cu", "decode_page.cuh", "k16v8_device.cuh"]),
}


def sources_sha256(names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "fp8_paged_kv_append_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_from_profiles(mode: str):
    """DRAM bytes per launch of the decode attention kernel of `mode` from the
    committed ncu summary, or None when its sources changed since that
    capture."""
    prof, srcs = KERNEL_SOURCES[mode]
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
        its merge) or "balanced_fused" (append fused into the load-balanced
        split, its merge)."""
        import torch
        from fp8_paged_kv_append_gb300 import k16v8 as K
        assert mode in MODES
        self.K, self.torch, self.w, self.dev = K, torch, w, device
        self.chunk = split_chunk
        self.mode = mode
        self.fused = mode in ("fused", "balanced_fused")
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
        if self.mode == "fused":
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
            if ki == 0 and self.fused:
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
            if self.mode == "balanced_fused":
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
            "split_frac_of_hbm_peak": round(split_bytes / (times[1] * 1e-3) / 1e9 / hbm_peak, 4)}


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


def prefill_line(p, device, steps, warmup, tensor_peak):
    """The prefill calls through the KV-split entry point (the library picks
    the parts; 1 when the items fill the GPU), and the plain call beside it
    when the split one split anything."""
    pb = PrefillBench(p, device, split=True)
    step_ms, attn_ms, app_ms = pb.run(steps, warmup)
    fl = prefill_flops(p)
    line = {"workload": p.name, "calls": len(p.calls), "query_tokens": int(p.q.shape[0]),
            "ms_per_prompt_batch": round(step_ms, 4),
            "prefill_attention_ms": round(attn_ms, 4), "kv_append_ms": round(app_ms, 4),
            "algorithmic_tflop": round(fl / 1e12, 4),
            "prefill_tflops": round(fl / (attn_ms * 1e-3) / 1e12, 1),
            "frac_of_fp16_tensor_peak": round(fl / (attn_ms * 1e-3) / 1e12 / tensor_peak, 4),
            "kv_split_workspace_bytes": pb.ws_bytes}
    if pb.ws_bytes:
        del pb
        plain = PrefillBench(p, device, split=False)
        _, attn0, _ = plain.run(steps, warmup)
        line["unsplit_prefill_attention_ms"] = round(attn0, 4)
        line["unsplit_prefill_tflops"] = round(fl / (attn0 * 1e-3) / 1e12, 1)
    return line


# ---- full-pool ragged decode across 40 layers ------------------------------------

def fullpool_line(device, steps, warmup, hbm_peak, layers=40, schedule="chunked"):
    """One decode step through all layers' attention (per layer: append the new
    token, split-KV attention, merge) over 32 GiB of pools, replayed as one
    CUDA graph."""
    import torch
    from fp8_paged_kv_append_gb300 import workloads
    from fp8_paged_kv_append_gb300.decode_step import MultiLayerDecode
    lay = workloads.fullpool_layout(seed=4)
    P, B = lay.num_pages, len(lay.seq_lens)
    pools = [workloads.device_layer_pool(1000 + l, P, device) for l in range(layers)]
    g = torch.Generator(device=device)
    g.manual_seed(44)
    qs = [torch.randn((B, 40, 128), generator=g, device=device, dtype=torch.float16)
          for _ in range(layers)]
    kn = [torch.randn((B, 10, 128), generator=g, device=device, dtype=torch.float16)
          for _ in range(layers)]
    vn = [torch.randn((B, 10, 128), generator=g, device=device, dtype=torch.float16)
          for _ in range(layers)]
    L = lay.seq_lens.astype(np.int64)
    slots = lay.block_table[np.arange(B), (L - 1) // 16].astype(np.int64) * 16 + (L - 1) % 16
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    step = MultiLayerDecode([p[0] for p in pools], [p[1] for p in pools], [p[2] for p in pools],
                            td(lay.block_table), td(lay.seq_lens), td(slots), int(L.max()), 40,
                            split_chunk=512, schedule=schedule)
    chosen = step.schedule
    outs = [torch.empty((B, 40, 128), dtype=torch.float16, device=device) for _ in range(layers)]
    lses = [torch.empty((B, 40), dtype=torch.float32, device=device) for _ in range(layers)]
    step.capture(qs, kn, vn, outs, lses)
    for _ in range(warmup):
        step.replay()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        step.replay()
    t1.record()
    torch.cuda.synchronize(device)
    if step.check() != 0:
        raise RuntimeError("device error flag raised during the full-pool benchmark")
    ms = t0.elapsed_time(t1) / steps
    kvb = layers * int(L.sum()) * 10 * 128 * 3
    del pools, step
    torch.cuda.empty_cache()
    gib = layers * P * 10 * 16 * 128 * 3 / 2 ** 30
    return {"workload": f"full pool: {layers} layers x {P} pages (223,696 slots, {gib:.1f} GiB), batch "
                        f"{B}, seq_lens {int(L.min())}..{int(L.max())} (sum {int(L.sum())}, "
                        f"{lay.draws} draw(s)), "
                        + {"chunked": "split 512", "fused": "split 512 with the append folded in",
                           "balanced": "load-balanced split",
                           "balanced_fused": "load-balanced split with the append folded in"}
                        [chosen] + (" (chosen by the tiles-per-CTA rule)" if schedule == "auto"
                                    else "") + ", one CUDA graph per step",
            "ms_per_step": round(ms, 4), "us_per_layer_step": round(ms * 1e3 / layers, 2),
            "kv_bytes_per_step": kvb, "value": round(kvb / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "frac_of_hbm_peak": round(kvb / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "gpu_launches_per_step": (2 if chosen in ("fused", "balanced_fused") else 3) * layers}


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


def run_cpu_baseline(w, chunk, budget_s=12.0):
    """Time the oracle, as it stands, on a bounded sample of the workload."""
    import oracle
    ncores = os.cpu_count() or 1
    okc = np.zeros((w.num_pages, w.num_kv_heads, 16, w.head_dim), np.float16)
    ovc = np.zeros((w.num_pages, w.num_kv_heads, 16, w.head_dim), np.uint8)
    oracle.kv_append(w.k_tok, w.v_tok, w.slot_mapping, w.v_scale, okc, ovc)
    n = min(w.batch, 4)
    sample = np.arange(n)
    t0 = time.perf_counter()
    bytes_done = 0
    passes = 0
    while True:
        bytes_done += oracle_decode_pass(w, okc, ovc, chunk, sample, ncores)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s or passes >= 5000:
            break
    return {"value": round(bytes_done / el / 1e9, 4), "unit": "GB/s", "cores": ncores,
            "kind": "oracle",
            "sample": f"{passes} oracle decode steps (append + split partials + merge) over "
                      f"sequences 0..{n - 1} of the workload, {el:.1f} s wall"}


# ---- main ---------------------------------------------------------------------------

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
    else:
        sched = f"split-KV chunks of {chunk} tokens, LSE merge"
    if mode in ("fused", "balanced_fused"):
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
}


def decode_line(w, label, chunk, mode, device, steps, hbm_peak):
    """Secondary decode line: one workload, one schedule."""
    import torch
    b = DecodeBench(w, device, split_chunk=chunk, mode=mode)
    ms, seg = b.run(steps, 3)
    split_name, merge_name, _ = KERNEL_NAMES[mode]
    kvb = kv_bytes(w)
    s_us = float(np.mean(seg[:, 1])) * 1e3
    sb = kvb + w.batch * w.num_qo_heads * w.head_dim * 2
    out = {"value": round(kvb / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "us_per_layer_step": round(ms * 1e3, 2),
           "kernel_us": {"kv_append": round(float(np.mean(seg[:, 0])) * 1e3, 2),
                         split_name: round(s_us, 2),
                         merge_name: round(float(np.mean(seg[:, 2])) * 1e3, 2)},
           "split_frac_of_hbm_peak": round(sb / (s_us * 1e-6) / 1e9 / hbm_peak, 4),
           "step_frac_of_hbm_peak": round(kvb / (ms * 1e-3) / 1e9 / hbm_peak, 4),
           "config": config_of(w, label, chunk, b.R, mode)}
    if mode in ("fused", "balanced_fused"):
        del out["kernel_us"]["kv_append"]
        out["step"] = "append fused into the split kernel, then merge (2 launches)"
    del b
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="1k", choices=["1k", "8k", "prefill", "fullpool"])
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the secondary 8K/b16 line inside the JSON")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--decode", default=DEFAULT_DECODE, choices=list(MODES),
                    help="decode schedule of the main line")
    ap.add_argument("--split-chunk", type=int, default=0,
                    help="tokens per split-KV chunk of the main workload (0: its default)")
    ap.add_argument("--layers", type=int, default=40,
                    help="layers of the full-pool workload (fewer for profiling captures)")
    args = ap.parse_args()
    rank, world, local_rank = dist_env()

    if args.impl == "reference":
        return main_reference(args, rank, world)
    if args.workload == "prefill":
        return main_prefill(args)
    if args.workload == "fullpool":
        import torch
        from fp8_paged_kv_append_gb300 import k16v8 as K
        torch.cuda.set_device(0)
        K.load_library()
        print(json.dumps({f"fullpool_{args.layers}_layers": fullpool_line(
            torch.device("cuda", 0), args.steps, max(3, args.warmup), load_peaks()[0],
            layers=args.layers, schedule=args.decode)}))
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    from fp8_paged_kv_append_gb300 import k16v8 as K
    K.load_library()

    # Replicas only: every rank runs the same seeded workload on its own GPU.
    w, label, chunk = make_workload(args.workload)
    if args.split_chunk:
        chunk = args.split_chunk
    bench = DecodeBench(w, device, split_chunk=chunk, mode=args.decode)
    clocks = ClockSampler(local_rank).start()
    ms, seg = bench.run(args.steps, max(args.warmup, 3))
    clk = clocks.stop()
    e2e_ms, h2d, d2h = bench.run_e2e(max(10, args.steps // 2), 3)
    kvb = kv_bytes(w)
    t_ms, units = aggregate(ms, kvb)
    te_ms, _ = aggregate(e2e_ms, kvb)

    hbm_peak, _, peak_kind = load_peaks()
    B, hq, d = w.q.shape
    split_us = float(np.mean(seg[:, 1])) * 1e3
    split_bytes = kvb + B * hq * d * 2
    achieved = split_bytes / (split_us * 1e-6) / 1e9
    traffic = traffic_from_profiles(args.decode) if args.workload == "1k" else None
    split_name, merge_name, kernel_name = KERNEL_NAMES[args.decode]
    line = {
        "metric": METRIC, "value": round(units / (t_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(t_ms, 5), "us_per_layer_step": round(t_ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) Q/K/V, E4M3 V with per-head amax/448 scales)",
        "config": config_of(w, label, chunk, bench.R, args.decode),
        "kernel_us": {"kv_append": round(float(np.mean(seg[:, 0])) * 1e3, 2),
                      split_name: round(split_us, 2),
                      merge_name: round(float(np.mean(seg[:, 2])) * 1e3, 2)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": traffic, "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "kernel": kernel_name,
                     "algorithmic_bytes_per_launch": split_bytes},
        "e2e": {"value": round(units / (te_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(te_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": (2 if args.decode in ("fused", "balanced_fused") else 3) * args.steps,
        "clocks": clk,
    }
    if args.decode in ("fused", "balanced_fused"):
        del line["kernel_us"]["kv_append"]
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = run_cpu_baseline(w, chunk, args.cpu_budget)
    if not args.no_extra and args.workload == "1k":
        from fp8_paged_kv_append_gb300 import workloads
        del bench
        torch.cuda.empty_cache()
        n2 = max(10, args.steps // 2)
        w8, label8, chunk8 = make_workload("8k")
        wls = (("decode_1k_b32", (w, label, chunk)), ("decode_8k_b16", (w8, label8, chunk8)))
        line["extra"] = {
            "decode_8k_b16": decode_line(w8, label8, chunk8, args.decode, device, n2, hbm_peak)}
        for m in MODES:
            if m != args.decode:
                for name, (wf, lf, cf) in wls:
                    line["extra"][f"{name}_{SUFFIX[m]}"] = decode_line(wf, lf, cf, m, device,
                                                                       n2, hbm_peak)
        for name, (wf, _, cf) in wls:
            torch.cuda.empty_cache()
            ctl = fp16_control_line(wf, device, cf, n2, 3, hbm_peak)
            ref = line["extra"].get(f"{name}_chunked")
            k16 = ref["us_per_layer_step"] if ref else (
                line["us_per_layer_step"] if name == "decode_1k_b32" else
                line["extra"]["decode_8k_b16"]["us_per_layer_step"])
            ctl["k16v8_speedup_over_fp16_kv"] = round(ctl["us_per_layer_step"] / k16, 3)
            ctl["compared_with"] = "K16/V8 with the same chunked split"
            line["extra"][f"{name}_fp16_kv_control"] = ctl
        torch.cuda.empty_cache()
        line["extra"]["fullpool_40_layers"] = fullpool_line(device, 10, 3, hbm_peak,
                                                            schedule="auto")
        for m in MODES:
            line["extra"][f"fullpool_40_layers_{SUFFIX[m]}"] = fullpool_line(
                device, 10, 3, hbm_peak, schedule=m)
        _, tpeak, tkind = load_peaks()
        torch.cuda.empty_cache()
        line["extra"]["prefill"] = {
            "peak_tflops": tpeak, "peak_kind": f"{tkind} dense bf16 (fp16 has the same nominal rate)",
            "8x1024": prefill_line(workloads.prefill_8x1k(), device, 10, 3, tpeak),
            "1x8192_in_8_chunks": prefill_line(workloads.prefill_1x8k(), device, 5, 2, tpeak)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main_prefill(args):
    """Prefill-only line (for profiling the tensor-core kernel)."""
    import torch
    from fp8_paged_kv_append_gb300 import k16v8 as K
    from fp8_paged_kv_append_gb300 import workloads
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    K.load_library()
    _, tpeak, tkind = load_peaks()
    res = {"8x1024": prefill_line(workloads.prefill_8x1k(), device, args.steps,
                                  max(3, args.warmup), tpeak)}
    if not args.no_extra:
        res["1x8192_in_8_chunks"] = prefill_line(workloads.prefill_1x8k(), device, args.steps,
                                                 max(3, args.warmup), tpeak)
    print(json.dumps({"prefill": res, "peak_tflops": tpeak, "peak_kind": tkind}), flush=True)


def main_reference(args, rank, world):
    """The reference arm: the oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    w, label, chunk = make_workload(args.workload)
    import oracle
    okc = np.zeros((w.num_pages, w.num_kv_heads, 16, w.head_dim), np.float16)
    ovc = np.zeros((w.num_pages, w.num_kv_heads, 16, w.head_dim), np.uint8)
    oracle.kv_append(w.k_tok, w.v_tok, w.slot_mapping, w.v_scale, okc, ovc)
    ncores = os.cpu_count() or 1
    sample = np.arange(min(w.batch, 2))
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
            "impl": "reference", "config": config_of(w, label, chunk, replicas_for(w), args.decode),
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": ncores, "kind": "oracle",
                             "sample": f"each step: sequences 0..{len(sample) - 1} of the "
                                       "workload (append + split partials + merge)"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
