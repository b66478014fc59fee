#!/usr/bin/env python3
"""Benchmark: compressed-KV decode attention GB/s and encode tokens/s on GB300.

One *step* is one decode step of every layer of the workload: per layer the
new token's k, v are appended to the exact ring (flushing 128 tokens into
the compressed pages when the ring is full) and decode attention runs for
all query heads over the compressed history plus the ring.  ``value`` is the
decode-attention throughput in GB/s of algorithmic bytes: compressed records
read (at the default widths 100 B per token-head in the main layout, 1.5 d + 2 B
in the alternate one) + fp16 ring tokens (4 d B per token-head) + fp16 queries
+ fp32 outputs.

Workloads (synthetic inputs from ``synth``; no weights or datasets):
  qwen2.5-7b-b8    28 layers, 28 / 4 heads, d 128, batch 8, 32768 tokens each, shuffled
                   pages (default: the largest single-GPU workload)
  qwen3-0.6b-32k   28 layers, 16 q / 4 KV heads, d 128, batch 1, 32768-token prefix
                   compressed in 128-token flushes, then decode steps
  tiny-1k          1 layer, 16 / 4, d 128, batch 1, 1024 tokens
  alt-d{64,128,256,512}  alternate layout, 8 / 8, batch 4, 65536 tokens, no ring
  qwen2.5-32b-ragged     1 of 64 layers, 40 / 8, d 128, batch 16, lengths U[1024, 131072]
  qwen2.5-7b-b8-v4       the batch-8 workload with 4-bit value codes
  alt-d128-v4 / -v8 / -k4 / -k5 / -k2 / -vonly
                   the d 128 alternate workload with 4- or 8-bit values (K8+V4, q8_0 / q8_0),
                   4-, 5- or 2-bit keys (q4_0 / q5_0 / uint2), or fp16 keys (the V-only cache)

Launch: ``python bench.py [--gpus N --steps K --warmup W --workload NAME]``;
for N > 1 under torchrun, each rank runs the same per-GPU workload (weak
scaling, no data-path collective) and rank 0 prints one JSON line.
``--impl reference`` times the CPU oracle instead (the reference arm).

On one GPU the line also carries ``configs``: every workload of CONFIG_SET
(tiny-1k, qwen3-0.6b-32k, qwen2.5-7b-b8, alt-d64..512, qwen2.5-32b-ragged)
timed a few steps each (--config-steps), with its decode-kernel fraction of
the HBM peak, the back-to-back decode call time and the end-to-end figure;
the Qwen3-0.6B entry adds the encode timed as 128-token ring flushes.  A
workload whose step reads less than twice the L2 size is timed with an L2
flush between steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode-attn compressed-KV GB/s (% of GB300 HBM peak); encode tokens/s"

WORKLOADS = {
    "tiny-1k": dict(layout="main", layers=1, batch=1, hq=16, hkv=4, d=128, ctx=1024, shuffled=False, seed=0),
    "qwen3-0.6b-32k": dict(layout="main", layers=28, batch=1, hq=16, hkv=4, d=128, ctx=32768, shuffled=False, seed=0),
    "qwen2.5-7b-b8": dict(layout="main", layers=28, batch=8, hq=28, hkv=4, d=128, ctx=32768, shuffled=True, seed=0),
    "alt-d64": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=64, ctx=65536, shuffled=False, seed=0),
    "alt-d128": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=128, ctx=65536, shuffled=False, seed=0),
    "alt-d256": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=256, ctx=65536, shuffled=False, seed=0),
    "alt-d512": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=512, ctx=65536, shuffled=False, seed=0),
    "qwen2.5-32b-ragged": dict(layout="main", layers=1, batch=16, hq=40, hkv=8, d=128, ctx=None, lo=1024, hi=131072,
                               shuffled=True, seed=7),
    # the batch-8 geometry with 4-bit value codes (--value-bits 4)
    "qwen2.5-7b-b8-v4": dict(layout="main", layers=28, batch=8, hq=28, hkv=4, d=128, ctx=32768, shuffled=True, seed=0,
                             vbits=4),
    # the alternate layout with 4-bit value indices (8-bit keys + 4-bit values: the K8+V4 mix)
    "alt-d128-v4": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=128, ctx=65536, shuffled=False, seed=0,
                        vbits=4),
    # the alternate layout with 4-bit keys (q4_0 keys + 3-bit values: the guide's low-memory option)
    "alt-d128-k4": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=128, ctx=65536, shuffled=False, seed=0,
                        kbits=4),
    # 5-bit keys (q5_0 keys + 3-bit values: the guide's next step down in memory)
    "alt-d128-k5": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=128, ctx=65536, shuffled=False, seed=0,
                        kbits=5),
    # 2-bit keys (uint2 keys + 3-bit values: the guide's aggressive row)
    "alt-d128-k2": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=128, ctx=65536, shuffled=False, seed=0,
                        kbits=2),
    # 8-bit keys and 8-bit values (q8_0 / q8_0: the widest value format of the guide)
    "alt-d128-v8": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=128, ctx=65536, shuffled=False, seed=0,
                        vbits=8),
    # fp16 keys, 3-bit values (the V-only cache)
    "alt-d128-vonly": dict(layout="alt", layers=1, batch=4, hq=8, hkv=8, d=128, ctx=65536, shuffled=False, seed=0,
                           kbits=16),
}
DEFAULT_WORKLOAD = "qwen2.5-7b-b8"


# ---------------------------------------------------------------------- helpers
def ring_split(length: int):
    if length <= 0:
        return 0, 0
    n_c = 128 * ((length - 1) // 128)
    return n_c, length - n_c


def record_bytes(w) -> int:
    d = w["d"]
    if w["layout"] == "main":
        # key bits (Lloyd-Max index + QJL), value codes, group (scale, min), two norms
        return (w.get("kbits", 3) * d) // 8 + (w.get("vbits", 2) * d) // 8 + d // 8 + 4
    # key codes, block (scale, min), value indices, norm; fp16 keys (16 bits) have no (scale, min)
    kb = w.get("kbits", 8)
    return (kb * d) // 8 + (0 if kb == 16 else 4 * (d // 32)) + (w.get("vbits", 3) * d) // 8 + 2


def step_bytes(w, lengths_after_append):
    """Algorithmic bytes one layer's decode attention moves at the given lengths."""
    rb, d = record_bytes(w), w["d"]
    tot = 0
    for L in lengths_after_append:
        L = int(L)
        if w["layout"] == "main":
            nc, nb = ring_split(L)
        else:
            nc, nb = L, 0
        tot += w["hkv"] * (nc * rb + nb * 4 * d)
    tot += w["batch"] * w["hq"] * d * (2 + 4)
    return int(tot)


def max_over_ranks(value: float, device="cpu") -> float:
    """The largest ``value`` over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank: int, ms_max: float, world: int) -> float:
    """Whole-job throughput: every rank moves ``bytes_per_rank`` (weak scaling) in ``ms_max``."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, local_index: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x for x in vis.split(",") if x.strip()]
        self.gpu = ids[local_index].strip() if local_index < len(ids) else str(local_index)
        self.proc = None
        self.lines = []
        self.stamped = []

    def __enter__(self):
        # The sampler is started and its first sample awaited before the timed region, and the
        # region is bracketed by timestamps: samples from 50 ms before it to 50 ms after it count,
        # and at least one sample after its end is awaited, so a region shorter than the 20 ms
        # sampling period still gets the samples around it.
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.time() + 5.0
            while not self.stamped and time.time() < deadline:
                time.sleep(0.005)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.stamped.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        self.t1 = time.time()
        if self.proc is not None:
            deadline = time.time() + 1.0
            while time.time() < deadline and not any(ts > self.t1 for ts, _ in self.stamped):
                time.sleep(0.005)
            self.lines = [ln for ts, ln in self.stamped if self.t0 - 0.05 <= ts <= self.t1 + 0.05]
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------- GPU arm
class Layer:
    """One layer's context, pool, ring and block table on the device."""

    def __init__(self, tq, torch, w, layer_idx, lengths, max_len, bt_np):
        lay = tq.TQ_LAYOUT_MAIN if w["layout"] == "main" else tq.TQ_LAYOUT_ALT
        self.ctx = tq.Context(lay, w["d"], w["hq"], w["hkv"], w["seed"] + layer_idx,
                              value_bits=w.get("vbits"), key_bits=w.get("kbits"))
        self.ctx.set_decode_path({"auto": tq.TQ_DECODE_AUTO, "mma_sync": tq.TQ_DECODE_MMA_SYNC,
                                  "tcgen05": tq.TQ_DECODE_TCGEN05}[w.get("decode_path", "auto")])
        self.max_blocks = bt_np.shape[1]
        self.bt = torch.from_numpy(bt_np).cuda()
        nblk = bt_np.shape[0] * bt_np.shape[1]
        self.pool = torch.empty((nblk, w["hkv"], self.ctx.page_bytes), dtype=torch.uint8, device="cuda")
        self.ring_k = torch.zeros((w["batch"], w["hkv"], 128, w["d"]), dtype=torch.float16, device="cuda")
        self.ring_v = torch.zeros_like(self.ring_k)
        self.out = None  # a view of the step's [layers, batch, Hq, d] output buffer (build_gpu_state)


def build_gpu_state(tq, torch, w, steps_total):
    bsz, hkv, d = w["batch"], w["hkv"], w["d"]
    if w["ctx"] is None:
        lengths = [int(x) for x in synth.ragged_lengths(w["seed"], bsz, w["lo"], w["hi"])]
    else:
        lengths = [w["ctx"]] * bsz
    max_len = max(lengths) + steps_total + 128 + 64  # room for the end-to-end steps
    max_blocks = (max_len + 15) // 16
    bt_np = synth.block_table(w["seed"], bsz, max_blocks, w["shuffled"])
    # one shared synthetic K/V prefix (layer 0 recipe), reused by every layer with its own tables
    kv_len = ((max(lengths) + 15) // 16) * 16
    if w["layout"] == "main":
        k_np, v_np = synth.kv_main(w["seed"], 1, hkv, kv_len, d)
    else:
        k_np, v_np = synth.kv_alt(w["seed"], 1, hkv, kv_len, d)
    k1 = torch.from_numpy(k_np).cuda()
    v1 = torch.from_numpy(v_np).cuda()
    layers = [Layer(tq, torch, w, li, lengths, max_len, bt_np) for li in range(w["layers"])]
    out_all = torch.empty((w["layers"], bsz, w["hq"], d), dtype=torch.float32, device="cuda")
    for li, lay in enumerate(layers):
        lay.out = out_all[li]
        lay.out_all = out_all
    return lengths, k1, v1, layers


def encode_prefix(tq, torch, w, lengths, k1, v1, layers, timed=True):
    """Compress every sequence's prefix (page-aligned part) and fill the rings; returns (ms, tokens)."""
    bsz = w["batch"]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_tok_total = 0
    torch.cuda.synchronize()
    ev0.record()
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    for lay in layers:
        for b in range(bsz):
            L = lengths[b]
            nc, nb = ring_split(L) if w["layout"] == "main" else (L, 0)
            if nc:
                lay.ctx.encode_flush(k1, v1, start, lay.bt[b:b + 1], lay.pool, n_tokens=nc)
                n_tok_total += nc
            if nb:
                lay.ring_k[b, :, :nb] = k1[0, :, nc:nc + nb]
                lay.ring_v[b, :, :nb] = v1[0, :, nc:nc + nb]
    ev1.record()
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1), n_tok_total


L2_BYTES = 129 * 2**20  # GB300 L2


class L2Flush:
    """Writes a buffer four times the L2 size: called between timed steps whose inputs fit in L2."""

    def __init__(self, torch):
        self.buf = torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.buf.fill_(1.0)


def fp32_peak_tflops():
    """FP32 FFMA peak from the unit counts: 152 SMs x 128 FP32 lanes x 2 FLOP x the measured maximum
    SM clock (MEASURED_PEAKS.json sm_max_mhz, else the 2070 MHz nominal)."""
    mhz = 2070.0
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def encode_io_bytes(w):
    """Algorithmic bytes per token-head of the encode: fp16 k and v in, the compressed record out."""
    return 4 * w["d"] + record_bytes(w)


def encode_fp32_flop(w):
    """Algorithmic FP32 work per token-head of the main encode: the dense QJL projection S r (d x m
    FFMA, m = d); the rotation, assignment and value quantisation add ~10 d operations."""
    return 2 * w["d"] * w["d"] + 10 * w["d"] if w["layout"] == "main" else 12 * w["d"]


def encode_fracs(w, token_heads_per_s):
    hbm, _ = measured_peaks()
    gbs = token_heads_per_s * encode_io_bytes(w) / 1e9
    tflops = token_heads_per_s * encode_fp32_flop(w) / 1e12
    return {"gbs": gbs, "frac_hbm": gbs / hbm, "tflops_fp32_equiv": tflops, "frac_fp32": tflops / fp32_peak_tflops(),
            "io_bytes_per_token_head": encode_io_bytes(w), "fp32_flop_per_token_head": encode_fp32_flop(w)}


def encode_throughput(tq, torch, w, layers, k1, v1, flush, reps=3):
    """tq_encode_flush alone: (a) one call over a page-aligned prefix of up to 32768 tokens, and
    (b) the same prefix as consecutive 128-token flushes, one call each (the ring-flush size of
    the decode step), with an L2 flush before each repetition."""
    n = min(k1.shape[2], 32768) // 128 * 128
    kb, vb = k1[:, :, :n].contiguous(), v1[:, :, :n].contiguous()
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty((n // 16 + 1, w["hkv"], layers[0].ctx.page_bytes), dtype=torch.uint8, device="cuda")
    bt = torch.arange(n // 16 + 1, dtype=torch.int32, device="cuda")[None, :]
    ctx = layers[0].ctx
    for _ in range(2):
        ctx.encode_flush(kb, vb, start, bt, scratch)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ms_one = 0.0
    for _ in range(reps):
        flush()
        e0.record()
        ctx.encode_flush(kb, vb, start, bt, scratch)
        e1.record()
        torch.cuda.synchronize()
        ms_one += e0.elapsed_time(e1)
    ms_one /= reps
    # 128-token flushes: the prefix cut into ring buffers of 128 tokens ([1, Hkv, 128, d] each, as the
    # decode step flushes them), start positions 0, 128, ... (captured in one graph)
    nf = n // 128
    rings_k = kb.view(1, w["hkv"], nf, 128, w["d"]).permute(2, 0, 1, 3, 4).contiguous()
    rings_v = vb.view(1, w["hkv"], nf, 128, w["d"]).permute(2, 0, 1, 3, 4).contiguous()
    slices_k = [rings_k[i] for i in range(nf)]
    slices_v = [rings_v[i] for i in range(nf)]
    starts = torch.arange(0, n, 128, dtype=torch.int32, device="cuda").view(nf, 1)

    def flushes():
        for i in range(nf):
            ctx.encode_flush(slices_k[i], slices_v[i], starts[i], bt, scratch, n_tokens=128)
    flushes()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        flushes()
    ms_fl = 0.0
    for _ in range(reps):
        flush()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_fl += e0.elapsed_time(e1)
    ms_fl /= reps
    del g
    th_one = n * w["hkv"] / (ms_one * 1e-3)
    th_fl = n * w["hkv"] / (ms_fl * 1e-3)
    return {"tokens_per_call": n, "ms_per_call": ms_one, "token_heads_per_s": th_one, "tokens_per_s": n / (ms_one * 1e-3),
            **encode_fracs(w, th_one),
            "flush128": {"calls": nf, "us_per_flush": ms_fl * 1e3 / nf, "token_heads_per_s": th_fl,
                         "tokens_per_s": n / (ms_fl * 1e-3), **encode_fracs(w, th_fl)}}


def dequant_throughput(torch, w, lay, lengths, reps=3, cap=32768):
    """Time tq_dequantize (prefill materialisation) of one layer: every sequence's compressed prefix
    (at most ``cap`` tokens each) read back as dense fp16 K and V."""
    bsz, hkv, d = w["batch"], w["hkv"], w["d"]
    n_c = [min(ring_split(L)[0] if w["layout"] == "main" else L, cap) // 16 * 16 for L in lengths]
    max_tokens = max(max(n_c), 16)
    ncd = torch.tensor(n_c, dtype=torch.int32, device="cuda")
    k_out = torch.empty((bsz, hkv, max_tokens, d), dtype=torch.float16, device="cuda")
    v_out = torch.empty_like(k_out)
    for _ in range(2):
        lay.ctx.dequantize(lay.pool, lay.bt, ncd, k_out, v_out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        lay.ctx.dequantize(lay.pool, lay.bt, ncd, k_out, v_out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    th = sum(n_c) * hkv
    nbytes = th * (record_bytes(w) + 4 * d)  # compressed record in, fp16 k and v out
    del k_out, v_out
    return {"token_heads_per_s": th / (ms * 1e-3), "gbs": nbytes / (ms * 1e-3) / 1e9, "ms_per_call": ms,
            "tokens_per_call": sum(n_c), "bytes_per_call": nbytes}


class StepGraph:
    """One decode step of every layer, captured once as a CUDA graph and replayed.

    Per-step state lives in fixed device buffers: ``pos`` (index of the token
    being appended), and the compressed / ring counts derived from it.  The
    graph appends the token in every layer (flushing a full ring), derives the
    counts, runs decode attention in every layer and advances ``pos``.
    """

    def __init__(self, torch, w, layers, lengths, max_ctx, ws, q, kn, vn, out_host=None, in_host=None):
        self.torch = torch
        self.w, self.layers, self.max_ctx, self.ws = w, layers, max_ctx, ws
        self.main = w["layout"] == "main"
        self.pos = torch.tensor(lengths, dtype=torch.int32, device="cuda")
        self.nc = torch.tensor(lengths, dtype=torch.int32, device="cuda")
        self.nb = torch.zeros_like(self.nc)
        self.q, self.kn, self.vn = q, kn, vn
        self.out_host, self.in_host = out_host, in_host
        self.graph = None

    def body(self):
        torch = self.torch
        if self.in_host is not None:
            qh, kh, vh = self.in_host
            self.q.copy_(qh, non_blocking=True)
            self.kn.copy_(kh, non_blocking=True)
            self.vn.copy_(vh, non_blocking=True)
        if self.main:
            for li, lay in enumerate(self.layers):
                lay.ctx.append_token(self.kn[li], self.vn[li], self.pos, lay.ring_k, lay.ring_v, lay.bt, lay.pool)
            t = self.pos + 1
            self.nc.copy_(torch.div(t - 1, 128, rounding_mode="floor") * 128)
            self.nb.copy_(t - self.nc)
        for li, lay in enumerate(self.layers):
            lay.ctx.decode_attention(self.q[li], lay.pool, lay.bt, self.nc, lay.ring_k if self.main else None,
                                     lay.ring_v if self.main else None, self.nb if self.main else None,
                                     self.max_ctx, lay.out, self.ws)

        if self.out_host is not None:  # every layer's output in one copy
            self.out_host.copy_(self.layers[0].out_all, non_blocking=True)
        if self.main:
            self.pos.add_(1)

    def capture(self):
        """Capture the step; returns the graph (also kept as ``self.graph``).  Capturing again
        (e.g. with the library's profiling events switched on) makes a second graph over the same
        state buffers."""
        torch = self.torch
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            self.body()
        self.graph = graph
        return graph

    def replay(self):
        self.graph.replay()


def timed_replays(torch, fn, n, flush=None):
    """Total ms of n calls of fn: one event pair around all of them, or, with an L2 flush between
    calls (inputs smaller than L2), one event pair per call with the flush outside."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if flush is None:
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)
    tot = 0.0
    for _ in range(n):
        flush()
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1)
    return tot


def run_gpu(tq, torch, w, rank, world, steps, warmup, extras=True, sample_clocks=True):
    """One workload on this rank's GPU: the timed decode steps, the per-launch decode-kernel times,
    the back-to-back decode calls, the end-to-end step through host buffers, and (extras) the
    encode and dequantise timings."""
    prof_steps = 3  # replays of the profiled graph (roofline events)
    steps_total = warmup + steps + prof_steps + 64  # + end-to-end steps
    lengths, k1, v1, layers = build_gpu_state(tq, torch, w, steps_total)
    flush_op = L2Flush(torch)
    encode_prefix(tq, torch, w, lengths, k1, v1, layers)
    enc = encode_throughput(tq, torch, w, layers, k1, v1, flush_op) if extras else None
    deq = dequant_throughput(torch, w, layers[0], lengths) if extras else None
    bsz, hq, hkv, d, nl = w["batch"], w["hq"], w["hkv"], w["d"], w["layers"]
    main = w["layout"] == "main"
    g = torch.Generator(device="cuda")
    g.manual_seed(1234 + rank)
    q = torch.randn((nl, bsz, hq, d), generator=g, device="cuda").half()
    kn = torch.randn((nl, bsz, hkv, d), generator=g, device="cuda").half()
    vn = torch.randn((nl, bsz, hkv, d), generator=g, device="cuda").half()
    max_ctx = int(((max(lengths) + steps_total + 15) // 16) * 16)
    ws = torch.empty(layers[0].ctx.workspace_size(bsz, max_ctx), dtype=torch.uint8, device="cuda")

    def bytes_at(pos_list):
        after = [p + 1 for p in pos_list] if main else list(pos_list)
        return nl * step_bytes(w, after)

    # a step whose inputs fit in L2 is timed with an L2 flush between steps
    small = bytes_at(lengths) < 2 * L2_BYTES
    flush = flush_op if small else None
    sg = StepGraph(torch, w, layers, lengths, max_ctx, ws, q, kn, vn)
    pos = list(lengths)
    for _ in range(warmup):  # eager warm-up steps (same calls as the graph)
        sg.body()
        if main:
            pos = [p + 1 for p in pos]
    torch.cuda.synchronize()
    launches0 = sum(l.ctx.launch_count for l in layers)
    timed_graph = sg.capture()  # the timed step: no profiling events inside
    launches_per_step = sum(l.ctx.launch_count for l in layers) - launches0
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    timed_bytes = 0
    if sample_clocks:
        with ClockSampler(torch.cuda.current_device()) as clk:
            ms = timed_replays(torch, sg.replay, steps, flush)
        clocks = clk.summary()
    else:
        ms = timed_replays(torch, sg.replay, steps, flush)
        clocks = None
    for _ in range(steps):
        timed_bytes += bytes_at(pos)
        if main:
            pos = [p + 1 for p in pos]
    # the same step captured again with the library's CUDA events around every decode and merge
    # launch; a few replays after the timed region give the per-kernel durations
    for lay in layers:
        lay.ctx.profile_begin()
    prof_graph = sg.capture()
    for _ in range(prof_steps):
        if flush:
            flush()
        prof_graph.replay()
        if main:
            pos = [p + 1 for p in pos]
    torch.cuda.synchronize()
    prof = [lay.ctx.profile_end() for lay in layers]  # events of the last replay
    del timed_graph, prof_graph
    # The same decode calls (decode + merge kernels of every layer, at the last step's counts)
    # captured back to back with no events between them, timed by one event pair: the per-launch
    # event pairs above each add the front end's drain and launch latency to the kernel they
    # bracket, which this figure does not contain.
    def decode_calls():
        for li, lay in enumerate(layers):
            lay.ctx.decode_attention(q[li], lay.pool, lay.bt, sg.nc, lay.ring_k if main else None,
                                     lay.ring_v if main else None, sg.nb if main else None, max_ctx, lay.out, ws)
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph, capture_error_mode="thread_local"):
        decode_calls()
    dgraph.replay()
    torch.cuda.synchronize()
    call_us = timed_replays(torch, dgraph.replay, prof_steps, flush) / (prof_steps * nl) * 1e3
    del dgraph
    if world > 1:
        ms = max_over_ranks(ms, device="cuda")
        torch.distributed.barrier()
    value = aggregate_gbs(timed_bytes, ms, world)

    # dominant kernel: the fused decode kernel, timed by the library's CUDA events captured into
    # the profiled step graph (its last replay)
    dec_ms = sum(p["decode_ms"] for p in prof)
    dec_n = sum(p["decode_launches"] for p in prof)
    kernel = prof[-1]["decode_kernel"]
    peak, peak_kind = measured_peaks()
    last_pos = [p - 1 for p in pos] if main else pos
    per_launch_bytes = bytes_at(last_pos) / nl
    achieved = per_launch_bytes / (dec_ms / max(dec_n, 1) * 1e-3) / 1e9 if dec_n else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak if achieved else None,
                "traffic": ncu_traffic(w["name"], kernel),
                "kernel": kernel,
                "peak_source": peak_kind, "launches": dec_n, "avg_launch_us": dec_ms / max(dec_n, 1) * 1e3,
                "merge_us_per_launch": sum(p["merge_ms"] for p in prof) / max(dec_n, 1) * 1e3,
                "decode_call_us_back_to_back": call_us,
                "bytes_per_launch": per_launch_bytes}

    e2e = run_e2e(torch, w, layers, pos, max_ctx, ws, q, kn, vn, bytes_at, flush)
    res = {
        "value": value, "ms_per_step": ms / steps, "roofline": roofline, "encode": enc, "dequantize": deq, "e2e": e2e,
        "gpu_launches": int(launches_per_step * steps), "clocks": clocks, "lengths": lengths,
        "l2": ("L2 flushed between timed steps (step inputs below 2x L2)" if small
               else "inputs larger than L2 (every step reads all layers' pools)"),
    }
    del layers, k1, v1, q, kn, vn, ws, sg, flush_op
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_e2e(torch, w, layers, pos, max_ctx, ws, q, kn, vn, bytes_at, flush=None, steps=16):
    """Same decode step through the same C ABI, with the step's q, k, v copied in from pinned host
    memory and every layer's output copied back to pinned host memory inside the timed region
    (captured in the step graph)."""
    rng = np.random.default_rng(5)
    qh = torch.from_numpy(rng.standard_normal(tuple(q.shape)).astype(np.float16)).pin_memory()
    kh = torch.from_numpy(rng.standard_normal(tuple(kn.shape)).astype(np.float16)).pin_memory()
    vh = torch.from_numpy(rng.standard_normal(tuple(vn.shape)).astype(np.float16)).pin_memory()
    out_h = torch.empty(tuple(layers[0].out_all.shape), dtype=torch.float32).pin_memory()
    sg = StepGraph(torch, w, layers, pos, max_ctx, ws, q, kn, vn, out_host=out_h, in_host=(qh, kh, vh))
    sg.capture()
    torch.cuda.synchronize()
    ms = timed_replays(torch, sg.replay, steps, flush)
    tot = 0
    main = w["layout"] == "main"
    p = list(pos)
    for _ in range(steps):
        tot += bytes_at(p)
        if main:
            p = [x + 1 for x in p]
    h2d = (qh.numel() + kh.numel() + vh.numel()) * 2
    d2h = out_h.numel() * 4
    return {"value": tot / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps}


def ncu_traffic(workload, kernel):
    """DRAM bytes (read + write) of one launch of `kernel` on `workload`, from the ncu capture listed
    in profiles/dram_traffic.json, if that capture was taken on the current source of the files the
    kernel is built from (sha256 of each); otherwise None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not kernel or not os.path.exists(path):
        return None
    import hashlib

    with open(path) as f:
        entry = json.load(f).get(workload)
    if not entry or entry.get("kernel") != kernel:
        return None
    for src, digest in entry.get("sources", {}).items():
        p = os.path.join(ROOT, "kv_cache_quantization_tq_gb300", "csrc", src)
        if not os.path.exists(p):
            return None
        with open(p, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return int(entry["dram_bytes"])


# ---------------------------------------------------------------------- CPU oracle arm
def oracle_layer_step(w, seed, sample_len):
    """Build one oracle-encoded (sequence, all KV heads) sample and return a closure timing its decode."""
    from oracle import attention, cache, codebook, layout, rng

    d, hkv, hq = w["d"], w["hkv"], w["hq"]
    L = sample_len
    if w["layout"] == "main":
        nc, nb = ring_split(L)
        c, _ = codebook.lloyd_max(d, 2)
        sg, sk = rng.signs(seed, d), rng.gaussian_matrix(seed, d, d)
        k, v = synth.kv_main(seed, 1, hkv, L, d)
        bt = np.arange((L + 15) // 16, dtype=np.int32)[None, :]
        pool = np.zeros((bt.shape[1], hkv, layout.main_tile_bytes(d, w.get("vbits", 2))), np.uint8)
        cache.encode_main_range(pool, bt, 0, k[:, :, :nc], v[:, :, :nc], sg, c, sk)
        ring_k = np.zeros((1, hkv, 128, d), np.float16)
        ring_v = np.zeros_like(ring_k)
        ring_k[0, :, :nb] = k[0, :, nc:nc + nb]
        ring_v[0, :, :nb] = v[0, :, nc:nc + nb]
        q = synth.queries(seed, 1, hq, d)

        def run():
            attention.decode_main(q, pool, bt, np.array([nc]), ring_k, ring_v, np.array([nb]), sg, c, sk, hkv)
        nbytes = hkv * (nc * record_bytes(w) + nb * 4 * d) + hq * d * 6
    else:
        vb = w.get("vbits", 3)
        c3, _ = codebook.lloyd_max(d, vb)
        sg = rng.signs(seed, d)
        k, v = synth.kv_alt(seed, 1, hkv, L, d)
        bt = np.arange(L // 16, dtype=np.int32)[None, :]
        pool = np.zeros((bt.shape[1], hkv, layout.alt_tile_bytes(d, vb, w.get("kbits", 8))), np.uint8)
        cache.encode_alt_range(pool, bt, 0, k, v, sg, c3)
        q = synth.queries(seed, 1, hq, d)

        def run():
            attention.decode_alt(q, pool, bt, np.array([L]), None, None, None, sg, c3, hkv)
        nbytes = hkv * L * record_bytes(w) + hq * d * 6
    return run, nbytes


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info

        info = threadpool_info()
        if info:
            return max(int(i.get("num_threads", 1)) for i in info)
    except Exception:
        pass
    return os.cpu_count() or 1


def run_oracle(w, reps, sample_len, budget_s=10.0):
    """Time the oracle decode of one sample; at most ``reps`` runs or ``budget_s`` seconds."""
    run, nbytes = oracle_layer_step(w, w["seed"], sample_len)
    run()  # warm
    t0 = time.perf_counter()
    n = 0
    while n < reps and (n == 0 or time.perf_counter() - t0 < budget_s):
        run()
        n += 1
    dt = (time.perf_counter() - t0) / n
    return nbytes / dt / 1e9, dt, nbytes, n


def oracle_one_thread(workload: str):
    """GB/s of the oracle arm re-run in a child process with one BLAS / OpenMP thread (None if the
    child fails): the single-core figure beside the all-cores one."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", workload,
           "--steps", "1", "--warmup", "0"]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=120, env=env)
        for line in r.stdout.splitlines():
            if line.startswith("{"):
                return float(json.loads(line)["value"])
    except (OSError, subprocess.SubprocessError, ValueError, KeyError):
        pass
    return None


def oracle_sample_len(w):
    base = w["ctx"] if w["ctx"] is not None else 32768
    return int(min(base, 32768 if w["layout"] == "main" else 16384))


# ---------------------------------------------------------------------- main
CONFIG_SET = ["tiny-1k", "qwen3-0.6b-32k", "qwen2.5-7b-b8", "alt-d64", "alt-d128", "alt-d256", "alt-d512",
              "qwen2.5-32b-ragged"]


def config_summary(res, peak):
    r = res["roofline"]
    out = {"value": res["value"], "unit": "GB/s", "frac_of_hbm_peak": res["value"] / peak,
           "ms_per_step": res["ms_per_step"], "decode_kernel": r["kernel"], "decode_kernel_gbs": r["achieved"],
           "decode_kernel_frac": r["frac"], "decode_kernel_avg_launch_us": r["avg_launch_us"],
           "decode_call_us_back_to_back": r["decode_call_us_back_to_back"], "e2e_gbs": res["e2e"]["value"],
           "l2": res["l2"]}
    if res.get("encode"):
        out["encode"] = res["encode"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload block of the other configs")
    ap.add_argument("--config-steps", type=int, default=10, help="timed steps of each workload in that block")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (small profiling runs)")
    ap.add_argument("--decode-path", default="auto", choices=["auto", "mma_sync", "tcgen05"],
                    help="main-layout decode kernels at head_dim 128 (tq_set_decode_path)")
    args = ap.parse_args()

    def workload(name):
        w = dict(WORKLOADS[name])
        w["name"] = name
        if args.layers:
            w["layers"] = args.layers
        w["decode_path"] = args.decode_path
        return w

    w = workload(args.workload)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    config = {"workload": args.workload, "layout": w["layout"], "layers": w["layers"], "batch": w["batch"],
              "q_heads": w["hq"], "kv_heads": w["hkv"], "head_dim": w["d"],
              "context": w["ctx"] if w["ctx"] is not None else f"U[{w['lo']},{w['hi']}]"}
    config["value_bits"] = w.get("vbits", 2 if w["layout"] == "main" else 3)
    config["key_bits"] = w.get("kbits", 3 if w["layout"] == "main" else 8)
    config["decode_path"] = args.decode_path

    if args.impl == "reference":
        if rank != 0:
            return
        sample_len = oracle_sample_len(w)
        for _ in range(args.warmup):
            run_oracle(w, 1, sample_len, budget_s=0)
        val, dt, nbytes, reps = run_oracle(w, max(1, args.steps), sample_len, budget_s=60.0)
        sample = f"oracle decode of one sequence x {w['hkv']} KV heads at {sample_len} tokens per step"
        config["l2"] = "host oracle (CPU)"
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
                "steps": reps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    from kv_cache_quantization_tq_gb300.build import build

    if rank == 0 or world == 1:
        build()
    if world > 1:
        torch.distributed.barrier()
    import kv_cache_quantization_tq_gb300 as tq

    res = run_gpu(tq, torch, w, rank, world, args.steps, args.warmup)
    config["l2"] = res["l2"]
    peak, _ = measured_peaks()
    configs = None
    if world == 1 and not args.no_configs:
        # every other workload of the set, a few steps each, on the same GPU (single-GPU runs only)
        configs = {}
        for name in CONFIG_SET:
            if name == args.workload:
                continue
            r = run_gpu(tq, torch, workload(name), rank, world, args.config_steps, 3,
                        extras=(name == "qwen3-0.6b-32k"), sample_clocks=False)
            configs[name] = config_summary(r, peak)
        configs[args.workload] = config_summary(res, peak)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline:
        sample_len = oracle_sample_len(w)
        val, dt, nbytes, reps = run_oracle(w, 20, sample_len, budget_s=10.0)
        cpu = {"value": val, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{reps} oracle decodes of one sequence x {w['hkv']} KV heads at {sample_len} tokens "
                         f"({nbytes / 1e6:.1f} MB of records each), {dt:.2f} s each",
               "value_one_thread": oracle_one_thread(args.workload)}
    line = {
        "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
        "frac_of_hbm_peak": res["value"] / world / peak,
        "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"], "gpu_launches": res["gpu_launches"],
        "clocks": res["clocks"], "encode": res["encode"], "dequantize": res["dequantize"], "configs": configs,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
