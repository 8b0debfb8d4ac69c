"""Benchmark of the paged KV cache decode step on GB300.

Workload (one layer): GQA 32 query / 8 KV heads, head_dim 128, block_size 16,
fp16 K/V, 256 sequences with context lengths uniform in [512, 4096] (seeded),
blocks scattered over a pool sized 1.1x what they need.  One step = the whole
decode path for one new token per sequence:

  a1  host: slots of the new tokens (device-timed runs use fixed slots)
  a2  pkv_write_kv of the 256 new K/V rows into their slots
  a3-a7  pkv_attn_decode over every cached key (split-K decode + merge)

``value`` is KV GB/s: algorithmic bytes of the step (K/V read once per KV
head, q, out, split-K records, tables, the written rows) divided by the
device time of the step with all inputs resident in HBM.  The KV bytes
(~2.4 GB per step) exceed the 129 MB L2, so no flush is needed between steps.
``e2e`` is the same metric through the public API with the step's inputs
copied from pinned host memory and the output copied back inside the timed
region, and the host allocator producing slots and tables every step.

The same JSON line carries ``configs``: every other workload of the scope
table, each in a short block of its own (median of 100 iterations, 50 for the
mixed step), with its roofline, the clocks sampled inside its timed window
and its CPU oracle baseline (all cores and one core): the tiny MHA decode,
the GPT-2-shaped 12-layer step, the long/skewed contexts, the GQA step over an
int8 cache, the GQA step with a 1,024-token sliding window, and the mixed
packed step (prefill chunks + decode rows, then a
width-4 beam split with copy-on-write).  Clocks come from NVML (read only)
sampled every few ms and while the GPU drains the enqueued work.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs an independent replica (the path has no
exchange step); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and tokens/s, 1 GPU"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DECODE_PROFILE = os.path.join(ROOT, "profiles", "attn_decode_gqa32_8_d128_b256.md")
DECODE_SOURCES = ["pagedattention_decode_gb300/csrc/decode.cu", "pagedattention_decode_gb300/csrc/ptx.cuh"]


# ---------------------------------------------------------------------------
# byte accounting
# ---------------------------------------------------------------------------

def kv_bytes_per_token(num_kv_heads: int, head_dim: int, dtype_bytes: int, layers: int = 1) -> int:
    """K and V of one token: 2 x layers x kv_heads x head_dim x dtype_bytes
    ('How to Implement Paged Attention in PyTorch and vLLM', sizing formula)."""
    return 2 * layers * num_kv_heads * head_dim * dtype_bytes


def split_records(lengths, ctas_max: int, sub: int = 16, min_per_cta: int = 4) -> int:
    """Partial records the split-K decode writes (one per cut sequence per CTA
    touching it): the same even split of concatenated 16-token sub-blocks."""
    n = [-(-L // sub) if L > 0 else 0 for L in lengths]
    total = sum(n)
    if total == 0:
        return 0
    if len(lengths) <= 32 and total <= 64 and len(lengths) <= ctas_max:
        return 0  # a CTA per sequence, each taking its sequence whole
    ctas = min(ctas_max, -(-total // min_per_cta))
    recs, start = 0, 0
    for k in n:
        if k:
            c0 = ((start + 1) * ctas - 1) // total
            c1 = ((start + k) * ctas - 1) // total
            if c1 != c0:
                recs += c1 - c0 + 1
        start += k
    return recs


def decode_bytes(lengths, hq, hkv, d, dtype_bytes, out_bytes, ctas_max, num_hg=1):
    kv = sum(lengths) * kv_bytes_per_token(hkv, d, dtype_bytes)
    qb = len(lengths) * hq * d * dtype_bytes
    ob = len(lengths) * hq * d * out_bytes
    recs = split_records(lengths, ctas_max // num_hg) * num_hg
    part = 2 * recs * (hq // num_hg) * (d + 2) * 4
    tables = sum(-(-L // 16) for L in lengths) * 4 + len(lengths) * 4
    return kv + qb + ob + part + tables


def windowed(lengths, window):
    """Keys each sequence attends: all of them, or its last ``window``."""
    return [min(L, window) for L in lengths] if window > 0 else list(lengths)


def write_bytes(tokens, hkv, d, dtype_bytes):
    return 2 * tokens * kv_bytes_per_token(hkv, d, dtype_bytes) + 8 * tokens


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """SM clock, its maximum, board power and the clock-event reasons, read
    (never set) through NVML -- ctypes on libnvidia-ml, every few ms on a
    thread -- with nvidia-smi's polling as the fallback.  Every sample carries
    the host time it was taken; ``summary(t0, t1)`` keeps the samples of one
    timed window, and ``poll_until(event)`` samples from the calling thread
    while the GPU drains the work already enqueued (so a window of a few ms
    still gets samples under load)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clocks-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu: str, period_s: float = 0.004):
        self.gpu = gpu
        self.period = period_s
        self.samples = []  # (host time, sm MHz, max sm MHz, power W, [reasons])
        self.proc = None
        self.nvml = None
        self.stop = threading.Event()
        self.thread = None

    # -- NVML ---------------------------------------------------------------
    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(self.gpu.encode(), ctypes.byref(h)) != 0:
                if not self.gpu.isdigit() or lib.nvmlDeviceGetHandleByIndex_v2(int(self.gpu), ctypes.byref(h)) != 0:
                    return None
            try:
                reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            return None
        c = ctypes
        sm, mx, pw, rs = c.c_uint(), c.c_uint(), c.c_uint(), c.c_ulonglong()

        def read():
            if lib.nvmlDeviceGetClockInfo(h, 1, c.byref(sm)) != 0:  # NVML_CLOCK_SM
                return None
            lib.nvmlDeviceGetMaxClockInfo(h, 1, c.byref(mx))
            p = pw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, c.byref(pw)) == 0 else None
            act = [nm for bit, nm in self.REASONS.items() if rs.value & bit] if reasons(h, c.byref(rs)) == 0 else []
            return (time.perf_counter(), float(sm.value), float(mx.value), p, act)

        return read if read() is not None else None

    def sample(self):
        if self.nvml is not None:
            s = self.nvml()
            if s is not None:
                self.samples.append(s)

    def _loop(self):
        while not self.stop.is_set():
            self.sample()
            self.stop.wait(self.period)

    # -- nvidia-smi fallback ----------------------------------------------
    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            f = [x.strip() for x in line.strip().split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            try:
                p = float(f[3])
            except ValueError:
                p = None
            act = [nm for nm, v in zip(names, f[5:9]) if v.lower().startswith("active")]
            self.samples.append((time.perf_counter(), sm, mx, p, act))

    def __enter__(self):
        self.nvml = self._open_nvml()
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", self.gpu], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def poll_until(self, event):
        """Sample from this thread until ``event`` (recorded after the timed
        work) has completed; the GPU is busy with the enqueued work meanwhile."""
        while not event.query():
            self.sample()
            time.sleep(0.0005)

    def summary(self, t0=None, t1=None):
        sel = [s for s in self.samples if (t0 is None or s[0] >= t0) and (t1 is None or s[0] <= t1)]
        src = "nvml" if self.nvml is not None else ("nvidia-smi" if self.proc is not None else None)
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": src,
                    "window_s": None if t0 is None or t1 is None else t1 - t0}
        sm = [s[1] for s in sel]
        pw = [s[3] for s in sel if s[3] is not None]
        reasons = sorted({r for s in sel for r in s[4]})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(s[2] for s in sel), "sm_mhz_min": min(sm),
                "reasons": reasons, "samples": len(sel), "power_w_max": max(pw) if pw else None, "source": src,
                "window_s": None if t0 is None or t1 is None else t1 - t0}


def gpu_id_for_smi(dev: torch.device) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:  # noqa: BLE001
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[dev.index or 0]
        return str(dev.index or 0)


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic():
    """dram bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since that capture."""
    h = hashlib.sha256()
    for p in DECODE_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    digest = h.hexdigest()[:16]
    try:
        with open(DECODE_PROFILE) as f:
            text = f.read()
    except OSError:
        return None, digest
    traffic, src = None, None
    for line in text.splitlines():
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1])
        if line.startswith("source_sha256_16:"):
            src = line.split(":", 1)[1].strip()
    return (traffic if src == digest else None), digest


# ---------------------------------------------------------------------------
# the workload on the device
# ---------------------------------------------------------------------------

class DecodeStep:
    """One decode step of a workload: per layer, write the new K/V rows into
    their slots, then attend (every layer has its own pool; the tables and
    lengths are shared, as the pages' pool tensor shares them across layers)."""

    def __init__(self, w: W.Workload, dev: torch.device):
        import pagedattention_decode_gb300 as P
        self.P, self.w, self.dev = P, w, dev
        B, hq, hkv, d, bs = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
        shape = (w.num_blocks, bs, hkv, d)
        self.k_caches = [W.normal_device(w.seed * 100 + 2 * l + 1, shape, w.sigma, w.dtype, str(dev))
                         for l in range(w.layers)]
        self.v_caches = [W.normal_device(w.seed * 100 + 2 * l + 2, shape, w.sigma, w.dtype, str(dev))
                         for l in range(w.layers)]
        self.k_cache, self.v_cache = self.k_caches[0], self.v_caches[0]
        g = W.generator(w.seed)
        self.q_host = W.normal(g, (B, hq, d), w.sigma, w.dtype)
        self.k_new_host = W.normal(g, (B, hkv, d), w.sigma, w.dtype)
        self.v_new_host = W.normal(g, (B, hkv, d), w.sigma, w.dtype)
        tables, order = W.scattered_tables(g, w.lengths, bs, w.num_blocks)
        self.order = order
        self.tables = tables.to(dev)
        self.lens = torch.tensor(w.lengths, dtype=torch.int32, device=dev)
        # the new token of each sequence sits at position L-1 (slot precomputed on the host)
        slots = [int(tables[i, (L - 1) // bs]) * bs + (L - 1) % bs for i, L in enumerate(w.lengths)]
        self.slots = torch.tensor(slots, dtype=torch.int64, device=dev)
        self.q = self.q_host.to(dev)
        self.k_new = self.k_new_host.to(dev)
        self.v_new = self.v_new_host.to(dev)
        self.out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
        ws = P.decode_workspace_size(B, hq, hkv, d, dev.index)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.sms = torch.cuda.get_device_properties(dev).multi_processor_count
        cap = 16 if d == 64 else 8
        hg = max(h for h in range(1, min(cap, hkv) + 1) if hkv % h == 0)
        self.num_hg = hkv // hg

    # fused: the new rows are written by the decode kernel (pkv_attn_decode_append)
    fused = False
    # window > 0: each sequence attends its most recent `window` keys (pkv_attn_decode_window)
    window = 0

    def write(self, layer=0):
        if self.fused:
            return
        self.P.write_kv(self.k_new, self.v_new, self.slots, self.k_caches[layer], self.v_caches[layer], err=self.err)

    def decode(self, layer=0):
        extra = dict(k_new=self.k_new, v_new=self.v_new) if self.fused else {}
        self.P.attn_decode(self.q, self.k_caches[layer], self.v_caches[layer], self.tables, self.lens, self.w.scale,
                           out=self.out, workspace=self.ws, err=self.err, window=self.window, **extra)

    def bytes(self):
        """(decode bytes, write bytes) of one layer (a window counts the keys it
        keeps)."""
        w = self.w
        dec = decode_bytes(windowed(w.lengths, self.window), w.num_q_heads, w.num_kv_heads, w.head_dim, 2, 4,
                           self.sms, self.num_hg)
        return dec, write_bytes(w.batch, w.num_kv_heads, w.head_dim, 2)


class DecodeStepInt8(DecodeStep):
    """The same decode step over an int8 cache (codes and per-block-per-head
    scales): write = quantised write of the new rows (re-quantising their
    blocks), decode = int8 split-K decode."""

    def __init__(self, w: W.Workload, dev: torch.device):
        super().__init__(w, dev)
        B, hkv, d, bs = w.batch, w.num_kv_heads, w.head_dim, w.block_size
        g = torch.Generator(device=str(dev))
        g.manual_seed(w.seed * 100 + 77)
        shape = (w.num_blocks, bs, hkv, d)
        self.kq = [torch.randint(-127, 128, shape, generator=g, dtype=torch.int8, device=dev) for _ in range(w.layers)]
        self.vq = [torch.randint(-127, 128, shape, generator=g, dtype=torch.int8, device=dev) for _ in range(w.layers)]
        self.ks = [torch.rand((w.num_blocks, hkv), generator=g, device=dev) * 0.03 + 0.01 for _ in range(w.layers)]
        self.vs = [torch.rand((w.num_blocks, hkv), generator=g, device=dev) * 0.03 + 0.01 for _ in range(w.layers)]
        self.k_caches = self.v_caches = None  # the 16-bit pools are not used
        torch.cuda.empty_cache()

    def write(self, layer=0):
        self.P.write_kv_int8(self.k_new, self.v_new, self.slots, self.kq[layer], self.vq[layer], self.ks[layer],
                             self.vs[layer], err=self.err)

    def decode(self, layer=0):
        self.P.attn_decode_int8(self.q, self.kq[layer], self.vq[layer], self.ks[layer], self.vs[layer], self.tables,
                                self.lens, self.w.scale, out=self.out, workspace=self.ws, err=self.err)

    def bytes(self):
        w = self.w
        hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
        dec = decode_bytes(w.lengths, hq, hkv, d, 1, 4, self.sms, self.num_hg)
        dec += len(w.lengths) * hq * d * 1  # q is 16-bit (decode_bytes counted it at 1 byte)
        dec += sum(-(-L // 16) for L in w.lengths) * 2 * hkv * 4  # the scale rows read per sub-block
        # each new token re-quantises its block: earlier rows read and rewritten, K and V
        wr = sum(2 * ((L - 1) % w.block_size) * hkv * d * 2 + 2 * hkv * d * (2 + 1) + 16 * hkv
                 for L in w.lengths)
        return dec, wr


def max_over_ranks(x: float, pg, dev) -> float:
    """The slowest rank's value (the job takes as long as its slowest replica)."""
    if pg is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def time_device(step: DecodeStep, steps: int, warmup: int, barrier):
    """The headline: ``steps`` steps between one start and one end event, the
    launches chained as a caller issues them (an event recorded between two
    launches would serialise them).  Then a second pass of the same steps with
    an event around every launch, for the per-launch times of the roofline and
    the per-step median."""
    stream = torch.cuda.current_stream()
    layers = step.w.layers
    for _ in range(warmup):
        for l in range(layers):
            step.write(l)
            step.decode(l)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3 * layers)] for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id_for_smi(step.dev)) as clk:
        t0 = time.perf_counter()
        start.record(stream)
        for i in range(steps):
            for l in range(layers):
                step.write(l)
                step.decode(l)
        end.record(stream)
        clk.poll_until(end)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        barrier()
        total_ms = start.elapsed_time(end)
        # per-launch pass (not part of the headline value)
        for i in range(steps):
            for l in range(layers):
                ev[i][3 * l].record(stream)
                step.write(l)
                ev[i][3 * l + 1].record(stream)
                step.decode(l)
                ev[i][3 * l + 2].record(stream)
        torch.cuda.synchronize()
    barrier()
    dec_ms = [e[3 * l + 1].elapsed_time(e[3 * l + 2]) for e in ev for l in range(layers)]
    wr_ms = [e[3 * l].elapsed_time(e[3 * l + 1]) for e in ev for l in range(layers)]
    step_ms = [e[0].elapsed_time(e[3 * layers - 1]) for e in ev]
    return total_ms, dec_ms, wr_ms, clk.summary(t0, t1), step_ms


def time_device_graph(step: DecodeStep, steps: int, warmup: int, barrier):
    """The whole step (every layer's write + decode) captured once as a CUDA
    graph and replayed: no per-call host work inside the timed region."""
    P = step.P
    layers = step.w.layers

    def one():
        for l in range(layers):
            step.write(l)
            step.decode(l)

    graph = P.StepGraph(one)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    # per-launch decode time for the roofline: the decode call of every layer
    # (distinct pools: together larger than L2 for every workload here)
    # captured as one graph, so no host work sits between the launches
    n_dec = max(layers, 4)
    dec_graph = P.StepGraph(lambda: [step.decode(i % layers) for i in range(n_dec)])
    a = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for i in range(5):
        a[i].record()
        dec_graph.replay()
    a[5].record()
    torch.cuda.synchronize()
    dec_eager = [a[i].elapsed_time(a[i + 1]) / n_dec for i in range(5)]
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(gpu_id_for_smi(step.dev)) as clk:
        t0 = time.perf_counter()
        start.record()
        for i in range(steps):
            marks[i].record()
            graph.replay()
        marks[steps].record()
        end.record()
        clk.poll_until(end)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
    barrier()
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
    return start.elapsed_time(end), dec_eager, [], clk.summary(t0, t1), step_ms


def _blob_layout(parts):
    """Byte offsets of named tensors packed into one buffer (256-byte aligned)."""
    off, lay = 0, {}
    for name, (shape, dtype) in parts.items():
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        lay[name] = (off, n, shape, dtype)
        off += (n + 255) // 256 * 256
    return lay, off


def _views(blob, lay):
    return {name: blob[o:o + n].view(dt).view(shape) for name, (o, n, shape, dt) in lay.items()}


def time_e2e(w: W.Workload, step: DecodeStep, steps: int, warmup: int, barrier, pipelined: bool = True):
    """Public-API step with host buffers: host allocator -> pinned host -> H2D ->
    pkv_write_kv + pkv_attn_decode -> D2H of the output -> host read of that
    output, all inside the timed region, every step.

    A step's inputs (q, new k/v rows, slot mapping, block tables, lengths) are
    packed into one pinned buffer and cross in one copy; the output comes back
    in one copy.  ``pipelined`` runs the loop the way a serving engine does:
    two buffer sets, the host prepares step i+1 while the GPU runs step i, the
    input copy of step i+1 and the output copy of step i-1 run on their own
    streams beside step i's kernels (one CUDA graph per set), and the host
    waits for step i's output after it has issued step i+1.  Otherwise every
    step runs on one stream and ends with the host reading its output before
    the next step starts."""
    P = step.P
    dev = step.dev
    B, hq, hkv, d, bs = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    alloc = P.BlockAllocator(w.num_blocks, bs)
    alloc.set_free_order(step.order)
    seqs = [alloc.create_sequence() for _ in range(B)]
    alloc.append_tokens(seqs, [L - 1 for L in w.lengths])  # cached context before the step
    max_blocks = W.blocks_for(max(w.lengths) + steps + warmup + 4, bs)
    lay, nbytes = _blob_layout({
        "q": (tuple(step.q.shape), step.q.dtype), "k": (tuple(step.k_new.shape), step.k_new.dtype),
        "v": (tuple(step.v_new.shape), step.v_new.dtype), "slots": ((B,), torch.int64),
        "tables": ((B, max_blocks), torch.int32), "lens": ((B,), torch.int32)})
    nsets = 2 if pipelined else 1

    class Set:
        def __init__(self):
            self.hin = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
            self.din = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            self.h, self.d = _views(self.hin, lay), _views(self.din, lay)
            self.h["q"].copy_(step.q_host)
            self.h["k"].copy_(step.k_new_host)
            self.h["v"].copy_(step.v_new_host)
            self.pairs = torch.empty(2 * B, dtype=torch.int64).pin_memory()
            self.hout = torch.empty((B, hq, d), dtype=torch.float32).pin_memory()
            self.dout = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
            self.in_done, self.comp_done, self.out_done = (torch.cuda.Event() for _ in range(3))
            self.graph = None

        def kernels(self):
            P.write_kv(self.d["k"], self.d["v"], self.d["slots"], step.k_cache, step.v_cache)
            P.attn_decode(self.d["q"], step.k_cache, step.v_cache, self.d["tables"], self.d["lens"], w.scale,
                          out=self.dout, workspace=step.ws)

    sets = [Set() for _ in range(nsets)]
    lens_seen, checksum = [], []
    compute = torch.cuda.current_stream()
    copy_in, copy_out = (torch.cuda.Stream() for _ in range(2)) if pipelined else (compute, compute)

    def host_part(s):
        npairs = alloc.append_tokens_into(seqs, s.h["slots"], s.pairs)
        assert npairs == 0
        alloc.fill_tables(seqs, max_blocks, s.h["tables"], s.h["lens"])
        lens_seen.append(int(s.h["lens"].sum()))

    for s in sets:  # captured on the first step's inputs; replays read the set's device buffers
        host_part(s)
        s.din.copy_(s.hin)
        s.graph = P.StepGraph(s.kernels)
    for s in sets:
        for e in (s.in_done, s.comp_done, s.out_done):
            e.record(compute)
    torch.cuda.synchronize()

    def launch(i):
        s = sets[i % nsets]
        s.in_done.synchronize()  # the pinned inputs of this set's previous step have been copied
        host_part(s)
        copy_in.wait_event(s.comp_done)  # the set's device inputs are no longer read
        with torch.cuda.stream(copy_in):
            s.din.copy_(s.hin, non_blocking=True)
        s.in_done.record(copy_in)
        compute.wait_event(s.in_done)
        compute.wait_event(s.out_done)  # the set's previous output has left the device
        s.graph.replay()
        s.comp_done.record(compute)
        copy_out.wait_event(s.comp_done)
        with torch.cuda.stream(copy_out):
            s.hout.copy_(s.dout, non_blocking=True)
        s.out_done.record(copy_out)

    def read(i):
        s = sets[i % nsets]
        s.out_done.synchronize()  # the host reads the step's result
        checksum.append(float(s.hout[0, 0, 0]))

    def run(n):
        if pipelined:
            launch(0)
            for i in range(1, n):
                launch(i)
                read(i - 1)
            read(n - 1)
        else:
            for i in range(n):
                launch(i)
                read(i)

    run(warmup)
    lens_seen.clear()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier()
    assert len(lens_seen) == steps and all(np.isfinite(checksum))
    h2d = sum(n for (_, n, _, _) in lay.values())
    d2h = sets[0].hout.numel() * sets[0].hout.element_size()
    kv_total = sum(lens_seen) * kv_bytes_per_token(hkv, d, 2)
    other = B * hq * d * (2 + 4) + write_bytes(B, hkv, d, 2)
    bytes_total = kv_total + steps * other
    return (t1 - t0) * 1e3, bytes_total, h2d, d2h


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_rate(w: W.Workload, budget_s: float, seqs_per_call=None, window: int = 0):
    """Times the binary64 oracle on a bounded sample of the workload (the first
    sequences, their blocks generated on the host with the workload's seed and
    shapes; window > 0: each sequence's last ``window`` keys).  Returns (GB/s
    of algorithmic KV bytes, seqs, seconds, cores)."""
    import oracle
    g = W.generator(w.seed + 1000)
    cores = len(os.sched_getaffinity(0))
    hq, hkv, d, bs = w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size

    def run(n):
        lens = w.lengths[:n]
        nb = sum(W.blocks_for(L, bs) for L in lens)
        kc = W.normal(g, (nb, bs, hkv, d), w.sigma, w.dtype)
        vc = W.normal(g, (nb, bs, hkv, d), w.sigma, w.dtype)
        q = W.normal(g, (n, hq, d), w.sigma, w.dtype)
        tables, _ = W.scattered_tables(g, lens, bs, nb)
        t0 = time.perf_counter()
        oracle.paged_attention(q, kc, vc, w.dtype, tables.numpy(), np.array(lens, dtype=np.int32), w.scale,
                               window=window)
        return time.perf_counter() - t0, sum(windowed(lens, window)) * kv_bytes_per_token(hkv, d, 2)

    oracle.build()
    if seqs_per_call is not None:
        dt, by = run(seqs_per_call)
        return by / dt / 1e9, seqs_per_call, dt, cores
    n, dt, by = 4, 0.0, 0
    while True:
        dt, by = run(n)
        if dt >= budget_s or n >= w.batch:
            break
        n = min(w.batch, max(n + 1, int(n * min(8.0, budget_s / max(dt, 1e-3)))))
    # the whole workload fits in less than the budget: repeat it and average
    reps, total_dt = 1, dt
    while total_dt < min(budget_s, 3.0):
        more, _ = run(n)
        total_dt += more
        reps += 1
    return by * reps / total_dt / 1e9, n, total_dt / reps, cores


def reference_arm(args, rank: int):
    if rank != 0:
        return
    w = W.gqa_decode()
    total = args.steps + args.warmup
    # size each step so the whole run stays near --ref-seconds of CPU time
    rate, n1, dt1, cores = oracle_sample_rate(w, min(0.5, args.ref_seconds))
    per_seq = dt1 / n1
    n = max(1, min(w.batch, int(args.ref_seconds / max(total, 1) / per_seq)))
    for _ in range(args.warmup):
        oracle_sample_rate(w, 0, seqs_per_call=n)
    times, gbs = [], []
    for _ in range(args.steps):
        r, _, dt, cores = oracle_sample_rate(w, 0, seqs_per_call=n)
        times.append(dt)
        gbs.append(r)
    value = float(np.mean(gbs))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "batch_sampled": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {w.batch} sequences per step, binary64 C oracle (OpenMP)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# secondary workload: the mixed packed step with a shared prefix and a beam split
# ---------------------------------------------------------------------------

class MixedStep:
    """GQA 32/8, D 128, fp16 (or ``dtype``), block_size 32.  Step 1: a 2048-token prefix
    shared (whole blocks) by 16 prefill chunks of 512 rows and 240 decode
    sequences with total contexts U[256, 8192]; 8432 new rows written, then one
    packed varlen call.  Step 2: 32 decode sequences fork to width 4, each beam
    appends a token (copy-on-write of non-full shared tails), copy_blocks,
    write, decode over the 128 beams.  Slots, tables and pairs come from the
    product allocator, set up once; the timed steps replay them."""

    def __init__(self, dev: torch.device, dtype: str = "f16"):
        import pagedattention_decode_gb300 as P
        self.P, self.dev = P, dev
        bs, hq, hkv, d, self.dtype = 32, 32, 8, 128, dtype
        self.bs, self.hq, self.hkv, self.d = bs, hq, hkv, d
        self.scale = 1.0 / math.sqrt(d)
        g = W.generator(5)
        dec_lens = W.mixed_step_decode_lengths()
        pre, chunk, nchunk = 2048, 512, 16
        shared = [min(pre // bs, (L - 1) // bs) for L in dec_lens]
        need = pre // bs + nchunk * W.blocks_for(pre + chunk, bs)
        need += sum(W.blocks_for(L, bs) - k for L, k in zip(dec_lens, shared)) + 32 * 4 * 2
        nb = int(math.ceil(1.1 * need))
        self.num_blocks = nb
        al = P.BlockAllocator(nb, bs)
        al.set_free_order(W.permutation(g, nb))
        owner = al.create_sequence()
        al.append_tokens([owner], [pre])
        prefix = al.block_table(owner)
        chunks = [al.create_sequence(prefix, pre) for _ in range(nchunk)]
        decs = []
        for L, k in zip(dec_lens, shared):
            sq = al.create_sequence(prefix[:k], k * bs)
            al.append_tokens([sq], [L - 1 - k * bs])
            decs.append(sq)
        seqs = chunks + decs
        q_lens = [chunk] * nchunk + [1] * len(decs)
        slots1, pairs = al.append_tokens(seqs, q_lens)
        assert not pairs
        self.k_cache = W.normal_device(51, (nb, bs, hkv, d), 1.0, self.dtype, str(dev))
        self.v_cache = W.normal_device(52, self.k_cache.shape, 1.0, self.dtype, str(dev))

        def tables_of(ids):
            mb = max(len(al.block_table(x)) for x in ids)
            t = torch.full((len(ids), mb), -1, dtype=torch.int32)
            ln = torch.empty(len(ids), dtype=torch.int32)
            al.fill_tables(ids, mb, t, ln)
            return t, ln

        t1, l1 = tables_of(seqs)
        cu = [0]
        for n in q_lens:
            cu.append(cu[-1] + n)
        self.s1 = dict(tables=t1.to(dev), lens=l1.to(dev), cu=torch.tensor(cu, dtype=torch.int32, device=dev),
                       q=W.normal(g, (cu[-1], hq, d), 1.0, self.dtype).to(dev),
                       k=W.normal(g, (len(slots1), hkv, d), 1.0, self.dtype).to(dev),
                       v=W.normal(g, (len(slots1), hkv, d), 1.0, self.dtype).to(dev),
                       slots=torch.tensor(slots1, dtype=torch.int64, device=dev), max_q=chunk)
        self.s1_lens_host = l1.tolist()
        self.q_lens = q_lens
        # the same rows split by kind, for per-kernel rates
        tp, lp = tables_of(chunks)
        self.pf = dict(tables=tp.to(dev), lens=lp.to(dev),
                       cu=torch.tensor(cu[:nchunk + 1], dtype=torch.int32, device=dev),
                       q=self.s1["q"][:nchunk * chunk])
        td, ld = tables_of(decs)
        self.dc = dict(tables=td.to(dev), lens=ld.to(dev), q=self.s1["q"][nchunk * chunk:])
        # step 2: beam split of 32 decode sequences
        pick = sorted(int(x) for x in torch.randperm(len(decs), generator=g)[:32])
        beams = []
        for i in pick:
            beams += [decs[i]] + [al.fork(decs[i]) for _ in range(3)]
        slots2, pairs2 = al.append_tokens(beams)
        t2, l2 = tables_of(beams)
        self.s2 = dict(tables=t2.to(dev), lens=l2.to(dev), q=W.normal(g, (len(beams), hq, d), 1.0, self.dtype).to(dev),
                       k=W.normal(g, (len(slots2), hkv, d), 1.0, self.dtype).to(dev),
                       v=W.normal(g, (len(slots2), hkv, d), 1.0, self.dtype).to(dev),
                       slots=torch.tensor(slots2, dtype=torch.int64, device=dev),
                       pairs=torch.tensor(pairs2 if pairs2 else [[0, 0]], dtype=torch.int64, device=dev)[:len(pairs2)])
        self.npairs = len(pairs2)
        self.s2_lens_host = l2.tolist()
        self.out1 = torch.empty((cu[-1], hq, d), dtype=torch.float32, device=dev)
        self.out2 = torch.empty((len(beams), hq, d), dtype=torch.float32, device=dev)
        self.ws = torch.empty(P.varlen_workspace_size(len(seqs), hq, hkv, d), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pre, self.chunk, self.nchunk, self.ndec = pre, chunk, nchunk, len(decs)

    def step1(self):
        P, s = self.P, self.s1
        P.write_kv(s["k"], s["v"], s["slots"], self.k_cache, self.v_cache, err=self.err)
        P.attn_varlen(s["q"], self.k_cache, self.v_cache, s["tables"], s["cu"], s["lens"], s["max_q"], self.scale,
                      out=self.out1, workspace=self.ws, err=self.err)

    def step2(self):
        P, s = self.P, self.s2
        if self.npairs:
            P.copy_blocks([self.k_cache], [self.v_cache], s["pairs"], err=self.err)
        P.write_kv(s["k"], s["v"], s["slots"], self.k_cache, self.v_cache, err=self.err)
        P.attn_decode(s["q"], self.k_cache, self.v_cache, s["tables"], s["lens"], self.scale, out=self.out2,
                      workspace=self.ws, err=self.err)

    def prefill_only(self):
        s = self.pf
        self.P.attn_varlen(s["q"], self.k_cache, self.v_cache, s["tables"], s["cu"], s["lens"], self.chunk,
                           self.scale, out=self.out1[:s["q"].shape[0]], workspace=self.ws, err=self.err)

    def decode_only(self):
        s = self.dc
        self.P.attn_decode(s["q"], self.k_cache, self.v_cache, s["tables"], s["lens"], self.scale,
                           out=self.out1[self.nchunk * self.chunk:], workspace=self.ws, err=self.err)

    def prefill_flops(self):
        # rows i of a chunk see prefix + i + 1 keys; 4 * D flops per key per head
        keys = sum(self.pre + i + 1 for i in range(self.chunk)) * self.nchunk
        return 4 * self.d * self.hq * keys

    def decode_rows_bytes(self):
        lens = self.s1_lens_host[self.nchunk:]
        sms = torch.cuda.get_device_properties(self.dev).multi_processor_count
        return decode_bytes(lens, self.hq, self.hkv, self.d, 2, 4, sms)  # logical KV (prefix re-reads included)


def time_fn(fn, steps, warmup):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def mixed_main(args):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    m = MixedStep(dev)
    with ClockSampler(gpu_id_for_smi(dev)) as clk:
        t1 = time_fn(m.step1, args.steps, args.warmup)
        t2 = time_fn(m.step2, args.steps, args.warmup)
        tp = time_fn(m.prefill_only, args.steps, args.warmup)
        td = time_fn(m.decode_only, args.steps, args.warmup)
    assert int(m.err.item()) == 0, f"device error word {int(m.err.item())}"
    fl = m.prefill_flops()
    db = m.decode_rows_bytes()
    line = {
        "workload": "mixed_prefix2048_16x512_prefill_240_decode_bs32_beam4x32", "steps": args.steps,
        "warmup": args.warmup, "step1_ms": t1, "step2_ms": t2,
        "step1_rows_per_s": (m.nchunk * m.chunk + m.ndec) / (t1 * 1e-3),
        "prefill_only_ms": tp, "prefill_tflops": fl / (tp * 1e-3) / 1e12, "prefill_gflop": fl / 1e9,
        "decode_rows_only_ms": td, "decode_rows_logical_GBps": db / (td * 1e-3) / 1e9,
        "step2_beams": len(m.s2_lens_host), "step2_cow_pairs": m.npairs, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# every workload of the scope table in the same run: one short timed block each
# ---------------------------------------------------------------------------

_T0 = time.perf_counter()


def log(msg: str) -> None:
    """Progress of the run on stderr (the JSON line stays alone on stdout)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f} s] {msg}", file=sys.stderr, flush=True)


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class OmpThreads:
    """Runs the oracle with n OpenMP threads (the oracle's libgomp), then
    restores the default."""

    def __init__(self, n: int):
        self.n = n

    def __enter__(self):
        import ctypes
        self.gomp = ctypes.CDLL("libgomp.so.1")
        self.before = self.gomp.omp_get_max_threads()
        self.gomp.omp_set_num_threads(int(self.n))
        return self

    def __exit__(self, *exc):
        self.gomp.omp_set_num_threads(int(self.before))


def cpu_baseline_decode(w: W.Workload, budget_s: float, budget_1core_s: float, int8: bool = False,
                        window: int = 0) -> dict:
    """The binary64 oracle on the host cores, all of them and one, on a bounded
    sample of the workload (its first sequences, host data of its shapes)."""
    if budget_s <= 0:
        return None
    import oracle
    oracle.build()
    if int8:
        rate_fn = oracle_sample_rate_int8
    else:
        def rate_fn(w_, b_):
            return oracle_sample_rate(w_, b_, window=window)
    rate, n, dt, cores = rate_fn(w, budget_s)
    with OmpThreads(1):
        rate1, n1, dt1, _ = rate_fn(w, budget_1core_s)
    kind = "int8 codes" if int8 else "K/V"
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "value_1core": rate1,
            "cpu_model": cpu_model(),
            "sample": f"first {n} of {w.batch} sequences ({dt:.2f} s per call); one core: first {n1} "
                      f"({dt1:.2f} s); GB/s of algorithmic {kind} bytes, binary64 C oracle"}


def oracle_sample_rate_int8(w: W.Workload, budget_s: float, seqs_per_call=None):
    """oracle_sample_rate for the int8 cache: codes and per-block-per-head scales."""
    import oracle
    g = W.generator(w.seed + 2000)
    rng = np.random.default_rng(w.seed + 2000)
    cores = len(os.sched_getaffinity(0))
    hq, hkv, d, bs = w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size

    def run(n):
        lens = w.lengths[:n]
        nb = sum(W.blocks_for(L, bs) for L in lens)
        kq = rng.integers(-127, 128, (nb, bs, hkv, d), dtype=np.int8)
        vq = rng.integers(-127, 128, (nb, bs, hkv, d), dtype=np.int8)
        ks = (rng.random((nb, hkv)) * 0.03 + 0.01).astype(np.float32)
        vs = (rng.random((nb, hkv)) * 0.03 + 0.01).astype(np.float32)
        q = W.normal(g, (n, hq, d), w.sigma, w.dtype)
        tables, _ = W.scattered_tables(g, lens, bs, nb)
        t0 = time.perf_counter()
        oracle.paged_attention_int8(q, w.dtype, kq, vq, ks, vs, tables.numpy(), np.array(lens, dtype=np.int32),
                                    w.scale)
        return time.perf_counter() - t0, sum(lens) * hkv * d * 2

    n, dt, by = 4, 0.0, 0
    while True:
        dt, by = run(n)
        if dt >= budget_s or n >= w.batch:
            break
        n = min(w.batch, max(n + 1, int(n * min(8.0, budget_s / max(dt, 1e-3)))))
    return by / dt / 1e9, n, dt, cores


def cpu_baseline_prefill(m, budget_s: float) -> dict:
    """The binary64 oracle on the mixed step's prefill chunks (512 causal rows
    over a 2048-token prefix each): once over all 16 chunks when the one-chunk
    estimate fits the budget, else over as many chunks as fit; one core on a
    slice of one chunk's rows."""
    if budget_s <= 0:
        return None
    import oracle
    oracle.build()
    g = W.generator(5000)
    hq, hkv, d, bs, pre, ch = m.hq, m.hkv, m.d, m.bs, m.pre, m.chunk
    npre, nown = pre // bs, W.blocks_for(ch, bs)
    cores = len(os.sched_getaffinity(0))

    def run(nchunks, rows):
        nb = npre + nchunks * nown
        kc = W.normal(g, (nb, bs, hkv, d), 1.0, "f16")
        vc = W.normal(g, (nb, bs, hkv, d), 1.0, "f16")
        tab = np.full((nchunks, npre + nown), -1, np.int32)
        for i in range(nchunks):
            tab[i, :npre] = np.arange(npre)
            tab[i, npre:] = npre + i * nown + np.arange(nown)
        # the last `rows` rows of each chunk (the most keys)
        lens = np.full(nchunks, pre + ch, np.int32)
        cu = np.arange(nchunks + 1, dtype=np.int32) * rows
        q = W.normal(g, (nchunks * rows, hq, d), 1.0, "f16")
        t0 = time.perf_counter()
        oracle.paged_attention(q, kc, vc, "f16", tab, lens, m.scale, cu_q=cu, causal=True)
        flops = 4 * d * hq * nchunks * sum(pre + ch - rows + i + 1 for i in range(rows))
        return time.perf_counter() - t0, flops

    dt1, fl1 = run(1, ch)
    k = m.nchunk if dt1 * m.nchunk * 8 / max(1, min(cores, 8 * m.nchunk)) <= budget_s else 1
    dt, fl = (dt1, fl1) if k == 1 else run(k, ch)
    with OmpThreads(1):
        dt_1, fl_1 = run(1, 64)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "value_1core": fl_1 / dt_1 / 1e12, "cpu_model": cpu_model(),
            "sample": f"{k} of {m.nchunk} chunks x {ch} causal rows ({fl / 1e9:.1f} GFLOP) in one call, "
                      f"{dt:.1f} s; one core: the last 64 rows of one chunk ({dt_1:.1f} s); binary64 C oracle"}


def time_parts(parts, iters, warmup, clk, before=None, clean=False):
    """CUDA-event time (ms) of each callable of ``parts`` per iteration, on the
    current stream; ``before`` (an L2 flush) runs outside the events.  Returns
    the [iters][parts] times and the clock summary of the timed window; with
    ``clean`` (no ``before``) also the mean time of one iteration from a first
    pass of ``iters`` iterations between one start and one end event (the
    launches chained as a caller issues them: an event recorded between two
    launches serialises them), whose clocks are then the ones returned."""
    for _ in range(warmup):
        if before is not None:
            before()
        for f in parts:
            f()
    torch.cuda.synchronize()
    clean_ms = None
    if clean and before is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record()
        for _ in range(iters):
            for f in parts:
                f()
        b.record()
        clk.poll_until(b)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        clean_ms = a.elapsed_time(b) / iters
        ck_clean = clk.summary(t0, t1)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(iters)]
    end = torch.cuda.Event()
    t0 = time.perf_counter()
    for i in range(iters):
        if before is not None:
            before()
        for j, f in enumerate(parts):
            ev[i][j].record()
            f()
        ev[i][-1].record()
    end.record()
    clk.poll_until(end)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    times = [[e[j].elapsed_time(e[j + 1]) for j in range(len(parts))] for e in ev]
    if clean_ms is not None:
        return times, ck_clean, clean_ms
    return times, clk.summary(t0, t1)


def _hbm_roofline(bytes_, ms, peak, kernel):
    a = bytes_ / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": a, "peak": peak, "unit": "GB/s", "frac": a / peak,
            "algorithmic_bytes_per_launch": bytes_, "launch_ms_median": ms}


CLEAN_NOTE = ("ms_per_step: mean over the iterations timed between one start and one end event (write and "
              "decode chained as a caller issues them); the roofline's launch time and ms_per_step_events_median "
              "from a second pass with an event around each launch")


def _med(xs):
    return statistics.median(xs)


def config_blocks(dev, iters: int, cpu_budget_s: float) -> dict:
    """Each workload of the scope table, timed in its own short block: median of
    ``iters`` iterations after 10 warm-up ones, its own roofline and clock
    window, and its own CPU oracle baseline."""
    import gc
    hbm, kind = measured_peak()
    tc, tc_kind = measured_tc_peak()
    gid = gpu_id_for_smi(dev)
    out = {}
    wu = 10
    with ClockSampler(gid) as clk:
        log("config block: 1 tiny MHA decode")
        # 1: tiny MHA decode, latency-bound; L2 flushed before every iteration
        w = W.tiny_decode()
        st = DecodeStep(w, dev)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        ms, ck = time_parts([st.write, st.decode], iters, wu, clk, before=flush.zero_)
        dec_b, wr_b = st.bytes()
        step = _med([a + b for a, b in ms])
        out["tiny"] = {
            "workload": w.name, "iters": iters, "ms_per_step": step,
            "ms_per_step_mean": float(np.mean([a + b for a, b in ms])), "tokens_per_s": w.batch / (step * 1e-3),
            "GB_per_s": (dec_b + wr_b) / (step * 1e-3) / 1e9, "l2": "512 MB written before every iteration",
            "roofline": dict(_hbm_roofline(dec_b, _med([b for _, b in ms]), hbm, "pkv_attn_decode"),
                             note="0.33 MB per call: launch- and latency-bound, not an HBM claim"),
            "clocks": ck, "cpu_baseline": cpu_baseline_decode(w, cpu_budget_s, cpu_budget_s / 2)}
        del st, flush
        gc.collect()
        torch.cuda.empty_cache()

        log("config block: 2 GPT-2-shaped 12-layer step")
        # 2: GPT-2-shaped 12-layer step, one CUDA graph per step
        w = W.gpt2_decode()
        st = DecodeStep(w, dev)
        layers = w.layers
        graph = st.P.StepGraph(lambda: [(st.write(l), st.decode(l)) for l in range(layers)])
        dec_graph = st.P.StepGraph(lambda: [st.decode(l) for l in range(layers)])
        # the same step with each layer's new row written by its decode kernel
        # (pkv_attn_decode_append: one launch fewer per layer, bit-identical)
        st.fused = True
        graph_fused = st.P.StepGraph(lambda: [(st.write(l), st.decode(l)) for l in range(layers)])
        st.fused = False
        ms, ck = time_parts([graph_fused.replay], iters, wu, clk)
        msp, _ = time_parts([graph.replay], iters, wu, clk)
        msd, _ = time_parts([dec_graph.replay], iters, wu, clk)
        dec_b, wr_b = st.bytes()
        step = _med([x[0] for x in ms])
        out["gpt2"] = {
            "workload": w.name, "iters": iters, "ms_per_step": step, "ms_per_step_mean": float(np.mean(ms)),
            "ms_per_step_write_then_decode": _med([x[0] for x in msp]),
            "tokens_per_s": w.batch / (step * 1e-3), "GB_per_s": layers * (dec_b + wr_b) / (step * 1e-3) / 1e9,
            "timed_as": "one CUDA graph per 12-layer step; each layer one pkv_attn_decode_append (the new row "
                        "written by the decode kernel, then attended); ms_per_step_write_then_decode: pkv_write_kv "
                        "then pkv_attn_decode per layer",
            "l2": "12 pools, %.0f MB of K/V per step vs 129 MB of L2, no flush" % (
                layers * sum(w.lengths) * kv_bytes_per_token(w.num_kv_heads, w.head_dim, 2) / 1e6),
            "roofline": _hbm_roofline(dec_b, _med([x[0] for x in msd]) / layers, hbm,
                                      "pkv_attn_decode (12 launches in one graph, per launch)"),
            "clocks": ck, "cpu_baseline": cpu_baseline_decode(w, cpu_budget_s, cpu_budget_s / 2)}
        del st, graph, dec_graph, graph_fused
        gc.collect()
        torch.cuda.empty_cache()

        log("config block: 4 long / skewed contexts")
        # 4: long / skewed contexts 1k .. 128k, split-K over every CTA
        w = W.long_skewed_decode()
        st = DecodeStep(w, dev)
        ms, ck, step = time_parts([st.write, st.decode], iters, wu, clk, clean=True)
        dec_b, wr_b = st.bytes()
        out["skew"] = {
            "workload": w.name, "iters": iters, "ms_per_step": step, "timed_as": CLEAN_NOTE,
            "ms_per_step_events_median": _med([a + b for a, b in ms]), "tokens_per_s": w.batch / (step * 1e-3),
            "GB_per_s": (dec_b + wr_b) / (step * 1e-3) / 1e9, "l2": "1.07 GB of K/V per step, no flush",
            "roofline": _hbm_roofline(dec_b, _med([b for _, b in ms]), hbm, "pkv_attn_decode (split-K + merge)"),
            "clocks": ck, "cpu_baseline": cpu_baseline_decode(w, cpu_budget_s, cpu_budget_s / 2)}
        del st
        gc.collect()
        torch.cuda.empty_cache()

        log("config block: GQA 32/8 over an int8 cache")
        # GQA 32/8 over an int8 cache (codes + per-block-per-head scales)
        w = W.gqa_decode()
        st = DecodeStepInt8(w, dev)
        ms, ck, step = time_parts([st.write, st.decode], iters, wu, clk, clean=True)
        dec_b, wr_b = st.bytes()
        out["gqa_int8"] = {
            "workload": w.name + "_int8", "iters": iters, "ms_per_step": step, "timed_as": CLEAN_NOTE,
            "ms_per_step_events_median": _med([a + b for a, b in ms]), "tokens_per_s": w.batch / (step * 1e-3),
            "GB_per_s": (dec_b + wr_b) / (step * 1e-3) / 1e9, "l2": "1.21 GB of codes per step, no flush",
            "roofline": _hbm_roofline(dec_b, _med([b for _, b in ms]), hbm, "pkv_attn_decode_int8 (split-K + merge)"),
            "clocks": ck, "cpu_baseline": cpu_baseline_decode(w, cpu_budget_s, cpu_budget_s / 2, int8=True)}
        del st
        gc.collect()
        torch.cuda.empty_cache()

        log("config block: GQA 32/8 with a sliding window")
        # GQA 32/8 with a 1,024-token window: each sequence reads only the
        # sub-blocks that cover its last 1,024 keys
        w = W.gqa_decode()
        st = DecodeStep(w, dev)
        st.window = 1024
        ms, ck, step = time_parts([st.write, st.decode], iters, wu, clk, clean=True)
        dec_b, wr_b = st.bytes()
        kept = sum(windowed(w.lengths, st.window)) * kv_bytes_per_token(w.num_kv_heads, w.head_dim, 2)
        out["window"] = {
            "workload": w.name + "_window1024", "iters": iters, "window": st.window, "ms_per_step": step,
            "timed_as": CLEAN_NOTE, "ms_per_step_events_median": _med([a + b for a, b in ms]),
            "tokens_per_s": w.batch / (step * 1e-3),
            "GB_per_s": (dec_b + wr_b) / (step * 1e-3) / 1e9,
            "l2": "%.2f GB of K/V in the windows per step, no flush" % (kept / 1e9),
            "roofline": _hbm_roofline(dec_b, _med([b for _, b in ms]), hbm, "pkv_attn_decode_window (split-K + merge)"),
            "clocks": ck, "cpu_baseline": cpu_baseline_decode(w, cpu_budget_s, cpu_budget_s / 2, window=st.window)}
        del st
        gc.collect()
        torch.cuda.empty_cache()

        log("config block: 5 mixed packed step")
        # 5: mixed packed step (prefill chunks + decode rows), then the beam split
        m = MixedStep(dev)
        n_mix = max(50, iters // 2)
        ms1, ck1 = time_parts([m.step1], n_mix, wu, clk)
        ms2, ck2 = time_parts([m.step2], n_mix, wu, clk)
        msp, ckp = time_parts([m.prefill_only], n_mix, wu, clk)
        msd, ckd = time_parts([m.decode_only], n_mix, wu, clk)
        assert int(m.err.item()) == 0, f"device error word {int(m.err.item())}"
        fl = m.prefill_flops()
        tp = _med([x[0] for x in msp])
        td = _med([x[0] for x in msd])
        a_tc = fl / (tp * 1e-3) / 1e12
        db = m.decode_rows_bytes()
        out["mixed"] = {
            "workload": "mixed_prefix2048_16x512_prefill_240_decode_bs32_beam4x32", "iters": n_mix,
            "step1_ms": _med([x[0] for x in ms1]), "step2_ms": _med([x[0] for x in ms2]),
            "step1_rows_per_s": (m.nchunk * m.chunk + m.ndec) / (_med([x[0] for x in ms1]) * 1e-3),
            "step2_beams": len(m.s2_lens_host), "step2_cow_pairs": m.npairs,
            "prefill_only": {"ms": tp, "gflop": fl / 1e9, "clocks": ckp,
                             "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel (tcgen05)",
                                          "achieved": a_tc, "peak": tc, "unit": "TFLOP/s", "frac": a_tc / tc,
                                          "peak_kind": tc_kind}},
            "decode_rows_only": {"ms": td, "clocks": ckd,
                                 "roofline": dict(_hbm_roofline(db, td, hbm, "pkv_attn_decode (240 rows)"),
                                                  note="logical bytes: the 2,048-token shared prefix is re-read "
                                                       "by every row and mostly served from L2")},
            "clocks": {"step1": ck1, "step2": ck2},
            "cpu_baseline": {"prefill": cpu_baseline_prefill(m, 7 * cpu_budget_s),
                             "decode_rows": cpu_baseline_decode(
                                 dataclasses.replace(W.gqa_decode(), name="mixed_decode_rows", lengths=list(
                                     m.s1_lens_host[m.nchunk:]), block_size=32, num_blocks=1, seed=5),
                                 cpu_budget_s, cpu_budget_s / 2)}}
        del m
        gc.collect()
        torch.cuda.empty_cache()
    return out


def measured_tc_peak():
    """Dense 16-bit tensor peak: the measured bf16 burst figure (fp16 has the
    same nominal rate), else the fallback 1.9 PFLOP/s."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst; fp16 = bf16 nominal)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback 1.9 PFLOP/s bf16 dense"


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                    help="replay each timed step as one CUDA graph (auto: on for multi-layer workloads)")
    ap.add_argument("--workload", default="gqa", choices=["gqa", "gqa_int8", "gpt2", "skew", "mixed"],
                    help="gqa: the headline decode step (GQA 32/8, B 256); gqa_int8: the same over an int8 "
                         "cache; gpt2: 12-layer MHA decode step; "
                         "skew: long/skewed split-K decode; mixed: the packed prefill+decode step")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: CPU seconds the whole --steps/--warmup run is sized to")
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first N sequences (a smaller case of the same workload, for profiling)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the short timed block of every other workload (tiny, gpt2, skew, int8, mixed)")
    ap.add_argument("--configs-iters", type=int, default=100,
                    help="timed iterations per workload block (median reported)")
    ap.add_argument("--fused-append", action="store_true",
                    help="gqa/gpt2/skew: write the new K/V rows inside the decode kernel (pkv_attn_decode_append) "
                         "instead of pkv_write_kv then pkv_attn_decode")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()

    if args.workload == "mixed" and args.impl == "pkv":
        mixed_main(args)
        return
    if args.impl == "reference":
        reference_arm(args, rank)
        if pg is not None:
            pg.destroy_process_group()
        return

    assert args.warmup >= 3, "at least 3 warm-up steps"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = {"gqa": W.gqa_decode, "gqa_int8": W.gqa_decode, "gpt2": W.gpt2_decode,
         "skew": W.long_skewed_decode}[args.workload]()
    if args.batch:
        w = W.first_sequences(w, args.batch)
    step = DecodeStepInt8(w, dev) if args.workload == "gqa_int8" else DecodeStep(w, dev)
    if args.fused_append:
        assert args.workload != "gqa_int8", "--fused-append: 16-bit caches only"
        step.fused = True
    use_graph = args.graph == "on" or (args.graph == "auto" and w.layers > 1)
    timer = time_device_graph if use_graph else time_device
    log(f"workload {w.name} set up")
    total_ms, dec_ms, wr_ms, clocks, step_ms = timer(step, args.steps, args.warmup, barrier)
    log("headline timed")
    dec_b, wr_b = step.bytes()
    step_bytes = (dec_b + wr_b) * w.layers
    total_ms = max_over_ranks(total_ms, pg, dev)
    ms_per_step = total_ms / args.steps
    value = world * step_bytes * args.steps / (total_ms * 1e-3) / 1e9
    tokens_per_s = world * w.batch * args.steps / (total_ms * 1e-3)  # one new token per sequence per step (all layers)
    assert int(step.err.item()) == 0, f"device error word {int(step.err.item())}"

    peak, peak_kind = measured_peak()
    dec_avg_ms = float(np.mean(dec_ms))
    if args.fused_append:
        dec_b += wr_b  # the decode launch also moves the new rows
    achieved = dec_b / (dec_avg_ms * 1e-3) / 1e9
    traffic, digest = profile_traffic()
    if args.workload != "gqa" or args.batch or args.fused_append:
        traffic = None  # the committed capture covers the full GQA 32/8 workload, write then decode
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_median": statistics.median(step_ms),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "block_size": w.block_size, "mean_context": sum(w.lengths) / w.batch,
                   "layers": w.layers,
                   "kv_bytes_per_step": w.layers * sum(w.lengths) * kv_bytes_per_token(
                       w.num_kv_heads, w.head_dim, 1 if args.workload == "gqa_int8" else 2),
                   "dtype": w.dtype, "kv_cache": "int8 + per-block-per-head fp32 scales"
                   if args.workload == "gqa_int8" else w.dtype,
                   "l2": ("inputs larger than L2 (%.2f GB of K/V per step vs 129 MB), no flush" %
                          (w.layers * sum(w.lengths) * kv_bytes_per_token(
                              w.num_kv_heads, w.head_dim, 1 if args.workload == "gqa_int8" else 2) / 1e9)),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "write": "in the decode kernel (pkv_attn_decode_append)" if args.fused_append
                   else "pkv_write_kv then pkv_attn_decode"},
        "tokens_per_s": tokens_per_s,
        "pct_of_hbm": {"nominal_8TBs": 100.0 * value / world / NOMINAL_HBM_GBS,
                       f"{peak_kind}_{peak:.0f}GBs": 100.0 * value / world / peak},
        "roofline": {"bound": "hbm", "kernel": ("pkv_attn_decode_int8" if args.workload == "gqa_int8"
                                                 else "pkv_attn_decode") + " (split-K decode + merge)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy, burst)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "traffic": traffic,
                     "algorithmic_bytes_per_launch": dec_b, "avg_launch_ms": dec_avg_ms,
                     "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS, "kernel_source_sha256_16": digest},
        "write_kv": ({"avg_launch_ms": float(np.mean(wr_ms)), "bytes": wr_b,
                      "GB_per_s": wr_b / (float(np.mean(wr_ms)) * 1e-3) / 1e9}
                     if wr_ms and not args.fused_append else None),
        "timed_as": "one CUDA graph per step" if use_graph else
        ("eager calls on one stream, K steps between a start and an end event; avg_launch_ms, write_kv and "
         "ms_per_step_median from a second pass of K steps with an event around every launch"),
        "clocks": clocks,
        "gpu_launches": args.steps * (2 if args.fused_append else 3) * w.layers,
    }
    if not args.no_e2e and w.layers == 1 and args.workload != "gqa_int8" and not args.fused_append:
        n_e2e = max(1, min(args.steps, 200))
        ser_ms, _, _, _ = time_e2e(w, step, n_e2e, 3, barrier, pipelined=False)
        e2e_ms, e2e_bytes, h2d, d2h = time_e2e(w, step, n_e2e, 3, barrier)
        e2e_ms, ser_ms = max_over_ranks(e2e_ms, pg, dev), max_over_ranks(ser_ms, pg, dev)
        line["e2e"] = {"value": world * e2e_bytes / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / n_e2e, "steps": n_e2e,
                       "tokens_per_s": world * w.batch * n_e2e / (e2e_ms * 1e-3),
                       "path": "host allocator -> one pinned H2D of the packed inputs -> [CUDA graph: "
                               "pkv_write_kv -> pkv_attn_decode] -> one D2H of the output -> host read; two buffer "
                               "sets: host work and both copies of neighbouring steps overlap step i's kernels",
                       "serial_ms_per_step": ser_ms / n_e2e}
    log("e2e timed")
    if rank == 0 and not args.no_cpu_baseline:
        rate, n, dt, cores = oracle_sample_rate(w, 5.0)
        with OmpThreads(1):
            rate1, n1, dt1, _ = oracle_sample_rate(w, 2.0)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "value_1core": rate1, "cpu_model": cpu_model(),
                                "sample": f"first {n} of {w.batch} sequences, one call, {dt:.1f} s; one core: "
                                          f"first {n1} ({dt1:.1f} s); binary64 C oracle"}
    if rank == 0 and not args.no_configs and args.workload == "gqa" and not args.batch:
        del step
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        line["configs"] = config_blocks(dev, args.configs_iters, 1.5 if not args.no_cpu_baseline else 0.0)
    log("done")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
