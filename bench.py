"""Benchmark of the lat_attn hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extra] [--no-cpu]

A step is one pass of the attention hot path over one batch of synthetic input.  The
headline workload is the largest configuration that fits one GPU: the Gemma-4 global
attention layer (16 query heads over 2 KV heads, head_dim 512), as a causal bf16 prefill
of 8192 tokens; the same layer's decode step (8 sequences at 32768 cached tokens) is
reported beside it under "decode".  Each timed step is bracketed by CUDA events on the
launching stream; before every step a 256 MiB write and a 256 MiB read leave L2 cold and
clean.

`value` is TFLOP/s of algorithmic work (4*D FLOPs per visible query-key pair per head);
decode values are GB/s of K/V read (each cached element counted once per KV head).
`e2e` runs the steps through the C ABI from pinned host buffers: a prefill step uploads
Q/K/V and downloads the output and lse; a decode step uploads the query, the new K/V row
and the lengths, appends the row into the device-resident cache, decodes and downloads
the output and lse.  Steps are pipelined over two buffer sets on three streams.
`roofline` rates the timed kernel against the tensor (prefill) or HBM (decode) roofline
of MEASURED_PEAKS.json.  `workloads` adds the other named shapes, each against its own
roofline, plus the tiny fp32 case (prefill, append, decode) in microseconds.
`cpu_baseline` is the fp64 oracle on the host cores over a deterministic sample (query
rows for prefill, sequences for decode), whose exact share of the algorithmic work is
known, so the sample's throughput is the oracle's throughput on the whole workload.
With --impl reference the oracle itself is the timed arm.  --workload NAME makes any
named workload the timed one.

Multi-GPU runs (torchrun) are independent replicas of the same workload (the path has no
exchange step); every rank times its own steps and the slowest rank sets the time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "GQA attention prefill TFLOP/s and decode KV GB/s, % of GB300 roofline"
HEADLINE = "gemma4_global_prefill"
COMPANION = "gemma4_global_decode"   # the same layer's decode step, reported beside it
FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed before every timed step: a 256 MiB write, then a 256 MiB read that "
           "leaves no dirty lines to write back during the step")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def visible_pairs(S, L, causal, window):
    """Number of (query row, key) pairs the mask leaves visible, per (batch, head)."""
    i = np.arange(S, dtype=np.int64)
    p = i + (L - S)
    hi = np.minimum(L, p + 1) if causal else np.full(S, L, dtype=np.int64)
    lo = np.maximum(0, p - window + 1) if window > 0 else np.zeros(S, dtype=np.int64)
    return int(np.maximum(hi - lo, 0).sum())


def prefill_work(wl):
    pairs = visible_pairs(wl.S, wl.L, wl.causal, wl.window)
    flops = 4.0 * wl.D * wl.Hq * wl.B * pairs
    es = 2 if wl.dtype == "bf16" else 4
    bytes_ = (wl.B * wl.S * wl.Hq * wl.D * es * 2          # Q read, out written
              + 2 * wl.B * wl.L * wl.Hkv * wl.D * es        # K, V read once
              + wl.B * wl.S * wl.Hq * 4)                    # lse written
    return flops, float(bytes_), pairs


def decode_work(wl, kv_lens):
    es = 2 if wl.dtype == "bf16" else 4
    keys = int(sum(min(int(n), wl.window) if wl.window > 0 else int(n) for n in kv_lens))
    kv_bytes = keys * wl.Hkv * wl.D * 2 * es
    bytes_ = kv_bytes + wl.B * wl.Hq * wl.D * es * 2 + wl.B * wl.Hq * 4
    flops = 4.0 * wl.D * wl.Hq * keys
    return flops, float(bytes_), keys


def code_lines(text):
    """The source without // comments and blank lines: what the hash of a kernel covers,
    so that editing a comment does not orphan its ncu summary."""
    out = []
    for line in text.splitlines():
        line = line.split("//", 1)[0].rstrip()
        if line:
            out.append(line)
    return "\n".join(out) + "\n"


def kernel_source_hash(names):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gqa_attention_lat_gb300", "csrc")
    for n in names:
        with open(os.path.join(csrc, n)) as f:
            h.update(code_lines(f.read()).encode())
    return h.hexdigest()[:16]


def profile_traffic(profile_name, src_names):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on the
    current kernel source (the summary records the source hash); else None."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha256_16") != kernel_source_hash(src_names):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the GPU is busy."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.idx = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ GPU arm

class Flusher:
    """Evicts the timed step's data from L2 before each step: a 256 MiB write (2x L2), then
    a 256 MiB read of a second buffer, which pushes the written lines back to DRAM before
    the step starts instead of during it (a write alone leaves ~L2-sized dirty data whose
    write-back would compete with the step's own reads)."""

    def __init__(self, device):
        self.buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.rd = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.zero_()
        torch.sum(self.rd, dim=0, out=self.sink)


def replica_throughput(ms_local, work, world, dist=None, device="cpu"):
    """Whole-job throughput of `world` replicas that each processed `work` units in
    `ms_local` milliseconds: the slowest rank (max over ranks) bounds the job, so the
    value is world * work / max_ms.  Returns (max_ms, value)."""
    ms = float(ms_local)
    if dist is not None:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, work * world / (ms / 1e3)


def time_steps(fn, steps, flush, stream):
    """Run `fn` `steps` times, L2 flushed before each; returns per-step ms (CUDA events
    recorded on the stream the kernels run on)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        flush()
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


class PrefillStep:
    def __init__(self, wl, device):
        from gqa_attention_lat_gb300 import binding
        self.b = binding
        self.wl = wl
        self.inp = W.prefill_inputs(wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D, dtype=wl.dtype,
                                    device=device, packed=wl.packed, k_mul=wl.k_mul)
        self.out = torch.empty((wl.B * wl.S, wl.Hq * wl.D), dtype=W.torch_dtype(wl.dtype),
                               device=device)
        self.lse = torch.empty((wl.B * wl.S, wl.Hq), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.dt = binding.LAT_BF16 if wl.dtype == "bf16" else binding.LAT_F32

    def __call__(self, q=None, k=None, v=None):
        i, wl = self.inp, self.wl
        q = i.q if q is None else q
        k = i.k if k is None else k
        v = i.v if v is None else v
        if wl.softcap > 0:
            self.b.lat_attn_prefill_softcap(self.dt, q, i.q.stride(0), k, i.k.stride(0), v,
                                            i.v.stride(0), self.out, self.out.stride(0), self.lse,
                                            wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D, wl.causal,
                                            wl.window, wl.scale, wl.softcap, self.status)
            return
        self.b.lat_attn_prefill(self.dt, q, i.q.stride(0), k, i.k.stride(0), v, i.v.stride(0),
                                self.out, self.out.stride(0), self.lse, wl.B, wl.S, wl.L, wl.Hq,
                                wl.Hkv, wl.D, wl.causal, wl.window, wl.scale, self.status)

    def check_status(self):
        st = int(self.status.item())
        if st != 0:
            raise RuntimeError("device status %s" % self.b.lat_status_string(st))


class PrefillCachedStep:
    """A chunk of S new query rows per sequence against the first L rows of a token-major
    KV cache of `cap` slots (slots past L hold NaN)."""

    def __init__(self, wl, device):
        from gqa_attention_lat_gb300 import binding
        self.b = binding
        self.wl = wl
        self.di = W.decode_inputs(wl.B, wl.Hq, wl.Hkv, wl.D, wl.cap, kv_lens=wl.L,
                                  dtype=wl.dtype, device=device, nan_fill=True)
        self.q = W.normal((wl.B * wl.S, wl.Hq * wl.D), dtype=wl.dtype, device=device,
                          seed=W.BASE_SEED, role="chunk_q")
        self.out = torch.empty((wl.B * wl.S, wl.Hq * wl.D), dtype=W.torch_dtype(wl.dtype),
                               device=device)
        self.lse = torch.empty((wl.B * wl.S, wl.Hq), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.dt = binding.LAT_BF16 if wl.dtype == "bf16" else binding.LAT_F32

    def __call__(self, q=None, k_cache=None, v_cache=None):
        wl, d = self.wl, self.di
        q = self.q if q is None else q
        k_cache = d.k_cache if k_cache is None else k_cache
        v_cache = d.v_cache if v_cache is None else v_cache
        self.b.lat_attn_prefill_cached(self.dt, q, self.q.stride(0), k_cache, v_cache,
                                       wl.Hkv * wl.D, wl.D, wl.cap * wl.Hkv * wl.D, self.out,
                                       self.out.stride(0), self.lse, wl.B, wl.S, wl.L, wl.Hq,
                                       wl.Hkv, wl.D, wl.causal, wl.window, wl.scale,
                                       self.status)

    def check_status(self):
        st = int(self.status.item())
        if st != 0:
            raise RuntimeError("device status %s" % self.b.lat_status_string(st))


class ProducerStep:
    """Q/K RMS norm + RoPE + V + cache append for S new rows per sequence from a fused
    QKV buffer (positions 0 .. S-1), into a token-major cache of `cap` slots."""

    def __init__(self, wl, device):
        from gqa_attention_lat_gb300 import binding
        self.b = binding
        self.wl = wl
        width = (wl.Hq + 2 * wl.Hkv) * wl.D
        self.qkv = W.normal((wl.B * wl.S, width), dtype=wl.dtype, device=device,
                            seed=W.BASE_SEED, role="new")
        self.q_w = W.normal((wl.D,), dtype=wl.dtype, device=device, seed=W.BASE_SEED, role="q")
        self.k_w = W.normal((wl.D,), dtype=wl.dtype, device=device, seed=W.BASE_SEED, role="k")
        tdt = W.torch_dtype(wl.dtype)
        self.k_cache = torch.zeros((wl.B, wl.cap, wl.Hkv * wl.D), dtype=tdt, device=device)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.q_out = torch.empty((wl.B * wl.S, wl.Hq * wl.D), dtype=tdt, device=device)
        self.pos = torch.zeros(wl.B, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.dt = binding.LAT_BF16 if wl.dtype == "bf16" else binding.LAT_F32
        self.out = self.q_out

    def __call__(self, qkv=None):
        wl = self.wl
        qkv = self.qkv if qkv is None else qkv
        self.b.lat_qkv_norm_rope_append(self.dt, qkv, self.qkv.stride(0), self.q_w, self.k_w,
                                        1e-6, 1e6, False, self.q_out, self.q_out.stride(0),
                                        self.k_cache, self.v_cache, wl.Hkv * wl.D, wl.D,
                                        wl.cap * wl.Hkv * wl.D, wl.cap, self.pos, wl.S, wl.B,
                                        wl.Hq, wl.Hkv, wl.D, self.status)

    def check_status(self):
        st = int(self.status.item())
        if st != 0:
            raise RuntimeError("device status %s" % self.b.lat_status_string(st))


def producer_bytes(wl):
    es = 2 if wl.dtype == "bf16" else 4
    rows = wl.B * wl.S
    return float(rows * (wl.Hq + 2 * wl.Hkv) * wl.D * es * 2 + 2 * wl.D * es)  # read + write


class DecodeStep:
    def __init__(self, wl, device):
        from gqa_attention_lat_gb300 import binding
        self.b = binding
        self.wl = wl
        if wl.ring:
            self.di = W.ring_decode_inputs(wl.B, wl.Hq, wl.Hkv, wl.D, wl.ring, wl.max_len,
                                           dtype=wl.dtype, device=device)
        else:
            self.di = W.decode_inputs(wl.B, wl.Hq, wl.Hkv, wl.D, wl.L, kv_lens=wl.kv_lens,
                                      dtype=wl.dtype, device=device, nan_fill=True)
        self.dt = binding.LAT_BF16 if wl.dtype == "bf16" else binding.LAT_F32
        self.nbytes = binding.lat_attn_decode_workspace_size(self.dt, wl.B, wl.Hq, wl.Hkv, wl.D,
                                                             wl.L)
        self.ws = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=device)
        self.out = torch.empty((wl.B, wl.Hq * wl.D), dtype=W.torch_dtype(wl.dtype), device=device)
        self.lse = torch.empty((wl.B, wl.Hq), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def __call__(self, q=None, k_cache=None, v_cache=None, kv_lens=None):
        d, wl = self.di, self.wl
        q = d.q if q is None else q
        k_cache = d.k_cache if k_cache is None else k_cache
        v_cache = d.v_cache if v_cache is None else v_cache
        kv_lens = d.kv_lens if kv_lens is None else kv_lens
        if wl.ring:
            self.b.lat_attn_decode_ring(self.dt, q, d.q.stride(0), k_cache, v_cache,
                                        wl.Hkv * wl.D, wl.D, wl.L * wl.Hkv * wl.D, wl.ring,
                                        kv_lens, wl.max_len, self.out, self.out.stride(0),
                                        self.lse, wl.B, wl.Hq, wl.Hkv, wl.D, wl.window,
                                        wl.scale, self.ws, self.nbytes, self.status)
            return
        self.b.lat_attn_decode(self.dt, q, d.q.stride(0), k_cache, v_cache, wl.Hkv * wl.D,
                               wl.D, wl.L * wl.Hkv * wl.D, kv_lens, wl.L, self.out,
                               self.out.stride(0), self.lse, wl.B, wl.Hq, wl.Hkv, wl.D,
                               wl.window, wl.scale, self.ws, self.nbytes, self.status)

    def check_status(self):
        st = int(self.status.item())
        if st != 0:
            raise RuntimeError("device status %s" % self.b.lat_status_string(st))


def prefill_bound(wl, peaks):
    """'tensor' when the workload's arithmetic intensity is above the ridge point of the
    measured peaks, else 'hbm'."""
    flops, bytes_, _ = prefill_work(wl)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return "hbm" if flops / bytes_ < ridge else "tensor"


def measure_extra(device, flush, stream, peaks, reps=20, skip=()):
    """The other named workloads, each against its own roofline."""
    res = {}
    for name in ("gemma4_sliding_prefill", "qwen3_0.6b_prefill", "gemma2_softcap_prefill",
                 "gemma4_global_prefill"):
        if name in skip:
            continue
        wl = W.WORKLOADS[name]
        step = PrefillStep(wl, device)
        for _ in range(3):
            step()
        ms = time_steps(step, reps, flush, stream)
        step.check_status()
        flops, bytes_, _ = prefill_work(wl)
        t = statistics.mean(ms) / 1e3
        tf = flops / t / 1e12
        res[name] = {"kind": "prefill", "ms": statistics.mean(ms), "tflops": tf,
                     "gbs": bytes_ / t / 1e9, "bound": prefill_bound(wl, peaks),
                     "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
                     "frac_of_hbm_peak": bytes_ / t / 1e9 / peaks["hbm_gbs"],
                     "gflop": flops / 1e9}
        del step
        torch.cuda.empty_cache()
    for name in ("qwen3_chunked_prefill",):
        wl = W.WORKLOADS[name]
        step = PrefillCachedStep(wl, device)
        for _ in range(3):
            step()
        ms = time_steps(step, reps, flush, stream)
        step.check_status()
        flops, bytes_, _ = prefill_work(wl)
        t = statistics.mean(ms) / 1e3
        tf = flops / t / 1e12
        res[name] = {"kind": "prefill_cached", "ms": statistics.mean(ms), "tflops": tf,
                     "gbs": bytes_ / t / 1e9, "bound": "hbm",
                     "frac_of_hbm_peak": bytes_ / t / 1e9 / peaks["hbm_gbs"],
                     "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "gflop": flops / 1e9}
        del step
        torch.cuda.empty_cache()
    for name in ("qwen3_qkv_producer",):
        wl = W.WORKLOADS[name]
        step = ProducerStep(wl, device)
        for _ in range(3):
            step()
        ms = time_steps(step, reps, flush, stream)
        step.check_status()
        bytes_ = producer_bytes(wl)
        t = statistics.mean(ms) / 1e3
        res[name] = {"kind": "producer", "ms": statistics.mean(ms), "gbs": bytes_ / t / 1e9,
                     "bound": "hbm", "frac_of_hbm_peak": bytes_ / t / 1e9 / peaks["hbm_gbs"],
                     "mbytes": bytes_ / 1e6}
        del step
        torch.cuda.empty_cache()
    for name in ("decode_b32_h32_kv8_d128", "gemma4_sliding_decode_ring",
                 "decode_b1_kv2_d128_128k", "gemma4_global_decode"):
        if name in skip:
            continue
        wl = W.WORKLOADS[name]
        step = DecodeStep(wl, device)
        for _ in range(3):
            step()
        ms = time_steps(step, reps, flush, stream)
        step.check_status()
        flops, bytes_, keys = decode_work(wl, step.di.kv_lens.cpu().tolist())
        t = statistics.mean(ms) / 1e3
        gbs = bytes_ / t / 1e9
        res[name] = {"kind": "decode", "ms": statistics.mean(ms), "gbs": gbs, "bound": "hbm",
                     "frac_of_hbm_peak": gbs / peaks["hbm_gbs"], "mbytes": bytes_ / 1e6,
                     "tflops": flops / t / 1e12}
        del step
        torch.cuda.empty_cache()
    # the Qwen3-shaped prefill with a warm L2: a burst of back-to-back steps between two
    # events (its 25 MB of inputs and outputs stay in the 129 MB L2)
    wl = W.WORKLOADS["qwen3_0.6b_prefill"]
    step = PrefillStep(wl, device)
    for _ in range(3):
        step()
    n = 50
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record(stream)
    for _ in range(n):
        step()
    s1.record(stream)
    torch.cuda.synchronize()
    step.check_status()
    flops, bytes_, _ = prefill_work(wl)
    t = s0.elapsed_time(s1) / n / 1e3
    res[wl.name + "_warm_l2"] = {"kind": "prefill", "ms": t * 1e3, "tflops": flops / t / 1e12,
                                 "bound": "latency", "gbs": bytes_ / t / 1e9,
                                 "note": "no flush: back-to-back steps, inputs resident in L2"}
    del step
    torch.cuda.empty_cache()
    # KV append of one new row per sequence into the decode cache shape (timed on its own)
    res.update(measure_append(device, flush, stream, reps))
    res.update(measure_tiny(device, flush, stream, reps))
    return res


def measure_tiny(device, flush, stream, reps):
    """The tiny fp32 case in microseconds: a causal prefill of 64 tokens (4 query heads, 2
    KV heads, head_dim 64), the append of token 63 into a 64-slot cache holding tokens
    0..62, then one decode step at kv_len 64 -- three launches per step, and each alone."""
    from gqa_attention_lat_gb300 import binding
    pw = W.WORKLOADS["tiny_f32_prefill"]
    B, S, Hq, Hkv, D = pw.B, pw.S, pw.Hq, pw.Hkv, pw.D
    inp = W.prefill_inputs(B, S, S, Hq, Hkv, D, dtype="f32", device=device)
    out = torch.empty((S, Hq * D), dtype=torch.float32, device=device)
    lse = torch.empty((S, Hq), dtype=torch.float32, device=device)
    cap = S
    kc = torch.zeros((1, cap, Hkv * D), dtype=torch.float32, device=device)
    vc = torch.zeros_like(kc)
    kc[0, :S - 1] = inp.k[:S - 1]
    vc[0, :S - 1] = inp.v[:S - 1]
    pos = torch.tensor([S - 1], dtype=torch.int32, device=device)
    lens = torch.tensor([S], dtype=torch.int32, device=device)
    q_last = inp.q[S - 1:].contiguous()
    dout = torch.empty((1, Hq * D), dtype=torch.float32, device=device)
    dlse = torch.empty((1, Hq), dtype=torch.float32, device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)

    def prefill():
        binding.lat_attn_prefill(binding.LAT_F32, inp.q, inp.q.stride(0), inp.k,
                                 inp.k.stride(0), inp.v, inp.v.stride(0), out, out.stride(0),
                                 lse, B, S, S, Hq, Hkv, D, True, 0, pw.scale, st)

    def append():
        binding.lat_kv_append(binding.LAT_F32, kc, vc, Hkv * D, D, cap * Hkv * D, cap,
                              inp.k[S - 1:], inp.v[S - 1:], inp.k.stride(0), pos, 1, 1, Hkv,
                              D, st)

    def decode():
        binding.lat_attn_decode(binding.LAT_F32, q_last, q_last.stride(0), kc, vc, Hkv * D, D,
                                cap * Hkv * D, lens, cap, dout, dout.stride(0), dlse, 1, Hq,
                                Hkv, D, 0, pw.scale, None, 0, st)

    def all3():
        prefill()
        append()
        decode()
    res = {}
    for name, fn in (("tiny_f32_prefill_append_decode", all3), ("tiny_f32_prefill", prefill),
                     ("tiny_f32_append", append), ("tiny_f32_decode", decode)):
        for _ in range(3):
            fn()
        ms = time_steps(fn, reps, flush, stream)
        res[name] = {"kind": "tiny_f32", "us": statistics.mean(ms) * 1e3,
                     "us_median": statistics.median(ms) * 1e3, "bound": "latency",
                     "launches": 3 if fn is all3 else 1,
                     "note": "B1 S64 Hq4 Hkv2 D64 fp32, L2 flushed; event-timed, including "
                             "the launch floor"}
    if int(st.item()) != 0:
        raise RuntimeError("device status %s" % binding.lat_status_string(int(st.item())))
    return res


def measure_append(device, flush, stream, reps):
    from gqa_attention_lat_gb300 import binding
    wl = W.WORKLOADS["decode_b32_h32_kv8_d128"]
    B, Hkv, D, cap = wl.B, wl.Hkv, wl.D, wl.L
    kc = torch.zeros((B, cap, Hkv * D), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    kn = W.normal((B, Hkv * D), dtype="bf16", device=device, seed=W.BASE_SEED, role="k")
    vn = W.normal((B, Hkv * D), dtype="bf16", device=device, seed=W.BASE_SEED, role="v")
    pos = torch.full((B,), cap - 1, dtype=torch.int32, device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)

    def run():
        binding.lat_kv_append(binding.LAT_BF16, kc, vc, Hkv * D, D, cap * Hkv * D, cap, kn, vn,
                              Hkv * D, pos, 1, B, Hkv, D, st)
    for _ in range(3):
        run()
    ms = time_steps(run, reps, flush, stream)
    if int(st.item()) != 0:
        raise RuntimeError("device status %s" % binding.lat_status_string(int(st.item())))
    t = statistics.mean(ms) / 1e3
    bytes_ = 2.0 * 2 * B * Hkv * D * 2  # K and V rows, read and written
    return {"kv_append_b32_kv8_d128": {"kind": "append", "ms": t * 1e3, "gbs": bytes_ / t / 1e9,
                                       "bound": "latency", "kbytes": bytes_ / 1e3,
                                       "note": "one new row per sequence, L2 flushed"}}


def pipelined_e2e(hosts, out_like, run, steps, stream):
    """Time `steps` end-to-end steps from pinned host buffers: each step uploads `hosts`
    into one of two device buffer sets, calls run(dev_inputs, dev_outputs) on `stream`,
    and downloads the outputs (shaped like `out_like`) into pinned host memory.  Steps
    are pipelined over the two sets on three streams (upload, compute, download), so the
    upload of step i+1 and the download of step i-1 overlap the kernels of step i, as a
    serving loop over independent batches would run.  Returns (ms per step, h2d bytes,
    d2h bytes), the time being the whole run's span divided by the steps."""
    nbuf = 2
    devs = [[torch.empty(h.shape, dtype=h.dtype, device=stream.device) for h in hosts]
            for _ in range(nbuf)]
    outs = [[torch.empty_like(o) for o in out_like] for _ in range(nbuf)]
    host_outs = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in out_like]
                 for _ in range(nbuf)]
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    up_done = [ev() for _ in range(nbuf)]
    run_done = [ev() for _ in range(nbuf)]
    down_done = [ev() for _ in range(nbuf)]
    used = [False] * nbuf

    def one(i):
        k = i % nbuf
        with torch.cuda.stream(s_up):
            if used[k]:
                s_up.wait_event(run_done[k])      # the kernels of step i-2 read devs[k]
            for dv, h in zip(devs[k], hosts):
                dv.copy_(h, non_blocking=True)
            up_done[k].record(s_up)
        stream.wait_event(up_done[k])
        if used[k]:
            stream.wait_event(down_done[k])       # step i-2's outputs are downloaded
        run(devs[k], outs[k])
        run_done[k].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(run_done[k])
            for h, o in zip(host_outs[k], outs[k]):
                h.copy_(o, non_blocking=True)
            down_done[k].record(s_down)
        used[k] = True

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_up)
    s_down.wait_stream(s_up)
    stream.wait_stream(s_up)
    for i in range(steps):
        one(i)
    s_up.wait_stream(s_down)
    s_up.wait_stream(stream)
    t1.record(s_up)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    h2d = sum(h.numel() * h.element_size() for h in hosts)
    d2h = sum(o.numel() * o.element_size() for o in host_outs[0])
    return ms, h2d, d2h


def pinned(t):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t.cpu())
    return h


def e2e_measure(step, steps, stream):
    """The step through the C ABI from pinned host buffers (see pipelined_e2e).

    Prefill: every step uploads Q/K/V (the packed QKV buffer when the workload has one)
    and downloads the output and lse.  Chunked prefill: the query chunk and the caches.
    Producer: the fused QKV rows up, the attention input down (the cache rows stay on the
    device for the attention kernels).  Decode: the cache is device-resident state; every
    step uploads the query, the step's new K/V row, its cache position and the lengths,
    appends the row (lat_kv_append, or lat_kv_append_ring for a ring cache), decodes and
    downloads the output and lse."""
    b = step.b
    if isinstance(step, DecodeStep):
        wl, d = step.wl, step.di
        lens = d.kv_lens.long()
        rows = torch.arange(wl.B, device=lens.device)
        slot = (lens - 1) % wl.ring if wl.ring else lens - 1
        # the new row re-writes the cache row it lands on, so the cache stays unchanged
        k_new = d.k_cache[rows, slot].contiguous()
        v_new = d.v_cache[rows, slot].contiguous()
        pos = (d.kv_lens - 1).to(torch.int32)
        hosts = [pinned(x) for x in (d.q, k_new, v_new, pos, d.kv_lens)]
        row_w = wl.Hkv * wl.D

        def run(dv, outs):
            q, kn, vn, ps, kl = dv
            if wl.ring:
                b.lat_kv_append_ring(step.dt, d.k_cache, d.v_cache, row_w, wl.D,
                                     wl.L * row_w, wl.ring, kn, vn, row_w, ps, 1, wl.B,
                                     wl.Hkv, wl.D, step.status)
            else:
                b.lat_kv_append(step.dt, d.k_cache, d.v_cache, row_w, wl.D, wl.L * row_w,
                                wl.L, kn, vn, row_w, ps, 1, wl.B, wl.Hkv, wl.D, step.status)
            step.out, step.lse = outs
            step(q, d.k_cache, d.v_cache, kl)
        out_like = [step.out, step.lse]
    else:
        if isinstance(step, PrefillStep):
            inp = step.inp
            parents = ([inp.packed] if inp.packed is not None else
                       [inp.q.contiguous(), inp.k.contiguous(), inp.v.contiguous()])
            out_names = ("out", "lse")
        elif isinstance(step, PrefillCachedStep):
            parents = [step.q, step.di.k_cache, step.di.v_cache]
            out_names = ("out", "lse")
        else:  # ProducerStep
            parents = [step.qkv]
            out_names = ("q_out",)
        hosts = [pinned(p) for p in parents]
        out_like = [getattr(step, n) for n in out_names]

        def run(dv, outs):
            for n, o in zip(out_names, outs):
                setattr(step, n, o)
            if isinstance(step, PrefillStep) and step.inp.packed is not None:
                qw, kw = step.wl.Hq * step.wl.D, step.wl.Hkv * step.wl.D
                buf = dv[0]
                step(buf[:, :qw], buf[:, qw:qw + kw], buf[:, qw + kw:])
            else:
                step(*dv)
    keep = {n: getattr(step, n) for n in ("out", "lse", "q_out") if hasattr(step, n)}
    try:
        return pipelined_e2e(hosts, out_like, run, steps, stream)
    finally:
        for n, o in keep.items():
            setattr(step, n, o)


# ------------------------------------------------------------------------------ CPU arm

def row_pairs(wl, rows):
    """Visible (query, key) pairs of each flattened query row r = b*S + i, per head."""
    i = np.asarray(rows, dtype=np.int64) % wl.S
    p = i + (wl.L - wl.S)
    hi = np.minimum(wl.L, p + 1) if wl.causal else np.full(i.shape, wl.L, dtype=np.int64)
    lo = np.maximum(0, p - wl.window + 1) if wl.window > 0 else np.zeros(i.shape, np.int64)
    return np.maximum(hi - lo, 0)


class OracleSample:
    """A deterministic sample of one workload for the fp64 oracle, with the exact share
    of the workload's algorithmic work it carries.

    Prefill: the query rows of W.sample_rows (the first and last 4 rows of every
    sequence, the rows around the window edge, `n_random` seeded rows), every head;
    work = 4*D*Hq * (visible pairs of those rows).  Decode: the first `n_seq` sequences
    at their drawn lengths, every head; work = their visible K/V bytes.  The inputs are
    converted to float64 once, before any timing."""

    def __init__(self, wl, n_random=256, n_seq=4):
        import oracle
        oracle.build_library()
        self.oracle = oracle
        self.wl = wl
        self.threads = oracle.default_threads()
        if wl.kind in ("prefill", "prefill_cached"):
            inp = W.prefill_inputs(wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D, dtype=wl.dtype,
                                   device="cpu", k_mul=wl.k_mul)
            self.q, self.k, self.v = (np.ascontiguousarray(inp.heads(x).double().numpy())
                                      for x in ("q", "k", "v"))
            extra = (wl.window - 1, wl.window, wl.window + 1) if wl.window > 0 else ()
            self.rows = W.sample_rows(wl.B * wl.S, wl.S, extra=extra, n_random=n_random)
            pairs = int(row_pairs(wl, self.rows).sum())
            total = visible_pairs(wl.S, wl.L, wl.causal, wl.window) * wl.B
            self.work = 4.0 * wl.D * wl.Hq * pairs / 1e12          # TFLOP
            self.unit = "TFLOP/s"
            self.share = pairs / total
            self.what = ("%d of %d query rows x %d heads (%d of %d visible pairs per head)"
                         % (len(self.rows), wl.B * wl.S, wl.Hq, pairs, total))
        else:
            if wl.ring:
                lens = W.ring_decode_inputs(wl.B, wl.Hq, wl.Hkv, wl.D, 1, wl.max_len).kv_lens
            else:
                lens = W.decode_inputs(wl.B, 1, 1, 8, max(wl.L, 1), kv_lens=wl.kv_lens,
                                       nan_fill=False).kv_lens
            lens = [int(x) for x in lens.tolist()]
            vis = [min(n, wl.window) if wl.window > 0 else n for n in lens]
            n = min(n_seq, wl.B)
            self.vis = vis[:n]
            mx = max(max(self.vis), 1)
            g = np.random.default_rng(W.BASE_SEED)
            self.q = g.standard_normal((n, wl.Hq, wl.D))
            self.kc = g.standard_normal((n, mx, wl.Hkv, wl.D))
            self.vc = g.standard_normal((n, mx, wl.Hkv, wl.D))
            es = 2 if wl.dtype == "bf16" else 4
            sample_keys = sum(self.vis)
            self.work = sample_keys * wl.Hkv * wl.D * 2 * es / 1e9    # GB of K/V
            self.unit = "GB/s"
            self.share = sample_keys / max(sum(vis), 1)
            self.what = ("%d of %d sequences (%d of %d visible keys) x %d KV heads"
                         % (n, wl.B, sample_keys, sum(vis), wl.Hkv))

    def run(self):
        wl, o = self.wl, self.oracle
        if wl.kind in ("prefill", "prefill_cached"):
            o.prefill(self.q, self.k, self.v, causal=wl.causal, window=wl.window,
                      scale=wl.scale, rows=self.rows, threads=self.threads,
                      softcap=wl.softcap)
        else:
            o.decode(self.q, self.kc, self.vc, self.vis, window=0, scale=wl.scale,
                     threads=self.threads)


def cpu_baseline(wl, seconds=10.0):
    """The oracle as it stands, on all host cores, over passes of a fixed sample of the
    workload (repeated until `seconds` have run)."""
    smp = OracleSample(wl)
    n, t0 = 0, time.perf_counter()
    while True:
        smp.run()
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    value = smp.work * n / dt
    return {"value": value, "unit": smp.unit, "cores": smp.threads, "kind": "oracle",
            "sample": "%d passes over %s of %s (fp64 oracle, %d threads, %.1f s); the sample "
                      "is %.4f of the workload's work, so a whole pass would take %.1f s"
                      % (n, smp.what, wl.name, smp.threads, dt, smp.share,
                         dt / n / smp.share)}


def run_reference(args, rank, world):
    """--impl reference: the oracle is the timed arm (rank 0 only); each step is one pass
    over the workload's oracle sample."""
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload]
    smp = OracleSample(wl, n_random=128)  # a step of a second or two on 16 cores
    for _ in range(args.warmup):
        smp.run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        smp.run()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = smp.work / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": smp.unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": smp.unit, "cores": smp.threads,
                         "kind": "oracle",
                         "sample": "each step is one pass over %s of %s (%.4f of the "
                                   "workload's work)" % (smp.what, wl.name, smp.share)},
        "e2e": {"value": value, "unit": smp.unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl):
    if wl.kind == "decode":
        lens = "uniform[1,%d]" % (wl.max_len if wl.ring else wl.L) if wl.kv_lens is None \
            else str(wl.kv_lens)
        return {"workload": "%s: decode B%d Hq%d Hkv%d D%d %s %d, kv_len %s%s %s" % (
            wl.name, wl.B, wl.Hq, wl.Hkv, wl.D, "ring cache" if wl.ring else "cache", wl.L,
            lens, " window %d" % wl.window if wl.window else "", wl.dtype),
            "batch": wl.B, "kv_capacity": wl.L, "n_heads": wl.Hq, "n_kv_heads": wl.Hkv,
            "head_dim": wl.D, "window": wl.window,
            "l2": L2_NOTE, "parallelism": "replicas"}
    if wl.kind == "producer":
        return {"workload": "%s: Q/K RMS norm + neox RoPE + cache append, %d rows of a fused "
                            "QKV [%d, %d], Hq%d Hkv%d D%d, token-major cache %d slots %s" % (
                                wl.name, wl.B * wl.S, wl.B * wl.S,
                                (wl.Hq + 2 * wl.Hkv) * wl.D, wl.Hq, wl.Hkv, wl.D, wl.cap,
                                wl.dtype),
                "batch": wl.B, "seq_len": wl.S, "n_heads": wl.Hq, "n_kv_heads": wl.Hkv,
                "head_dim": wl.D, "l2": L2_NOTE, "parallelism": "replicas"}
    where = ""
    if wl.packed:
        where = ", packed QKV [%d, %d]" % (wl.B * wl.S, (wl.Hq + 2 * wl.Hkv) * wl.D)
    elif wl.kind == "prefill_cached":
        where = ", K/V from a token-major cache [%d, %d, %d] (kv_len %d)" % (
            wl.B, wl.cap, wl.Hkv * wl.D, wl.L)
    return {"workload": "%s: B%d S%d Hq%d Hkv%d D%d %s%s %s%s" % (
        wl.name, wl.B, wl.S, wl.Hq, wl.Hkv, wl.D, "causal" if wl.causal else "full",
        " window %d" % wl.window if wl.window else "", wl.dtype,
        where + (", softcap %g" % wl.softcap if wl.softcap else "")),
        "batch": wl.B, "seq_len": wl.S, "kv_len": wl.L, "n_heads": wl.Hq, "n_kv_heads": wl.Hkv,
        "head_dim": wl.D, "causal": wl.causal, "window": wl.window,
        "l2": L2_NOTE,
        "parallelism": "replicas"}


# ------------------------------------------------------------------------------ main

def kernel_info(wl, step, peaks):
    """(algorithmic flops, bytes, work in the value's unit, unit, kernel name, roofline
    bound, ncu summary name, kernel sources) of one workload."""
    if wl.kind in ("prefill", "prefill_cached"):
        flops, alg_bytes, _ = prefill_work(wl)
        return (flops, alg_bytes, flops / 1e12, "TFLOP/s", "prefill_tc_kernel<%d>" % wl.D,
                prefill_bound(wl, peaks), "prefill_tc_%s.md" % wl.name,
                ["prefill_tc.cu", "device_common.cuh", "kernels.h"])
    if wl.kind == "producer":
        alg_bytes = producer_bytes(wl)
        return (0.0, alg_bytes, alg_bytes / 1e9, "GB/s", "qkv_producer_fast<%d>" % wl.D, "hbm",
                "qkv_producer_%s.md" % wl.name,
                ["qkv_producer.cu", "device_common.cuh", "kernels.h"])
    flops, alg_bytes, _ = decode_work(wl, step.di.kv_lens.cpu().tolist())
    return (flops, alg_bytes, alg_bytes / 1e9, "GB/s", "decode_bf16_kernel<%d>" % wl.D, "hbm",
            "decode_bf16_%s.md" % wl.name, ["decode_bf16.cu", "device_common.cuh", "kernels.h"])


def launches_per_step(wl, device):
    """The library's kernel launches in one timed step: one, plus the deferred split-KV
    merge for decode shapes whose units are too few to keep every CTA streaming (the
    plan's rule: more than 8 pieces per unit needed, at the kernel's CTAs per SM)."""
    if wl.kind != "decode" or wl.dtype != "bf16":
        return 1
    ctas_per_sm = {64: 3, 80: 2, 128: 2, 256: 2, 512: 1}[wl.D]
    grid = torch.cuda.get_device_properties(device).multi_processor_count * ctas_per_sm
    units = wl.B * wl.Hkv * ((wl.Hq // wl.Hkv + 7) // 8)
    return 2 if -(-grid // units) > 8 else 1


def measure_main(wl, device, flush, stream, peaks, peak_src, args, world, dist):
    """Warm-up, the timed steps (max over ranks), roofline and e2e of one workload."""
    step = {"prefill": PrefillStep, "prefill_cached": PrefillCachedStep,
            "decode": DecodeStep, "producer": ProducerStep}[wl.kind](wl, device)
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    step.check_status()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ms_steps = time_steps(step, args.steps, flush, stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    step.check_status()
    flops, alg_bytes, work, unit, kernel, bound, profile, srcs = kernel_info(wl, step, peaks)
    ms_total, _ = replica_throughput(sum(ms_steps), work, world, dist, device)
    ms_per_step, value = replica_throughput(ms_total / args.steps, work, world)

    e2e_ms, h2d, d2h = e2e_measure(step, args.steps, stream)
    step.check_status()
    e2e_ms, e2e_value = replica_throughput(e2e_ms, work, world, dist, device)

    kernel_ms = statistics.mean(ms_steps)
    tflops = flops / (kernel_ms / 1e3) / 1e12
    if bound == "hbm":
        achieved, peak, r_unit = alg_bytes / (kernel_ms / 1e3) / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, r_unit = tflops, peaks["bf16_tflops"], "TFLOP/s"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": r_unit,
                "frac": achieved / peak, "traffic": profile_traffic(profile, srcs),
                "kernel": kernel, "peak_source": peak_src, "algorithmic_bytes": alg_bytes,
                "algorithmic_flops": flops,
                "tensor_frac": tflops / peaks["bf16_tflops"],
                "hbm_frac": alg_bytes / (kernel_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
    e2e = {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
    # our kernels inside the timed region (the flush is torch's)
    return {"value": value, "unit": unit, "ms_per_step": ms_per_step, "roofline": roofline,
            "e2e": e2e, "gpu_launches": args.steps * launches_per_step(wl, device)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)

    if args.impl == "reference":
        run_reference(args, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return

    from gqa_attention_lat_gb300.build import build_library
    if rank == 0 or world == 1:
        build_library()
    if dist is not None:
        dist.barrier()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    peaks, peak_src = load_peaks()
    wl = W.WORKLOADS[args.workload]
    if wl.dtype != "bf16":
        raise SystemExit("bench workloads are bf16 (the fp32 shapes are parity cases)")
    flush = Flusher(device)
    sampler = ClockSampler(local)
    sampler.start()
    head = measure_main(wl, device, flush, stream, peaks, peak_src, args, world, dist)
    torch.cuda.empty_cache()
    # the headline layer's decode step beside it
    comp = None
    if args.workload == HEADLINE:
        cwl = W.WORKLOADS[COMPANION]
        comp = measure_main(cwl, device, flush, stream, peaks, peak_src, args, world, dist)
        comp["workload"] = workload_config(cwl)["workload"]
        torch.cuda.empty_cache()
    extra = None
    if not args.no_extra:
        extra = measure_extra(device, flush, stream, peaks,
                              skip=(args.workload, COMPANION if comp else None))
    clocks = sampler.stop()

    if not args.no_cpu and rank == 0 and world == 1:
        head["cpu_baseline"] = cpu_baseline(wl)
        if comp is not None:
            comp["cpu_baseline"] = cpu_baseline(W.WORKLOADS[COMPANION])
    else:
        head["cpu_baseline"] = None

    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": workload_config(wl),
        "roofline": head["roofline"],
        "cpu_baseline": head["cpu_baseline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": clocks,
        "decode": comp,
        "workloads": extra,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
