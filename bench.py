"""Benchmark of the fused GQA attention path on GB300.

Headline (one JSON line on stdout, rank 0): single-token GQA decode at
Qwen2.5-7B head geometry (B=1, Hq=28, Hkv=4, D=128), kv_len 32,768, fp32 KV
cache, 28 layer calls on 28 distinct layer buffers per step.  Metric: decode
K/V GB/s (algorithmic Q+K+V+O bytes / time), with its fraction of the measured
HBM copy bandwidth.  The other rows of the hot path (the kv_len sweep in fp32
and bf16, ragged batched decode, 4-bit decode, causal and chunked prefill) are
measured in the same run and reported as sub-objects of the line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gqa|reference]
    python bench.py --kernel CASE --steps K --warmup W   # one launch configuration

Timing: CUDA events on the launching stream, W untimed warm-up steps, K timed
steps bracketed by a barrier and a device synchronise; the inputs of one step
(3.76 GB) are far larger than L2, so nothing is reused between steps.  For
N > 1 (torchrun) every rank runs its own replica (weak scaling) and the time
is the max over ranks.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gqa_attention_kv_decode_gb300 import inputs, metrics  # noqa: E402

HQ, HKV, D, LAYERS, S_HEAD = 28, 4, 128, 28, 32768
METRIC = "GQA decode-attend KV GB/s (% of HBM peak); causal prefill TFLOP/s"
WORKLOAD = ("single-token GQA decode, Qwen2.5-7B head geometry: B=1, Hq=28, Hkv=4, D=128, "
            "kv_len=32768, fp32 KV cache, 28 layer calls on distinct buffers per step")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def replica_value(world: int, step_units: float, ms_per_step: float) -> float:
    """Whole-job rate in units/s / 1e9 (GB/s for bytes): every one of the
    `world` replicas processes `step_units` per step, and the step time is the
    maximum over ranks."""
    return world * step_units / (ms_per_step * 1e-3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Dist:
    """Barrier and max-over-ranks for replica timing (gloo, host-side only)."""

    def __init__(self, world):
        self.world = world
        if world > 1:
            import torch.distributed as td
            td.init_process_group("gloo")
            self.td = td

    def barrier(self):
        if self.world > 1:
            self.td.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64)
        self.td.all_reduce(t, op=self.td.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            self.td.destroy_process_group()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="gqa_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_hash(name):
    """Hash of a kernel source with its // comments and blank lines left out,
    so that a comment edit does not retire an ncu record of unchanged code."""
    with open(os.path.join(ROOT, "gqa_attention_kv_decode_gb300", "csrc", name)) as f:
        lines = (line.split("//", 1)[0].rstrip() for line in f)
        code = "\n".join(line for line in lines if line)
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def recorded_ncu(kernel_file, key):
    """The committed ncu record of one kernel (DRAM bytes and duration per
    launch), if the kernel source is unchanged since it was captured (else
    None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[key]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_sha256_16") != kernel_source_hash(kernel_file):
        return None
    return rec


def recorded_traffic(kernel_file, key):
    """Per-launch DRAM bytes from the committed ncu summary (or None)."""
    rec = recorded_ncu(kernel_file, key)
    return None if rec is None else rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- decode workload

def make_layers(S, dtype, device, n_layers=LAYERS, B=1, hq=HQ, hkv=HKV, d=D):
    return [inputs.qkv(B, hq, hkv, d, 1, S, dtype, layer=l, device=device) for l in range(n_layers)]


def time_decode_step(binding, layers, outs, ws, S, stream, evs=None):
    """One step: the 28 layer calls.  With `evs`, each launch is bracketed
    by events (start, end) appended to the list."""
    scale = D ** -0.5
    for (q, k, v), o in zip(layers, outs):
        if evs is not None:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        binding.gqa_attn_decode(q, k, v, o, None, scale, ws, max_kv_len=S, stream=stream)
        if evs is not None:
            e1.record(stream)
            evs.append((e0, e1))


def flush_l2(buf):
    buf.add_(1)


def sweep_point(binding, S, dtype, device, stream, flush, iters=20, graph=True):
    """µs per layer call for 28 calls at kv_len S (cold L2 per sequence)."""
    layers = make_layers(S, dtype, device)
    outs = [torch.empty_like(q) for q, _, _ in layers]
    ws = binding.decode_workspace(1, HQ, HKV, D, S, binding._dtype_code(layers[0][0]), device)
    torch.cuda.synchronize()  # inputs are made on the default stream; time on `stream` only after
    with torch.cuda.stream(stream):
        for _ in range(3):
            time_decode_step(binding, layers, outs, ws, S, stream)
    res = {}
    modes = ["launch"]
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            time_decode_step(binding, layers, outs, ws, S, stream)
        modes.append("graph")
    for mode in modes:
        ts = []
        for _ in range(iters):
            with torch.cuda.stream(stream):
                flush_l2(flush)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if mode == "graph":
                    g.replay()
                else:
                    time_decode_step(binding, layers, outs, ws, S, stream)
                e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / LAYERS)
        us = statistics.median(ts)
        nbytes = metrics.decode_bytes(HQ, HKV, D, [S], layers[0][0].element_size())
        res[mode] = {"us_per_call": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
                     "p10_us": round(float(np.percentile(ts, 10)), 3),
                     "p90_us": round(float(np.percentile(ts, 90)), 3)}
    del layers, outs, ws, g
    torch.cuda.empty_cache()
    return res


def capacity_points(binding, lens, device, stream, flush, iters=20, cap=32768):
    """fp32, 7B geometry, 28 layer calls in a CUDA graph on a cache of `cap`
    rows holding L keys: the call planned for the capacity (max_kv_len = cap,
    what a graph replayed over many decode steps is captured with) against
    the call planned for the length itself (max_kv_len = L)."""
    layers = make_layers(cap, torch.float32, device)
    outs = [torch.empty_like(q) for q, _, _ in layers]
    res = []
    for L in lens:
        lens_t = torch.tensor([L], dtype=torch.int32, device=device)
        row = {"L": L, "capacity": cap}
        for key, mkl in (("planned_for_capacity", cap), ("planned_for_L", L)):
            ws = binding.decode_workspace(1, HQ, HKV, D, mkl, binding.GQA_F32, device)
            torch.cuda.synchronize()

            def step():
                for (q, k, v), o in zip(layers, outs):
                    binding.gqa_attn_decode(q, k, v, o, lens_t, D ** -0.5, ws, max_kv_len=mkl, stream=stream)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    step()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            ts = []
            for _ in range(iters):
                with torch.cuda.stream(stream):
                    flush_l2(flush)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3 / LAYERS)
            us = statistics.median(ts)
            nbytes = metrics.decode_bytes(HQ, HKV, D, [L], 4)
            row[key] = {"us_per_call": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
                        "n_split": binding.gqa_attn_decode_num_splits(1, HQ, HKV, D, mkl, binding.GQA_F32)}
            del g, ws
        res.append(row)
    del layers, outs
    torch.cuda.empty_cache()
    return res


def ragged_point(binding, B, device, stream, flush, iters=10):
    """Hq=32, Hkv=8, D=128, bf16, lengths uniform in [64, 8192], 36 layers."""
    kv_lens = inputs.ragged_kv_lens(B, 64, 8192, seed=inputs.BASE_SEED + B)
    lens_t = torch.from_numpy(kv_lens).to(device)
    n_layers = 36
    layers = make_layers(8192, torch.bfloat16, device, n_layers=n_layers, B=B, hq=32, hkv=8)
    outs = [torch.empty_like(q) for q, _, _ in layers]
    ws = binding.decode_workspace(B, 32, 8, 128, 8192, binding.GQA_BF16, device)
    torch.cuda.synchronize()

    def step():
        for (q, k, v), o in zip(layers, outs):
            binding.gqa_attn_decode(q, k, v, o, lens_t, 128 ** -0.5, ws, max_kv_len=8192, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    ts = []
    for _ in range(iters):
        with torch.cuda.stream(stream):
            flush_l2(flush)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / n_layers)
    us = statistics.median(ts)
    nbytes = metrics.decode_bytes(32, 8, 128, kv_lens, 2)
    del layers, outs
    torch.cuda.empty_cache()
    return {"B": B, "us_per_call": round(us, 3), "GBps": round(nbytes / us / 1e3, 1)}


def paged_point(binding, B, device, stream, flush, iters=10, block_size=64):
    """The ragged workload above on a paged cache (block size 64, blocks in a
    random order in the pool) with the new token of every request appended
    inside the call: Hq=32, Hkv=8, D=128, bf16, 36 layers."""
    kv_lens = inputs.ragged_kv_lens(B, 64, 8192, seed=inputs.BASE_SEED + B)
    lens_t = torch.from_numpy(kv_lens).to(device)
    n_layers, hkv, D = 36, 8, 128
    nbs = [-(-int(L) // block_size) for L in kv_lens]
    max_blocks = 8192 // block_size  # the table spans max_kv_len; entries past a request's blocks are unused
    layers = []
    for l in range(n_layers):
        n_pool = sum(nbs) + 4
        kp = inputs.randn((n_pool, hkv, block_size, D), inputs.tensor_seed(l, 1), torch.bfloat16, device)
        vp = inputs.randn((n_pool, hkv, block_size, D), inputs.tensor_seed(l, 2), torch.bfloat16, device)
        perm = torch.from_numpy(np.random.default_rng(l).permutation(n_pool).astype(np.int32))
        table = torch.zeros((B, max_blocks), dtype=torch.int32)
        at = 0
        for b, nb in enumerate(nbs):
            table[b, :nb] = perm[at:at + nb]
            at += nb
        q = inputs.randn((B, 32, 1, D), inputs.tensor_seed(l, 0), torch.bfloat16, device)
        kn = inputs.randn((B, hkv, 1, D), inputs.tensor_seed(l, 3), torch.bfloat16, device)
        vn = inputs.randn((B, hkv, 1, D), inputs.tensor_seed(l, 4), torch.bfloat16, device)
        layers.append((q, kp, vp, table.to(device), kn, vn))
    outs = [torch.empty_like(x[0]) for x in layers]
    ws = binding.decode_workspace(B, 32, hkv, D, 8192, binding.GQA_BF16, device)
    torch.cuda.synchronize()

    def step():
        for (q, kp, vp, table, kn, vn), o in zip(layers, outs):
            binding.gqa_attn_decode_paged(q, kn, vn, kp, vp, table, lens_t, o, D ** -0.5, ws, 8192,
                                          stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    ts = []
    for _ in range(iters):
        with torch.cuda.stream(stream):
            flush_l2(flush)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / n_layers)
    us = statistics.median(ts)
    # Q, K, V of the valid rows and O, plus the appended token (read, then
    # written into the pools)
    nbytes = metrics.decode_bytes(32, hkv, D, kv_lens, 2) + 4 * B * hkv * D * 2
    del layers, outs
    torch.cuda.empty_cache()
    return {"B": B, "block_size": block_size, "us_per_call": round(us, 3),
            "GBps": round(nbytes / us / 1e3, 1)}


PREFILL_LAYERS = 24  # Qwen2.5-0.5B: one prefill step is this many layer launches


def varlen_prefill_point(binding, B, device, stream, flush, bf16_peak, iters=8, chunk=512, NL=PREFILL_LAYERS):
    """Serving-style chunked prefill of B requests at once (Hq=14, Hkv=2,
    D=64, bf16, causal): request b prefills a chunk of `chunk` queries at the
    end of its kv_lens[b] keys, kv_lens uniform in [chunk, 8192] (seeded).
    Timed like prefill_point: NL launches on distinct buffers per step."""
    kv_lens = inputs.ragged_kv_lens(B, chunk, 8192, seed=inputs.BASE_SEED + 7 * B)
    S = int(kv_lens.max())
    layers = []
    for l in range(NL):
        q = inputs.randn((B, 14, chunk, 64), inputs.tensor_seed(l, 0), torch.bfloat16, device)
        k = inputs.randn((B, 2, S, 64), inputs.tensor_seed(l, 1), torch.bfloat16, device)
        v = inputs.randn((B, 2, S, 64), inputs.tensor_seed(l, 2), torch.bfloat16, device)
        layers.append((q, k, v, torch.empty_like(q)))
    ql = torch.full((B,), chunk, dtype=torch.int32, device=device)
    kl = torch.from_numpy(kv_lens).to(device)
    torch.cuda.synchronize()

    def step():
        for q, k, v, o in layers:
            binding.gqa_attn_prefill_varlen(q, k, v, o, ql, kl, 0.125, True, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(iters):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            flush_l2(flush)
            e0.record(stream)
            step()
            e1.record(stream)
            evs.append((e0, e1))
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs) / NL
    flops = sum(metrics.prefill_flops(14, 64, chunk, int(L), causal=True) for L in kv_lens)
    tf = flops / us / 1e6
    del layers
    torch.cuda.empty_cache()
    return {"requests": B, "chunk": chunk, "layers": NL, "us": round(us, 2), "TFLOPs": round(tf, 1),
            "tokens_per_s": round(B * chunk / us * 1e6, 1), "frac_of_bf16_peak": round(tf / bf16_peak, 4)}


def layers_point(binding, S, device, stream, flush, iters=10, NL=28):
    """Qwen2.5-7B head geometry, fp32, B=1: NL layers as NL gqa_attn_decode
    calls versus one gqa_attn_decode_layers launch over the stacked layers
    (the pages' cross-layer batching; a microbenchmark of the per-call cost)."""
    q = inputs.randn((NL, 1, HQ, 1, D), inputs.tensor_seed(0, 0), torch.float32, device)
    k = inputs.randn((NL, 1, HKV, S, D), inputs.tensor_seed(0, 1), torch.float32, device)
    v = inputs.randn((NL, 1, HKV, S, D), inputs.tensor_seed(0, 2), torch.float32, device)
    o = torch.empty_like(q)
    ws_l = torch.zeros(binding.gqa_attn_decode_layers_workspace_size(NL, 1, HQ, HKV, D, S, binding.GQA_F32),
                       dtype=torch.uint8, device=device)
    ws_1 = binding.decode_workspace(1, HQ, HKV, D, S, binding.GQA_F32, device)
    torch.cuda.synchronize()
    views = [(q[l], k[l], v[l], o[l]) for l in range(NL)]  # slicing stays out of the timed region
    seq = lambda: [binding.gqa_attn_decode(ql, kl, vl, ol, None, D ** -0.5, ws_1, max_kv_len=S, stream=stream)
                   for ql, kl, vl, ol in views]
    one = lambda: binding.gqa_attn_decode_layers(q, k, v, o, None, D ** -0.5, ws_l, max_kv_len=S, stream=stream)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        ts = []
        for _ in range(iters):
            with torch.cuda.stream(stream):
                flush_l2(flush)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / NL)
        return statistics.median(ts)
    us_seq, us_one = timed(seq), timed(one)
    nbytes = metrics.decode_bytes(HQ, HKV, D, [S], 4)
    del q, k, v, o, views
    torch.cuda.empty_cache()
    return {"S": S, "layers": NL, "per_layer_calls_us": round(us_seq, 3), "one_launch_us_per_layer": round(us_one, 3),
            "one_launch_GBps": round(nbytes / us_one / 1e3, 1)}


def q4_residual_point(binding, S, device, stream, flush, iters=10, window=100, R_cap=128):
    """q4 decode (Hq=32, Hkv=8, D=128, B=4, 36 layers) with `window` further
    tokens in a bf16 residual window: S quantized keys + the window."""
    B, n_layers = 4, 36
    layers = []
    for l in range(n_layers):
        cache = inputs.q4_cache(B, 8, 128, S, layer=l, device=device)
        kr = inputs.randn((B, 8, R_cap, 128), inputs.tensor_seed(l, 5), torch.bfloat16, device)
        vr = inputs.randn((B, 8, R_cap, 128), inputs.tensor_seed(l, 6), torch.bfloat16, device)
        q = inputs.randn((B, 32, 1, 128), inputs.tensor_seed(l, 0), torch.bfloat16, device)
        layers.append((q, cache, kr, vr))
    outs = [torch.empty_like(x[0]) for x in layers]
    nq = torch.full((B,), S, dtype=torch.int32, device=device)
    lens = torch.full((B,), S + window, dtype=torch.int32, device=device)
    ws = torch.zeros(binding.gqa_attn_decode_q4_residual_workspace_size(B, 32, 8, 128, S), dtype=torch.uint8,
                     device=device)
    torch.cuda.synchronize()

    def step():
        for (q, cache, kr, vr), o in zip(layers, outs):
            binding.gqa_attn_decode_q4_residual(q, *cache, kr, vr, nq, lens, o, 128 ** -0.5, ws, max_quant=S,
                                                stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    ts = []
    for _ in range(iters):
        with torch.cuda.stream(stream):
            flush_l2(flush)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / n_layers)
    us = statistics.median(ts)
    nbytes = metrics.q4_decode_bytes(32, 8, 128, [S] * B) + 2 * B * 8 * window * 128 * 2
    del layers, outs
    torch.cuda.empty_cache()
    return {"S_quantized": S, "window": window, "us_per_call": round(us, 3), "GBps": round(nbytes / us / 1e3, 1)}


def quantize_point(binding, device, stream, flush, iters=10):
    """4-bit quantization of KV rows (Hkv=8, D=128, B=4): a whole 16384-token K
    cache in one call (HBM-bound), and the per-step flush of one aged block of
    64 tokens of K and of V (launch-bound) over 36 layers."""
    B, hkv, D, S = 4, 8, 128, 16384
    x = inputs.randn((B, hkv, S, D), inputs.tensor_seed(0, 1), torch.bfloat16, device)
    codes = torch.empty((B, hkv, S, D // 2), dtype=torch.uint8, device=device)
    scale = torch.empty((B, hkv, S, D // 64), dtype=torch.float16, device=device)
    bias = torch.empty_like(scale)
    blocks = [inputs.randn((B, hkv, 64, D), inputs.tensor_seed(l, 5 + t), torch.bfloat16, device)
              for l in range(36) for t in range(2)]
    torch.cuda.synchronize()

    def timed(fn, n):
        ts = []
        for _ in range(iters):
            with torch.cuda.stream(stream):
                flush_l2(flush)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / n)
        return statistics.median(ts)
    full = lambda: binding.gqa_attn_quantize_q4(x, codes, scale, bias, stream=stream)
    step = lambda: [binding.gqa_attn_quantize_q4(blk, codes, scale, bias, dst_row0=8192, stream=stream)
                    for blk in blocks]
    with torch.cuda.stream(stream):
        for _ in range(3):
            full()
            step()
    us_full = timed(full, 1)
    us_flush = timed(step, 36)
    rows = B * hkv * S
    nbytes = metrics.quantize_bytes(rows, D)
    del x, codes, scale, bias, blocks
    torch.cuda.empty_cache()
    return {"full_cache_B4_S16384": {"us": round(us_full, 3), "GBps": round(nbytes / us_full / 1e3, 1)},
            "flush_64_tokens_K_and_V": {"us_per_layer": round(us_flush, 3)}}


def q4_point(binding, S, device, stream, flush, iters=10):
    """Hq=32, Hkv=8, D=128, B=4, 4-bit group-affine cache, 36 layer calls."""
    B, n_layers = 4, 36
    layers = []
    for l in range(n_layers):
        cache = inputs.q4_cache(B, 8, 128, S, layer=l, device=device)
        q = inputs.randn((B, 32, 1, 128), inputs.tensor_seed(l, 0), torch.bfloat16, device)
        layers.append((q, cache))
    outs = [torch.empty_like(q) for q, _ in layers]
    ws = binding.decode_q4_workspace(B, 32, 8, 128, S, device)
    torch.cuda.synchronize()

    def step():
        for (q, cache), o in zip(layers, outs):
            binding.gqa_attn_decode_q4(q, *cache, o, None, 128 ** -0.5, ws, max_kv_len=S, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    ts = []
    for _ in range(iters):
        with torch.cuda.stream(stream):
            flush_l2(flush)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / n_layers)
    us = statistics.median(ts)
    nbytes = metrics.q4_decode_bytes(32, 8, 128, [S] * B)
    del layers, outs
    torch.cuda.empty_cache()
    return {"S": S, "us_per_call": round(us, 3), "GBps": round(nbytes / us / 1e3, 1)}


def prefill_point(binding, q_len, kv_len, device, stream, flush, bf16_peak, iters=8, NL=PREFILL_LAYERS,
                  Hq=14, Hkv=2, D=64):
    """bf16, causal, queries aligned to the end of the keys; head geometry
    Hq=14, Hkv=2, D=64 (Qwen2.5-0.5B) unless given.

    One step is NL launches on NL distinct buffer sets (a prefill through the
    model's layers), timed with one event pair after an L2 flush: no launch
    finds its inputs in L2, and launches follow each other as in a model
    instead of each being bracketed by its own events.  Per-launch time =
    step time / NL (median over the steps)."""
    layers = []
    for l in range(NL):
        q = inputs.randn((1, Hq, q_len, D), inputs.tensor_seed(l, 0), torch.bfloat16, device)
        k = inputs.randn((1, Hkv, kv_len, D), inputs.tensor_seed(l, 1), torch.bfloat16, device)
        v = inputs.randn((1, Hkv, kv_len, D), inputs.tensor_seed(l, 2), torch.bfloat16, device)
        layers.append((q, k, v, torch.empty_like(q)))
    torch.cuda.synchronize()

    def step():
        for q, k, v, o in layers:
            binding.gqa_attn_prefill(q, k, v, o, kv_len, D ** -0.5, True, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(iters):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            flush_l2(flush)
            e0.record(stream)
            step()
            e1.record(stream)
            evs.append((e0, e1))
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs) / NL
    flops = metrics.prefill_flops(Hq, D, q_len, kv_len, causal=True)
    tf = flops / us / 1e6
    del layers
    torch.cuda.empty_cache()
    row = {"q_len": q_len, "kv_len": kv_len, "layers": NL, "us": round(us, 2), "TFLOPs": round(tf, 1),
           "tokens_per_s": round(q_len / us * 1e6, 1), "frac_of_bf16_peak": round(tf / bf16_peak, 4)}
    if (Hq, Hkv, D) != (14, 2, 64):
        row = {"Hq": Hq, "Hkv": Hkv, "D": D, **row}
    return row


# ----------------------------------------------------------------------------- CPU oracle

ORACLE_SAMPLE = ("one KV head group (7 query heads, 1 of 4) of one layer call at kv_len=32768, "
                 "fp32 inputs widened to fp64; GB/s scaled by that sample's algorithmic bytes")
ORACLE_SAMPLES = {
    "decode": ORACLE_SAMPLE,
    "prefill": ("causal prefill at Qwen2.5-0.5B head geometry, T=16384, bf16 inputs widened to fp64: "
                "the last 512 query rows of one query head (each sees about 16,100 keys); "
                "TFLOP/s from that sample's visible (query, key) pairs, 4*D flops each"),
    "q4": ("4-bit decode at Qwen3-4B head geometry, kv_len=16384: one request's KV head group "
           "(4 query heads, 1 of 8 heads x 4 requests), codes dequantised in fp64 then attended; "
           "GB/s scaled by that sample's algorithmic bytes (codes, scales, biases, q, o)"),
}
PF_T, PF_ROWS = 16384, 512
Q4_S = 16384


def _oracle_sample(kind, seed_layer):
    """Inputs of one oracle sample and a function that runs it."""
    import oracle as _oracle
    from gqa_attention_kv_decode_gb300 import inputs as _inputs
    import torch as _torch
    if kind == "decode":
        q, k, v = _inputs.qkv(1, HQ, HKV, D, 1, S_HEAD, _torch.float32, layer=seed_layer)
        qs, ks, vs = q[:, 0:7].numpy(), k[:, 0:1].numpy(), v[:, 0:1].numpy()
        return lambda: _oracle.attention(qs, ks, vs, scale=D ** -0.5)
    if kind == "prefill":
        q, k, v = _inputs.qkv(1, 14, 2, 64, PF_T, PF_T, _torch.bfloat16, layer=seed_layer)
        qs = q[:, 0:1, PF_T - PF_ROWS:].float().numpy()
        ks, vs = k[:, 0:1].float().numpy(), v[:, 0:1].float().numpy()
        return lambda: _oracle.attention(qs, ks, vs, scale=0.125, causal=True)
    if kind == "q4":
        kc, ksc, kb, vc, vsc, vb = _inputs.q4_cache(1, 8, 128, Q4_S, layer=seed_layer)
        q = _inputs.randn((1, 32, 1, 128), _inputs.tensor_seed(seed_layer, 0), _torch.bfloat16)
        qs = q[:, 0:4].float().numpy()
        cache = [t[:, 0:1].contiguous().numpy() for t in (kc, ksc, kb, vc, vsc, vb)]
        return lambda: _oracle.attention_q4(qs, *cache, scale=128 ** -0.5)
    raise ValueError(kind)


def oracle_sample_units(kind):
    """Algorithmic bytes (decode, q4) or flops (prefill) of one sample."""
    if kind == "decode":
        return 2 * 1 * S_HEAD * D * 4 + 2 * 7 * D * 4
    if kind == "prefill":
        pairs = sum(PF_T - PF_ROWS + i + 1 for i in range(PF_ROWS))
        return 4 * 64 * pairs
    if kind == "q4":
        return Q4_S * (64 + 4 + 4) * 2 + 2 * 4 * 128 * 2
    raise ValueError(kind)


def _oracle_sample_worker(kinds, n_steps, seed_layer, starts, conn):
    # one spawned process per host core, single-threaded BLAS (set by the parent)
    for kind in kinds:
        run = _oracle_sample(kind, seed_layer)
        conn.send("ready")
        starts[kind].wait()
        times = []
        for _ in range(n_steps):
            t0 = time.perf_counter()
            run()
            times.append(time.perf_counter() - t0)
        conn.send(times)
    conn.close()


def host_cores():
    return len(os.sched_getaffinity(0))


def cpu_oracle_times(n_steps, workers=1, kinds=("decode",)):
    """Per-step wall time of `workers` oracle processes (one per core, each on
    its own layer's sample, single-threaded, started together), per kind of
    sample: step i takes the slowest worker's i-th sample."""
    import multiprocessing as mp
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"
    out = {}
    try:
        ctx = mp.get_context("spawn")
        starts = {kind: ctx.Event() for kind in kinds}
        procs, pipes = [], []
        for w in range(workers):
            parent, child = ctx.Pipe()
            p = ctx.Process(target=_oracle_sample_worker, args=(tuple(kinds), n_steps, w, starts, child))
            p.start()
            procs.append(p)
            pipes.append(parent)
        for kind in kinds:
            for parent in pipes:
                assert parent.recv() == "ready"
            starts[kind].set()
            per_worker = [parent.recv() for parent in pipes]
            out[kind] = [max(ts[i] for ts in per_worker) for i in range(n_steps)]
        for p in procs:
            p.join()
    finally:
        for k, val in saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val
    return out


def oracle_sample_bytes():
    return oracle_sample_units("decode")


def _oracle_rate(kind, cores, seconds):
    units = cores * oracle_sample_units(kind) / seconds
    return units / 1e12 if kind == "prefill" else units / 1e9


def cpu_baseline(n_steps=3):
    """The oracle on every host core this process may use (one sample per
    core, run together), and on one core: the headline decode sample, and
    beside it a causal-prefill and a 4-bit-decode sample."""
    cores = host_cores()
    kinds = ("decode", "prefill", "q4")
    many = cpu_oracle_times(n_steps, cores, kinds)
    one = cpu_oracle_times(n_steps, 1, kinds)
    res = {}
    for kind in kinds:
        t, t1 = statistics.median(many[kind]), statistics.median(one[kind])
        res[kind] = {"value": round(_oracle_rate(kind, cores, t), 4),
                     "unit": "TFLOP/s" if kind == "prefill" else "GB/s", "cores": cores, "kind": "oracle",
                     "sample": ORACLE_SAMPLES[kind] + f"; {cores} samples (one per core, distinct layers) at "
                                                      f"once, median of {n_steps}",
                     "seconds_per_sample": round(t, 4),
                     "single_core": {"value": round(_oracle_rate(kind, 1, t1), 4), "cores": 1,
                                     "seconds_per_sample": round(t1, 4)}}
    base = dict(res["decode"])
    base["prefill_T16384"] = res["prefill"]
    base["q4_decode_S16384"] = res["q4"]
    return base


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cores = host_cores()
    times = cpu_oracle_times(args.warmup + args.steps, cores)["decode"][args.warmup:]
    t = sum(times) / len(times)
    value = cores * oracle_sample_bytes() / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": ORACLE_SAMPLE + f"; {cores} samples at once, one per core"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": ORACLE_SAMPLE + f"; {cores} samples at once, one per core"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- single-kernel cases

def _case_inputs(name, device):
    """(launch, units, unit_name) for one launch configuration of the path,
    small enough (a few hundred MB on the device) for an ncu capture."""
    if name == "decode-f32-S32768" or name == "decode-bf16-S32768":
        dt = torch.float32 if "f32" in name else torch.bfloat16
        q, k, v = inputs.qkv(1, HQ, HKV, D, 1, S_HEAD, dt, device=device)
        o = torch.empty_like(q)
        ws = binding_mod().decode_workspace(1, HQ, HKV, D, S_HEAD, binding_mod()._dtype_code(q), device)
        nbytes = metrics.decode_bytes(HQ, HKV, D, [S_HEAD], q.element_size())
        return (lambda st: binding_mod().gqa_attn_decode(q, k, v, o, None, D ** -0.5, ws, max_kv_len=S_HEAD,
                                                         stream=st)), nbytes, "bytes"
    if name == "decode-bf16-ragged-B64":
        lens = inputs.ragged_kv_lens(64, 64, 8192, seed=inputs.BASE_SEED + 64)
        lens_t = torch.from_numpy(lens).to(device)
        q, k, v = inputs.qkv(64, 32, 8, 128, 1, 8192, torch.bfloat16, device=device)
        o = torch.empty_like(q)
        ws = binding_mod().decode_workspace(64, 32, 8, 128, 8192, binding_mod().GQA_BF16, device)
        nbytes = metrics.decode_bytes(32, 8, 128, lens, 2)
        return (lambda st: binding_mod().gqa_attn_decode(q, k, v, o, lens_t, 128 ** -0.5, ws, max_kv_len=8192,
                                                         stream=st)), nbytes, "bytes"
    if name == "decode-bf16-paged-B64":
        lens = inputs.ragged_kv_lens(64, 64, 8192, seed=inputs.BASE_SEED + 64)
        lens_t = torch.from_numpy(lens).to(device)
        nbs = [-(-int(L) // 64) for L in lens]
        n_pool = sum(nbs)
        kp = inputs.randn((n_pool, 8, 64, 128), inputs.tensor_seed(0, 1), torch.bfloat16, device)
        vp = inputs.randn((n_pool, 8, 64, 128), inputs.tensor_seed(0, 2), torch.bfloat16, device)
        perm = torch.from_numpy(np.random.default_rng(0).permutation(n_pool).astype(np.int32))
        table = torch.zeros((64, 8192 // 64), dtype=torch.int32)
        at = 0
        for b, nb in enumerate(nbs):
            table[b, :nb] = perm[at:at + nb]
            at += nb
        table = table.to(device)
        q = inputs.randn((64, 32, 1, 128), inputs.tensor_seed(0, 0), torch.bfloat16, device)
        kn = inputs.randn((64, 8, 1, 128), inputs.tensor_seed(0, 3), torch.bfloat16, device)
        vn = inputs.randn((64, 8, 1, 128), inputs.tensor_seed(0, 4), torch.bfloat16, device)
        o = torch.empty_like(q)
        ws = binding_mod().decode_workspace(64, 32, 8, 128, 8192, binding_mod().GQA_BF16, device)
        nbytes = metrics.decode_bytes(32, 8, 128, lens, 2) + 4 * 64 * 8 * 128 * 2
        return (lambda st: binding_mod().gqa_attn_decode_paged(q, kn, vn, kp, vp, table, lens_t, o, 128 ** -0.5,
                                                               ws, 8192, stream=st)), nbytes, "bytes"
    if name == "quantize-B4-S16384":
        x = inputs.randn((4, 8, 16384, 128), inputs.tensor_seed(0, 1), torch.bfloat16, device)
        codes = torch.empty((4, 8, 16384, 64), dtype=torch.uint8, device=device)
        scale = torch.empty((4, 8, 16384, 2), dtype=torch.float16, device=device)
        bias = torch.empty_like(scale)
        nbytes = metrics.quantize_bytes(4 * 8 * 16384, 128)
        return (lambda st: binding_mod().gqa_attn_quantize_q4(x, codes, scale, bias, stream=st)), nbytes, "bytes"
    if name == "q4-B4-S16384":
        S = 16384
        cache = inputs.q4_cache(4, 8, 128, S, device=device)
        q = inputs.randn((4, 32, 1, 128), inputs.tensor_seed(0, 0), torch.bfloat16, device)
        o = torch.empty_like(q)
        ws = binding_mod().decode_q4_workspace(4, 32, 8, 128, S, device)
        nbytes = metrics.q4_decode_bytes(32, 8, 128, [S] * 4)
        return (lambda st: binding_mod().gqa_attn_decode_q4(q, *cache, o, None, 128 ** -0.5, ws, max_kv_len=S,
                                                            stream=st)), nbytes, "bytes"
    if name == "varlen-prefill-B16":
        B, chunk = 16, 512
        kv_lens = inputs.ragged_kv_lens(B, chunk, 8192, seed=inputs.BASE_SEED + 7 * B)
        S = int(kv_lens.max())
        q = inputs.randn((B, 14, chunk, 64), inputs.tensor_seed(0, 0), torch.bfloat16, device)
        k = inputs.randn((B, 2, S, 64), inputs.tensor_seed(0, 1), torch.bfloat16, device)
        v = inputs.randn((B, 2, S, 64), inputs.tensor_seed(0, 2), torch.bfloat16, device)
        o = torch.empty_like(q)
        ql = torch.full((B,), chunk, dtype=torch.int32, device=device)
        kl = torch.from_numpy(kv_lens).to(device)
        flops = sum(metrics.prefill_flops(14, 64, chunk, int(L), causal=True) for L in kv_lens)
        return (lambda st: binding_mod().gqa_attn_prefill_varlen(q, k, v, o, ql, kl, 0.125, True, st)), flops, "flop"
    if name == "decode-f32-layers8-S32768":
        NL = 8
        q = inputs.randn((NL, 1, HQ, 1, D), inputs.tensor_seed(0, 0), torch.float32, device)
        k = inputs.randn((NL, 1, HKV, S_HEAD, D), inputs.tensor_seed(0, 1), torch.float32, device)
        v = inputs.randn((NL, 1, HKV, S_HEAD, D), inputs.tensor_seed(0, 2), torch.float32, device)
        o = torch.empty_like(q)
        ws = torch.zeros(binding_mod().gqa_attn_decode_layers_workspace_size(NL, 1, HQ, HKV, D, S_HEAD,
                                                                              binding_mod().GQA_F32),
                         dtype=torch.uint8, device=device)
        nbytes = NL * metrics.decode_bytes(HQ, HKV, D, [S_HEAD], 4)
        return (lambda st: binding_mod().gqa_attn_decode_layers(q, k, v, o, None, D ** -0.5, ws, max_kv_len=S_HEAD,
                                                                stream=st)), nbytes, "bytes"
    if name.startswith("prefill-"):
        # prefill-T4097, prefill-q512-kv4096 (Qwen2.5-0.5B heads, D=64) or
        # prefill-d128-T4097 (Qwen2.5-7B heads, D=128)
        parts = name.split("-")[1:]
        hq, hkv, hd = 14, 2, 64
        if parts[0] == "d128":
            hq, hkv, hd = 28, 4, 128
            parts = parts[1:]
        if len(parts) == 1:
            q_len = kv_len = int(parts[0][1:])
        else:
            q_len, kv_len = int(parts[0][1:]), int(parts[1][2:])
        q = inputs.randn((1, hq, q_len, hd), inputs.tensor_seed(0, 0), torch.bfloat16, device)
        k = inputs.randn((1, hkv, kv_len, hd), inputs.tensor_seed(0, 1), torch.bfloat16, device)
        v = inputs.randn((1, hkv, kv_len, hd), inputs.tensor_seed(0, 2), torch.bfloat16, device)
        o = torch.empty_like(q)
        flops = metrics.prefill_flops(hq, hd, q_len, kv_len, causal=True)
        return (lambda st: binding_mod().gqa_attn_prefill(q, k, v, o, kv_len, hd ** -0.5, True, st)), flops, "flop"
    raise SystemExit(f"unknown kernel case {name!r}")


KERNEL_CASES = ("decode-f32-S32768", "decode-bf16-S32768", "decode-bf16-ragged-B64", "decode-bf16-paged-B64",
                "q4-B4-S16384", "quantize-B4-S16384",
                "prefill-T4097", "prefill-T16384", "prefill-q512-kv4096", "varlen-prefill-B16",
                "prefill-d128-T4097", "prefill-d128-T16384",
                "decode-f32-layers8-S32768")


def binding_mod():
    from gqa_attention_kv_decode_gb300 import binding
    return binding


def run_kernel_case(args):
    """W + K launches of one configuration, each after an L2 flush, timed per
    launch with events; prints one JSON line.  Used as the command under ncu."""
    import __graft_entry__
    __graft_entry__.build()
    device = torch.device("cuda", 0)
    launch, units, unit_name = _case_inputs(args.kernel, device)
    flush = torch.empty(256 * 2**20 // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    evs = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush_l2(flush)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch(stream)
            e1.record(stream)
            if i >= args.warmup:
                evs.append((e0, e1))
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)
    rate = units / us / 1e3 if unit_name == "bytes" else units / us / 1e6
    print(json.dumps({"kernel_case": args.kernel, "us_per_launch": round(us, 3),
                      ("GB/s" if unit_name == "bytes" else "TFLOP/s"): round(rate, 1),
                      "algorithmic_" + unit_name: units}), flush=True)
    return 0


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gqa", choices=["gqa", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="headline only (for profiling)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--kernel", choices=KERNEL_CASES,
                    help="time one launch configuration only (the command profiled under ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel:
        return run_kernel_case(args)

    import __graft_entry__
    from gqa_attention_kv_decode_gb300 import binding

    world, rank, local = dist_env()
    dist = Dist(world)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        __graft_entry__.build()
    dist.barrier()
    binding.lib()
    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks()

    # CPU baseline first (spawned process, before any large device allocation)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline()

    stream = torch.cuda.Stream(device)
    S = S_HEAD
    layers = make_layers(S, torch.float32, device)
    outs = [torch.empty_like(q) for q, _, _ in layers]
    ws = binding.decode_workspace(1, HQ, HKV, D, S, binding.GQA_F32, device)
    step_bytes = LAYERS * metrics.decode_bytes(HQ, HKV, D, [S], 4)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            time_decode_step(binding, layers, outs, ws, S, stream)
    torch.cuda.synchronize()
    # The step as a decode step is run in production: its 28 calls (made
    # through the public API) captured once in a CUDA graph and replayed.
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=stream):
        time_decode_step(binding, layers, outs, ws, S, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step_graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            step_graph.replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    elapsed_ms = dist.max(t_start.elapsed_time(t_end))
    ms_per_step = elapsed_ms / args.steps

    # the same K steps as plain launches (the 28 calls issued one by one)
    l_start = torch.cuda.Event(enable_timing=True)
    l_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        l_start.record(stream)
        for _ in range(args.steps):
            time_decode_step(binding, layers, outs, ws, S, stream)
        l_end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    launch_ms_per_step = dist.max(l_start.elapsed_time(l_end)) / args.steps

    # the spread of the step times, from K more steps with an event at every
    # step boundary (outside the region above, which has none)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with torch.cuda.stream(stream):
        marks[0].record(stream)
        for i in range(args.steps):
            time_decode_step(binding, layers, outs, ws, S, stream)
            marks[i + 1].record(stream)
    torch.cuda.synchronize()
    step_ms = sorted(a.elapsed_time(b) for a, b in zip(marks[:-1], marks[1:]))
    step_spread = {"p10": round(step_ms[int(0.1 * (len(step_ms) - 1))], 4),
                   "p50": round(step_ms[int(0.5 * (len(step_ms) - 1))], 4),
                   "p90": round(step_ms[int(0.9 * (len(step_ms) - 1))], 4)}

    # the same K steps again with every layer call bracketed by events on the
    # launching stream (kept out of the region above: an event pair between
    # calls adds a few microseconds to each)
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            time_decode_step(binding, layers, outs, ws, S, stream, evs)
    torch.cuda.synchronize()
    clk = clocks.stop()
    launch_us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    isolated_call_us = sum(launch_us) / len(launch_us)
    # calls overlap (each split kernel is launched early and prefetches while
    # the previous merge runs), so the per-call duration is the timed region
    # divided by its calls; an event pair around a call serialises it
    avg_launch_us = elapsed_ms * 1e3 / (args.steps * LAYERS)
    per_launch_bytes = metrics.decode_bytes(HQ, HKV, D, [S], 4)
    n_split = binding.gqa_attn_decode_num_splits(1, HQ, HKV, D, S, binding.GQA_F32)
    launches_per_call = 2 if n_split > 1 else 1  # split kernel (+ merge kernel)
    achieved = per_launch_bytes / avg_launch_us / 1e3
    value = replica_value(world, step_bytes, ms_per_step)

    # end to end through the public API with host buffers
    e2e_steps = 3
    host = [(q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()) for q, k, v in layers]
    host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    h2d = sum(q.numel() * q.element_size() + k.numel() * k.element_size() + v.numel() * v.element_size()
              for q, k, v in host)
    d2h = sum(o.numel() * o.element_size() for o in host_out)

    # Each layer's inputs are copied on a stream of their own and its call
    # waits for them, so layer l attends while layer l + 1 is still copying;
    # a step's copies wait for the previous step to be done with the buffers.
    copy_stream = torch.cuda.Stream(device)

    def e2e_step():
        copy_stream.wait_stream(stream)
        landed = []
        with torch.cuda.stream(copy_stream):
            for (hq, hk, hv), (q, k, v) in zip(host, layers):
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                landed.append(ev)
        for ev, (q, k, v), o in zip(landed, layers, outs):
            stream.wait_event(ev)
            binding.gqa_attn_decode(q, k, v, o, None, D ** -0.5, ws, max_kv_len=S, stream=stream)
        for o, ho in zip(outs, host_out):
            ho.copy_(o, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
    torch.cuda.synchronize()
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = dist.max(e0.elapsed_time(e1)) / e2e_steps
    e2e_value = replica_value(world, step_bytes, e2e_ms)
    # the same step's host-to-device copies alone: the rate of the host link,
    # which bounds the end-to-end number (the attention calls hide under it).
    # The faster of two timings: a bound wants the best rate the link gave
    # (single timings have come out up to 3x slow on a shared host).
    copy_ms = None
    for _ in range(2):
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(copy_stream)
        with torch.cuda.stream(copy_stream):
            for _ in range(e2e_steps):
                for (hq, hk, hv), (q, k, v) in zip(host, layers):
                    q.copy_(hq, non_blocking=True)
                    k.copy_(hk, non_blocking=True)
                    v.copy_(hv, non_blocking=True)
        c1.record(copy_stream)
        torch.cuda.synchronize()
        t = dist.max(c0.elapsed_time(c1)) / e2e_steps
        copy_ms = t if copy_ms is None else min(copy_ms, t)
    del host, host_out

    traffic = recorded_traffic("decode.cu", "decode_f32_d128_nrep7_S32768")
    # the split kernel alone, as ncu timed it (cold, serialised, no overlap)
    rec = recorded_ncu("decode.cu", "decode_f32_d128_nrep7_S32768")
    isolated_kernel_frac = None
    if rec and rec.get("ncu_duration_ns"):
        isolated_kernel_frac = {"value": round(per_launch_bytes / (rec["ncu_duration_ns"] * 1e-9) / 1e9 / hbm_peak, 4),
                                "kernel_us": rec["ncu_duration_ns"] / 1e3,
                                "source": "profiles/traffic.json (ncu gpu__time_duration.sum of the split kernel)"}
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": S,
                   "layers_per_step": LAYERS, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (3.76 GB per step on distinct buffers); no flush needed",
                   "launch": "the step's 28 public-API calls captured once in a CUDA graph, replayed K times"},
        "plain_launches": {"value": round(replica_value(world, step_bytes, launch_ms_per_step), 1), "unit": "GB/s",
                           "ms_per_step": round(launch_ms_per_step, 4),
                           "note": "the same K steps with the 28 calls issued one by one"},
        "hbm_fraction": round(value / world / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                     "kernel": "decode_split_kernel<float,128,7,2,3> + decode_merge_kernel",
                     "peak_source": peak_src, "avg_launch_us": round(avg_launch_us, 3),
                     "timing": "events on the launching stream around the K timed graph replays / (K x 28 calls)",
                     "isolated_call_us": round(isolated_call_us, 3),
                     "basis": "per-call stream average: consecutive calls overlap (each split kernel "
                              "is launched early and prefetches into L2 while the previous merge runs)",
                     "isolated_kernel_frac": isolated_kernel_frac,
                     "n_split": n_split},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "h2d_copies_alone": {"ms_per_step": round(copy_ms, 3), "timings": "faster of 2",
                                     "h2d_gbs": round(h2d / copy_ms / 1e6, 1),
                                     "e2e_frac": round(copy_ms / e2e_ms, 4),
                                     "note": "the step's host-to-device copies with no attention call: "
                                             "the host link bounds e2e"}},
        "gpu_launches": LAYERS * args.steps * launches_per_call,
        "step_ms_spread": step_spread,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    del layers, outs, ws
    torch.cuda.empty_cache()

    if rank == 0 and world == 1 and not args.no_extras:
        flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=device)
        sweep = {}
        for dtype, name in ((torch.float32, "f32"), (torch.bfloat16, "bf16")):
            for s in (128, 256, 512, 1024, 2048, 4096, 32768):
                sweep[f"{name}_S{s}"] = sweep_point(binding, s, dtype, device, stream, flush)
        line["decode_sweep_qwen7b_28_layers"] = sweep
        line["ragged_decode_qwen3_4b_36_layers"] = [ragged_point(binding, B, device, stream, flush)
                                                   for B in (1, 2, 4, 8, 16, 64)]
        line["capacity_planned_decode_qwen7b_f32_28_layers"] = capacity_points(binding, (512, 2048, 8192), device,
                                                                               stream, flush)
        line["q4_decode_qwen3_4b_B4_36_layers"] = [q4_point(binding, S, device, stream, flush)
                                                  for S in (64, 2048, 16384)]
        if cpu is not None:  # the oracle beside the GPU figure, same metric
            line["q4_decode_qwen3_4b_B4_36_layers"][-1]["cpu_oracle"] = cpu["q4_decode_S16384"]
        line["paged_decode_qwen3_4b_36_layers"] = [paged_point(binding, B, device, stream, flush)
                                                   for B in (16, 64)]
        line["quantize_q4_qwen3_4b"] = quantize_point(binding, device, stream, flush)
        line["q4_residual_decode_qwen3_4b_B4_36_layers"] = [q4_residual_point(binding, S, device, stream, flush)
                                                            for S in (2048, 16384)]
        line["cross_layer_decode_qwen7b_f32_28_layers"] = [layers_point(binding, S, device, stream, flush)
                                                           for S in (128, 2048, 32768)]
        line["varlen_prefill_qwen05b_chunks_512"] = [varlen_prefill_point(binding, B, device, stream, flush, bf16_peak)
                                                     for B in (4, 16)]
        pf = [prefill_point(binding, T, T, device, stream, flush, bf16_peak) for T in (513, 2049, 4097, 16384)]
        pf.append(prefill_point(binding, 512, 4096, device, stream, flush, bf16_peak))
        if cpu is not None:
            pf[3]["cpu_oracle"] = cpu["prefill_T16384"]
        line["prefill_causal_qwen05b_bf16"] = pf
        # head dimension 128 at the Qwen2.5-7B head geometry (28 layers per step)
        pf128 = [prefill_point(binding, T, T, device, stream, flush, bf16_peak, NL=28, Hq=28, Hkv=4, D=128)
                 for T in (4097, 16384)]
        pf128.append(prefill_point(binding, 512, 4096, device, stream, flush, bf16_peak, NL=28, Hq=28, Hkv=4,
                                   D=128))
        line["prefill_causal_qwen7b_d128_bf16"] = pf128
        line["roofline_prefill_d128"] = {"bound": "tensor", "achieved": pf128[1]["TFLOPs"], "peak": bf16_peak,
                                         "unit": "TFLOP/s", "frac": pf128[1]["frac_of_bf16_peak"],
                                         "traffic": recorded_traffic("prefill.cu", "prefill_causal_d128_T16384"),
                                         "kernel": "prefill_kernel<128> (T=16384 causal, 28 layer launches per step)",
                                         "peak_source": peak_src + " bf16 burst"}
        big = pf[3]
        line["roofline_prefill"] = {"bound": "tensor", "achieved": big["TFLOPs"], "peak": bf16_peak,
                                    "unit": "TFLOP/s", "frac": big["frac_of_bf16_peak"],
                                    "traffic": recorded_traffic("prefill.cu", "prefill_causal_T16384"),
                                    "kernel": "prefill_kernel (T=16384 causal, 24 layer launches per step)",
                                    "peak_source": peak_src + " bf16 burst"}
        del flush
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
