#!/usr/bin/env python3
"""Benchmark of the GB300 gated-delta-rule library on synthetic inputs.

Headline workload: one decode step of a 24-layer stack of gated delta rule
layers, 32 value heads x head_dim 128, one sequence, one token, bf16 q/k/v,
fp32 state per layer (the geometry the "marcsun13/ggml-gated-delta-net"
model card measures in section "Measured", where it quotes 0.40 ms per token
over 24 layers on an Apple M2 Max: context, not a target).  The 24 calls are
captured once in a CUDA graph and replayed; L2 is flushed before every step
(the 24 states would otherwise stay in the 129 MB L2).

The same JSON line carries, under "workloads", batched decode (64 sequences)
and long prefill (4096 tokens x 1 sequence; 16384 tokens x 8 sequences at
head_dim 128, 64 and 256), each with its own roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun) every rank runs an independent replica on its own GPU:
the op has no exchange step, so no collective is used on the data path; the
barrier and the max over ranks are for timing only.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s and decode µs/step at 32h×128; % HBM / tensor roofline"
# 0.40 ms per token over 24 layers, 32 value heads x 128 (Apple M2 Max,
# model card section "Measured"): the same workload on other hardware.
PUBLISHED_US_PER_24L_STEP = 400.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
N_SMS = 152
L2_FLUSH_BYTES = 512 << 20
# DRAM bytes per launch measured with ncu, keyed by workload; an entry only
# counts while the kernel sources it was measured on are unchanged.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


# ----------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    p = dict(FALLBACK_PEAKS)
    p["source"] = "fallback"
    return p


def sources_sha(rel_paths):
    import hashlib
    h = hashlib.sha256()
    for rel in rel_paths.split("+"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def load_traffic():
    """{workload: dram bytes per launch} for entries whose sources still match."""
    out = {}
    if not os.path.exists(TRAFFIC_FILE):
        return out
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#") or len(parts) < 4:
                continue
            workload, srcs, sha, nbytes = parts[:4]
            try:
                if sources_sha(srcs) == sha:
                    out[workload] = float(nbytes)
            except OSError:
                continue
    return out


def alu_fp32_tflops(peaks):
    # 152 SMs x 128 fp32 lanes x 2 flops (FMA) x max SM clock
    return N_SMS * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12


def decode_bytes_per_head(d, in_bytes):
    # state read + write (fp32) + q, k, v + out (fp32) + g, beta
    return 8 * d * d + 3 * d * in_bytes + 4 * d + 8


def run_bytes(B, T, H, Hk, d, in_bytes):
    """Algorithmic bytes of one call on the recurrent path: the state read and
    written once (fp32), q and k once per key head, v, out (fp32), g and beta
    once per value head and token."""
    return B * H * 8 * d * d + B * T * (2 * Hk * d * in_bytes + H * (d * in_bytes + 4 * d + 8))


def prefill_bytes_per_token_head(d, in_bytes):
    return 3 * d * in_bytes + 4 * d + 8


def chunked_flops_per_token_head(d, C=64):
    # issued MMA tiles: K K^T, Q K^T, T (beta K), T (beta V), P U at 2Cd each;
    # W S^T, Q S^T, U^T K at 2d^2 each
    return 10 * C * d + 6 * d * d


def recurrent_flops_per_token_head(d):
    # per row: S.k and S.q (2d each), decay + rank-1 update (2d)
    return 6 * d * d


class ClockSampler:
    """nvidia-smi samples during the timed region (read-only queries)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------ distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x):
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([float(x)], device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------- our implementation

class Timer:
    """CUDA-event timing of K steps on one stream, L2 flushed before each."""

    def __init__(self, torch, stream, flush):
        self.torch, self.stream, self.flush = torch, stream, flush

    def run(self, fn, steps, warmup, dist):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                self.flush.zero_()
                fn()
            torch.cuda.synchronize()
            dist.barrier()
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]
            for a, b in evs:
                self.flush.zero_()
                a.record(self.stream)
                fn()
                b.record(self.stream)
            torch.cuda.synchronize()
            dist.barrier()
            torch.cuda.synchronize()
        times = [a.elapsed_time(b) for a, b in evs]  # ms
        return times


def run_decode24(torch, gdn, W, dev, timer, args, dist, peaks):
    """Headline: 24 layers x (1 seq, 1 token, 32 heads, d 128), graph-replayed."""
    w = W.DECODE_24L
    L = w.layers
    B, H, d = w.B, w.H, w.d
    layers = [W.make_inputs(w, dev, layer=l) for l in range(L)]
    # one packed device buffer for every layer's per-step inputs so that the
    # end-to-end leg moves them with one host->device copy
    n_in = B * H * d
    in_elems_bf16 = 3 * n_in
    per_layer_bytes = in_elems_bf16 * 2 + 2 * B * H * 4
    per_layer_bytes = (per_layer_bytes + 255) // 256 * 256
    dev_in = torch.empty(L * per_layer_bytes, dtype=torch.uint8, device=dev)
    views = []
    for l, x in enumerate(layers):
        base = l * per_layer_bytes
        qkv = dev_in[base:base + in_elems_bf16 * 2].view(torch.bfloat16).view(3, B, 1, H, d)
        gb = dev_in[base + in_elems_bf16 * 2: base + in_elems_bf16 * 2 + 2 * B * H * 4] \
            .view(torch.float32).view(2, B, 1, H)
        qkv[0].copy_(x["q"]); qkv[1].copy_(x["k"]); qkv[2].copy_(x["v"])
        gb[0].copy_(x["g"]); gb[1].copy_(x["beta"])
        views.append((qkv[0], qkv[1], qkv[2], gb[0], gb[1], x["state"]))
    dev_out = torch.empty((L, B, 1, H, d), dtype=torch.float32, device=dev)

    stream = timer.stream

    def step():
        for l in range(L):
            q, k, v, g, beta, st = views[l]
            gdn.forward(q, k, v, g, beta, st, out=dev_out[l], state_out=st)

    with torch.cuda.stream(stream):
        step()                                   # lazy set-up outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    if gdn.device_status() != gdn.OK:
        raise RuntimeError("device status after capture")

    times = timer.run(graph.replay, args.steps, args.warmup, dist)
    if gdn.device_status() != gdn.OK:
        raise RuntimeError("device status after timing")
    ms = sum(times) / len(times)
    ms = dist.max(ms)
    us_step = ms * 1e3
    bytes_launch = H * B * decode_bytes_per_head(d, 2)
    launch_s = ms / 1e3 / L
    achieved = bytes_launch / launch_s / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": load_traffic().get(w.name),
            "kernel": "recurrent_kernel<128,8,1,bf16>",
            "bytes_per_launch": bytes_launch,
            "note": "per-launch time = graph step time / 24 (includes inter-kernel gaps); "
                    f"peak {peaks['source']}"}

    # end to end: pinned host inputs -> device, 24 layers, outputs -> pinned host
    host_in = torch.empty_like(dev_in, device="cpu").pin_memory()
    host_in.copy_(dev_in)
    host_out = torch.empty_like(dev_out, device="cpu").pin_memory()
    e2e_times = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            timer.flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            dev_in.copy_(host_in, non_blocking=True)
            graph.replay()
            host_out.copy_(dev_out, non_blocking=True)
            stream.synchronize()
            t1 = time.perf_counter()
            if i >= args.warmup:
                e2e_times.append((t1 - t0) * 1e6)
    e2e_us = dist.max(sum(e2e_times) / len(e2e_times))
    e2e = {"value": e2e_us, "unit": "us/step", "h2d_bytes_per_step": int(dev_in.numel()),
           "d2h_bytes_per_step": int(dev_out.numel() * 4),
           "how": "pinned host inputs copied in, 24-layer graph of C-ABI calls, outputs copied "
                  "out, host wall clock around each step (synchronised)"}
    launches = L * args.steps
    cfg = {"workload": w.name, "n_seqs": B, "n_tokens": 1, "n_heads": H, "head_dim": d,
           "layers": L, "io_dtype": "bf16", "state_dtype": "f32",
           "l2": "flushed (512 MB write) before every timed step", "graph": True}
    return {"value": us_step, "ms": ms, "roofline": roof, "e2e": e2e, "launches": launches,
            "config": cfg, "times_ms": times, "spread": spread(times)}


def spread(times_ms, scale=1e3, unit="us"):
    """Median, minimum and maximum of the timed repetitions (in `unit`)."""
    xs = sorted(times_ms)
    n = len(xs)
    med = xs[n // 2] if n % 2 else 0.5 * (xs[n // 2 - 1] + xs[n // 2])
    return {"median": med * scale, "min": xs[0] * scale, "max": xs[-1] * scale, "unit": unit,
            "n": n}


def attn_bytes(w, elt):
    """Algorithmic bytes of one decode-attention call: the cache (k, v) and q
    read once, the mask read once, the fp32 output written once."""
    kv = 2 * w.B * w.Hkv * w.n_kv * w.d * elt
    qb = w.B * w.H * w.n_q * w.d * elt
    mb = w.B * w.n_q * w.n_kv * elt if w.mask else 0
    return kv + qb + mb + w.B * w.n_q * w.H * w.d * 4


def run_attn(torch, gdn, W, w, dev, timer, args, dist, peaks):
    """One decode-attention call per step (L2 flushed before each)."""
    inp = W.make_attn_inputs(w, dev)
    out = torch.empty((w.B, w.n_q, w.H, w.d), dtype=torch.float32, device=dev)

    def fn():
        gdn.flash_attn(inp["q"], inp["k"], inp["v"], inp["mask"], out=out)

    times = timer.run(fn, args.steps, args.warmup, dist)
    ms = dist.max(sum(times) / len(times))
    elt = 4 if w.dtype == "f32" else 2
    by = attn_bytes(w, elt)
    ach = by / (ms / 1e3) / 1e9
    del inp, out
    return {"workload": w.name, "path": "flash_attn", "metric": "attention us/call",
            "value": ms * 1e3, "unit": "us/call", "ms_per_step": ms, "launches_per_step": 1,
            "spread": spread(times),
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "traffic": load_traffic().get(w.name),
                         "bytes_per_launch": by}}


def run_single_call(torch, gdn, W, w, dev, timer, args, dist, peaks, kind, in_place=True):
    inp = W.make_inputs(w, dev)
    B, T, H, d = w.B, w.T, w.H, w.d
    out = torch.empty((B, T, H, d), dtype=torch.float32, device=dev)
    st = inp["state"] if inp["state"] is not None else None
    st_out = st if (in_place and st is not None) else torch.empty((B, H, d, d), device=dev)
    path = gdn.select_path(B, T, H, d, w.dtype)
    ws = None
    nws = gdn.workspace_bytes(B, T, H, d, w.dtype, path)
    if nws:
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)

    def fn():
        gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], st, out=out,
                    state_out=st_out, path=path, workspace=ws)

    times = timer.run(fn, args.steps, args.warmup, dist)
    if gdn.device_status() != gdn.OK:
        raise RuntimeError(f"device status after {w.name}")
    ms = dist.max(sum(times) / len(times))
    in_b = 2 if w.dtype == "bf16" else 4
    res = {"workload": w.name, "path": path, "ms_per_step": ms, "spread": spread(times),
           "launches_per_step": launches_per_call(
               path, nws, B * H, d, torch.cuda.get_device_properties(dev).multi_processor_count)}
    if kind == "decode":
        bytes_launch = run_bytes(B, T, H, w.n_k, d, in_b)
        achieved = bytes_launch / (ms / 1e3) / 1e9
        res.update({"metric": "decode us/step", "value": ms * 1e3, "unit": "us/step",
                    "roofline": {"bound": "hbm", "achieved": achieved,
                                 "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": achieved / peaks["hbm_gbs"],
                                 "traffic": load_traffic().get(w.name),
                                 "bytes_per_launch": bytes_launch}})
    else:
        toks = B * T
        res.update({"metric": "prefill tokens/s", "value": toks / (ms / 1e3), "unit": "tokens/s"})
        io = B * T * H * prefill_bytes_per_token_head(d, in_b) + 8 * B * H * d * d
        hbm_ach = io / (ms / 1e3) / 1e9
        if path == "chunked":
            fl = B * T * H * chunked_flops_per_token_head(d)
            ach = fl / (ms / 1e3) / 1e12
            peak = peaks["bf16_tflops"]
            res["roofline"] = {"bound": "tensor", "achieved": ach, "peak": peak,
                               "unit": "TFLOP/s", "frac": ach / peak,
                               "traffic": load_traffic().get(w.name),
                               "flops_per_launch": fl,
                               "hbm_achieved_gbs": hbm_ach,
                               "hbm_frac": hbm_ach / peaks["hbm_gbs"]}
        else:
            fl = B * T * H * recurrent_flops_per_token_head(d)
            ach = fl / (ms / 1e3) / 1e12
            peak = alu_fp32_tflops(peaks)
            res["roofline"] = {"bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                               "frac": ach / peak, "traffic": None, "flops_per_launch": fl,
                               "peak_how": "152 SMs x 128 fp32 lanes x 2 x max SM clock",
                               "hbm_achieved_gbs": hbm_ach,
                               "hbm_frac": hbm_ach / peaks["hbm_gbs"]}
    del inp, out
    return res


def run_decode_steady(torch, gdn, W, w, dev, args, dist, peaks, n_bufs=4):
    """Batched decode in steady state: K back-to-back calls between one pair
    of events, each updating in place one of `n_bufs` state buffers in turn
    (each larger than L2), with no flush in between.  Every call's state
    write-back then lands inside the timed window, as it does in a decode
    loop where step n + 1 pays for step n's writes."""
    B, T, H, d = w.B, w.T, w.H, w.d
    inp = W.make_inputs(w, dev)
    states = [inp["state"].clone() for _ in range(n_bufs)]
    out = torch.empty((B, T, H, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    calls = max(args.steps, 4 * n_bufs)

    def call(i):
        st = states[i % n_bufs]
        gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], st, out=out,
                    state_out=st, path="recurrent")

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, n_bufs)):
            call(i)
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(calls):
            call(i)
        b.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
    if gdn.device_status() != gdn.OK:
        raise RuntimeError(f"device status after {w.name} (steady state)")
    ms = dist.max(a.elapsed_time(b) / calls)
    by = run_bytes(B, T, H, w.n_k, d, 2 if w.dtype == "bf16" else 4)
    ach = by / (ms / 1e3) / 1e9
    del inp, states, out
    return {"workload": w.name + "_steady", "path": "recurrent", "metric": "decode us/step",
            "value": ms * 1e3, "unit": "us/step", "ms_per_step": ms, "launches_per_step": 1,
            "launches_timed": calls,
            "how": f"{calls} back-to-back in-place calls over {n_bufs} rotating state buffers "
                   "(128 MiB each), one pair of CUDA events, no L2 flush: each call's state "
                   "write-back lands inside the window",
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": ach / peaks["hbm_gbs"], "traffic": None,
                         "bytes_per_launch": by,
                         "note": "algorithmic bytes; in steady state the DRAM bytes per call "
                                 "equal them (state read + written back once)"}}


def walk_launches(pairs, d, sms):
    """State-walk launches of a two-kernel chunked call: the library's value
    block split (64-row blocks for the full waves, the rest at 32 rows after
    them when 64-row blocks leave a partial last wave that fits one wave at
    32 rows), restated here to count kernels."""
    if pairs * (d // 32) <= sms:
        return 1
    ctas64 = pairs * (d // 64)
    full = ctas64 // sms
    if full >= 1 and ctas64 % sms and (full * sms) % (d // 64) == 0:
        p64 = full * sms // (d // 64)
        if (pairs - p64) * (d // 32) <= sms:
            return 2
    return 1


def launches_per_call(path, workspace_bytes, pairs=0, d=0, sms=0):
    """Kernels one call launches.  A chunked call that needs a workspace
    (head_dim 256, and head_dim 128 with few (sequence, head) pairs) runs the
    chunk-transform kernel and then the state walk (one or two launches);
    every other call one."""
    if path == "chunked" and workspace_bytes > 0:
        return 1 + walk_launches(pairs, d, sms)
    return 1


# ------------------------------------------------------------ CPU oracle

def oracle_decode24_us(W, min_seconds, n_threads=0):
    """The float64 C oracle, as it stands, on the 24-layer decode step
    (n_threads 0: every OpenMP thread)."""
    import numpy as np
    import oracle
    oracle.build()
    w = W.DECODE_24L
    layers = [W.to_numpy_f32(W.make_inputs(w, "cpu", layer=l)) for l in range(w.layers)]
    steps = 0
    t0 = time.perf_counter()
    while True:
        for x in layers:
            oracle.recurrent_c(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"],
                               n_threads=n_threads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    _ = np
    return el / steps * 1e6, steps, (n_threads or oracle.max_threads())


def oracle_prefill_tokens_per_s(W, w, seconds_hint=3.0):
    """Oracle throughput on a bounded sample of a prefill workload: as many
    (sequence, head) pairs as there are OpenMP threads, over a prefix of the
    tokens, scaled to tokens/s of the full head count."""
    import oracle
    oracle.build()
    nthr = oracle.max_threads()
    pairs = min(nthr, w.B * w.H)
    T = min(w.T, 256)
    x = W.to_numpy_f32(W.make_inputs(w.replace(B=1, H=pairs), "cpu", T=T))
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.recurrent_c(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"])
        reps += 1
        if time.perf_counter() - t0 >= seconds_hint:
            break
    el = time.perf_counter() - t0
    token_heads_per_s = reps * pairs * T / el
    return {"value": token_heads_per_s / w.H, "unit": "tokens/s", "cores": nthr, "kind": "oracle",
            "sample": f"{pairs} (seq, head) pairs x {T} tokens, {reps} repeats, scaled to "
                      f"{w.H} heads"}


def oracle_decode_us(W, w, seconds_hint=2.0):
    """The float64 C oracle on a whole decode / short-run workload (every
    (sequence, head) pair), repeated for about `seconds_hint` seconds."""
    import oracle
    oracle.build()
    x = W.to_numpy_f32(W.make_inputs(w, "cpu"))
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.recurrent_c(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"])
        reps += 1
        if time.perf_counter() - t0 >= seconds_hint:
            break
    el = time.perf_counter() - t0
    return {"value": el / reps * 1e6, "unit": "us/step", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"the whole workload ({w.B * w.H} (seq, head) pairs x {w.T} token(s)), "
                      f"{reps} repeats"}


def oracle_attn_us(W, w, seconds_hint=2.0):
    """The float64 numpy attention oracle on a bounded sample of a decode
    attention workload (whole sequences), scaled to one call."""
    from oracle.attn import attention
    nb = 1 if w.B > 1 else w.B
    x = W.make_attn_inputs(w.replace(B=nb), "cpu")
    f64 = lambda t: None if t is None else t.double().numpy()
    q, k, v, m = f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["mask"])
    t0 = time.perf_counter()
    reps = 0
    while True:
        attention(q, k, v, m)
        reps += 1
        if time.perf_counter() - t0 >= seconds_hint:
            break
    el = time.perf_counter() - t0
    return {"value": el / reps * 1e6 * (w.B / nb), "unit": "us/call", "cores": 1,
            "kind": "oracle",
            "sample": f"{nb} of {w.B} sequence(s), {reps} repeats, scaled to the whole call "
                      "(numpy float64, one Python thread)"}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--oracle-seconds", type=float, default=10.0)
    ap.add_argument("--only", default=None,
                    help="time only this named extra workload (for profiling); prints its "
                         "entry as the JSON line")
    ap.add_argument("--only-seqs", type=int, default=None,
                    help="with --only: override n_seqs (smaller profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    dist = Dist()
    from linear_attention_sequence_gated_gb300 import workloads as W

    if args.impl == "reference":
        # The reference arm is the float64 oracle on the host cores, rank 0 only.
        if dist.rank != 0:
            return
        us, steps, cores = oracle_decode24_us(W, max(1.0, args.oracle_seconds / 2))
        w = W.DECODE_24L
        cfg = {"workload": w.name, "n_seqs": w.B, "n_tokens": 1, "n_heads": w.H,
               "head_dim": w.d, "layers": w.layers, "io_dtype": "bf16", "state_dtype": "f32"}
        times = []
        import oracle
        layers = [W.to_numpy_f32(W.make_inputs(w, "cpu", layer=l)) for l in range(w.layers)]
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            for x in layers:
                oracle.recurrent_c(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"])
            if i >= args.warmup:
                times.append((time.perf_counter() - t0) * 1e6)
        v = sum(times) / len(times)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/step",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
                "vs_baseline": v / PUBLISHED_US_PER_24L_STEP, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": v, "unit": "us/step", "cores": cores, "kind": "oracle",
                                 "sample": f"{args.steps} timed 24-layer decode steps"},
                "e2e": {"value": v, "unit": "us/step", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import linear_attention_sequence_gated_gb300 as gdn
    from linear_attention_sequence_gated_gb300 import _build
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    _build.build()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    timer = Timer(torch, stream, flush)

    # the entries with a stated target (batched decode, the 4k and 8 x 16k
    # head_dim-128 prefills) come last in "workloads"
    specs = [(W.MULTITOKEN_B64_T4, "decode"), (W.DECODE_B64_HK16, "decode"),
             (W.PREFILL_16K_D64, "prefill"), (W.PREFILL_16K_D256, "prefill"),
             (W.DECODE_B64, "decode"), (W.PREFILL_4K, "prefill"), (W.PREFILL_16K, "prefill")]
    if args.only and args.only in W.ATTN_BY_NAME:
        r = run_attn(torch, gdn, W, W.ATTN_BY_NAME[args.only], dev, timer, args, dist, peaks)
        if dist.rank == 0:
            print(json.dumps(r))
        dist.close()
        return
    if args.only and args.only == W.DECODE_B64.name + "_steady":
        r = run_decode_steady(torch, gdn, W, W.DECODE_B64, dev, args, dist, peaks)
        if dist.rank == 0:
            print(json.dumps(r))
        dist.close()
        return
    if args.only:
        w, kind = next((w, k) for w, k in specs if w.name == args.only)
        if args.only_seqs:
            w = w.replace(name=f"{w.name}_seqs{args.only_seqs}", B=args.only_seqs)
        r = run_single_call(torch, gdn, W, w, dev, timer, args, dist, peaks, kind)
        if dist.rank == 0:
            print(json.dumps(r))
        dist.close()
        return

    clocks = ClockSampler(dist.local)
    clocks.start()
    head = run_decode24(torch, gdn, W, dev, timer, args, dist, peaks)
    extra = []
    launches = head["launches"]
    if not args.no_extra:
        for w in W.ATTN_ALL:
            r = run_attn(torch, gdn, W, w, dev, timer, args, dist, peaks)
            launches += r["launches_per_step"] * args.steps
            extra.append(r)
            torch.cuda.empty_cache()
        for w, kind in specs:
            r = run_single_call(torch, gdn, W, w, dev, timer, args, dist, peaks, kind)
            launches += r["launches_per_step"] * args.steps
            extra.append(r)
            torch.cuda.empty_cache()
            if w is W.DECODE_B64:
                r = run_decode_steady(torch, gdn, W, w, dev, args, dist, peaks)
                launches += r["launches_timed"]
                extra.append(r)
                torch.cuda.empty_cache()
    clocks.stop()

    cpu = None
    if dist.rank == 0:
        us, n, cores = oracle_decode24_us(W, args.oracle_seconds)
        us1, n1, _ = oracle_decode24_us(W, max(1.0, args.oracle_seconds / 4), n_threads=1)
        cpu = {"value": us, "unit": "us/step", "cores": cores, "kind": "oracle",
               "sample": f"{n} repeats of the full 24-layer decode step (float64 C, OpenMP over "
                         f"(seq, head) pairs)",
               "one_core": {"value": us1, "unit": "us/step", "cores": 1,
                            "sample": f"{n1} repeats of the same step on one thread"}}
        cpu_decode = {}
        for r in extra:
            name = r["workload"]
            if r["metric"] == "prefill tokens/s":
                r["cpu_baseline"] = oracle_prefill_tokens_per_s(W, W.BY_NAME[name])
            elif r["metric"] == "decode us/step":
                base = name[:-len("_steady")] if name.endswith("_steady") else name
                if base not in cpu_decode:
                    cpu_decode[base] = oracle_decode_us(W, W.BY_NAME[base])
                r["cpu_baseline"] = cpu_decode[base]
            elif r["path"] == "flash_attn":
                r["cpu_baseline"] = oracle_attn_us(W, W.ATTN_BY_NAME[name])

    if dist.rank == 0:
        us = head["value"]
        line = {"metric": METRIC, "value": us, "unit": "us/step", "n_gpus": dist.world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms"],
                "higher_is_better": False, "scaling": "weak",
                "vs_baseline": us / PUBLISHED_US_PER_24L_STEP, "dtype": "f32",
                "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), "
                        "beta sigmoid(N(0,1)), g -softplus(N(0,1)), state N(0,0.02))",
                "config": head["config"], "roofline": head["roofline"], "cpu_baseline": cpu,
                "e2e": head["e2e"], "gpu_launches": launches, "clocks": clocks.summary(),
                "spread": head["spread"], "peaks_source": peaks["source"], "workloads": extra}
        print(json.dumps(line))
    dist.close()


if __name__ == "__main__":
    main()
