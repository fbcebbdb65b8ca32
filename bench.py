"""Benchmark of the Markov draft walk on one GB300 (or N independent replicas).

A step is one full K-position walk over one batch: the timed region holds exactly the
walk kernel(s) of each step, with an L2 flush (a write of a buffer larger than L2)
between steps outside the per-step CUDA events, so every walk starts with a cold L2 as
in the pages' own kernel benchmark. Inputs are seeded synthetic tensors of the
workload's shapes and distributions, resident in HBM before timing starts.

Default workload: V=151936, rank 256, K=7, bs=64, int8 W2 (per-row fp32 scales),
greedy, base logits N(0, 3^2) with one +8 peak per row and position. Every other
configuration of the workload family is timed too and reported under "variants".

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs an independent replica on its own GPU (the walk does
not shard: every rank walks its own batch); rank 0 prints one JSON line.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft tokens/s of a K-step Markov draft walk (µs per walk alongside)"
UNIT = "draft tokens/s"
R = 256

MAIN = dict(name="v151936_k7_bs64_int8_greedy", V=151936, K=7, bs=64, int8=True, mode=0, T=1.0,
            top_k=0, peak=8.0, logits=False)


def _cfg(name, V, K, bs, int8, mode, T, top_k=0, peak=None, logits=False):
    return dict(name=name, V=V, K=K, bs=bs, int8=int8, mode=mode, T=T, top_k=top_k, peak=peak, logits=logits)


# Every configuration of the workload family, timed as "variants" beside the main line:
# V=129280 K=5 bs=1 bf16 greedy; V=151936 K=7 int8 at bs 1/16/64, greedy and sampled at
# T=1 with a +8 peak; V=151936 K=16 bf16 sampled at T=0.7 writing draft_logits, bs 1/64;
# V=248320 K=16 int8 greedy at bs 1/16/64; the top-k walk at V=151936 K=7 bs=64, k 512 and
# 4096, sampled at T=1.
VARIANTS = [
    _cfg("v129280_k5_bs1_bf16_greedy", 129280, 5, 1, False, 0, 1.0),
    _cfg("v151936_k7_bs1_int8_greedy", 151936, 7, 1, True, 0, 1.0, peak=8.0),
    _cfg("v151936_k7_bs1_int8_prob", 151936, 7, 1, True, 1, 1.0, peak=8.0),
    _cfg("v151936_k7_bs16_int8_greedy", 151936, 7, 16, True, 0, 1.0, peak=8.0),
    _cfg("v151936_k7_bs16_int8_prob", 151936, 7, 16, True, 1, 1.0, peak=8.0),
    _cfg("v151936_k7_bs64_int8_prob", 151936, 7, 64, True, 1, 1.0, peak=8.0),
    _cfg("v151936_k16_bs1_bf16_prob_logits", 151936, 16, 1, False, 1, 0.7, peak=8.0, logits=True),
    _cfg("v151936_k16_bs64_bf16_prob_logits", 151936, 16, 64, False, 1, 0.7, peak=8.0, logits=True),
    _cfg("v248320_k16_bs1_int8_greedy", 248320, 16, 1, True, 0, 1.0),
    _cfg("v248320_k16_bs16_int8_greedy", 248320, 16, 16, True, 0, 1.0),
    _cfg("v248320_k16_bs64_int8_greedy", 248320, 16, 64, True, 0, 1.0),
    _cfg("v151936_k7_bs64_topk512_prob", 151936, 7, 64, False, 1, 1.0, top_k=512),
    _cfg("v151936_k7_bs64_topk4096_prob", 151936, 7, 64, False, 1, 1.0, top_k=4096),
]
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    sm_mhz=float(d.get("sm_max_mhz", 2070.0)), src="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, sm_mhz=2070.0, src="fallback")


# Per-SM rates used for the on-chip floors: shared memory 512 bytes per clock (16-byte
# loads without bank conflicts, measured on this GPU with a single-SM probe), 128 fp32
# FMA lanes per clock, 16 multi-function-unit lanes per clock (logarithms).
SMEM_B_PER_CLK = 512
FFMA_PER_CLK = 128
MUFU_PER_CLK = 16
# Instructions per Gumbel draw on the integer/fp32 pipes besides the two logarithms:
# a quarter of a Philox4x32-10 block (10 rounds of two 32x32 multiplies with high halves
# and four xors, ~8 instructions per round) plus the uniform and the series.
GUMBEL_ALU_PER_DRAW = 30


def row_bytes(cfg) -> int:
    return R * (1 if cfg["int8"] else 2)


def hbm_bytes(cfg) -> float:
    """Algorithmic HBM bytes of one walk: W2 (+ scales) once, every base logit once, the
    K embedding rows per request, the tokens, and draft_logits when written. The top-k
    walk reads each gathered bf16 W2 row from L2 (see floors); HBM sees W2 at most once."""
    V, K, bs = cfg["V"], cfg["K"], cfg["bs"]
    w2 = V * row_bytes(cfg) + (4 * V if cfg["int8"] else 0)
    base = bs * K * V * 2
    emb = bs * K * R * 2
    out = bs * K * 4 + (bs * K * V * 2 if cfg["logits"] else 0)
    return float(w2 + base + emb + out)


def gathered_bytes(cfg) -> float:
    """Bytes of the candidate rows the top-k walk gathers (from L2): one W2 row per
    candidate, request row and position (int8 rows carry their fp32 scale)."""
    k = cfg["top_k"]
    return float(cfg["bs"] * cfg["K"] * k * (row_bytes(cfg) + (4 if cfg["int8"] else 0)))


def uses_tensor_cores(cfg) -> bool:
    return cfg["top_k"] == 0 and cfg["bs"] >= 3


def contraction_flops(cfg) -> float:
    """The method's multiply-adds (2 flops each): every vocabulary row (top-k: every
    candidate) against every request row's embedding, at every position."""
    rows = cfg["top_k"] if cfg["top_k"] else cfg["V"]
    return 2.0 * rows * R * cfg["bs"] * cfg["K"]


def floors(cfg, peaks, sms: int, resident_rows: int, l2_gbs: float):
    """Lower bounds (us) of one walk, per resource. Memory: HBM (W2 once, base logits,
    outputs), shared memory (the resident W2 rows read at every position), L2 (the
    streamed W2 rows at positions 1..K-1; top-k: every gathered candidate row).
    Contraction: the method's flops on the tensor cores (tensor-core walk, bs >= 3) or on
    the fp32 FMA pipe (CUDA-core and top-k walks). The roofline is the slowest of them.
    Sampled walks also get an informational floor for the Gumbel draws ("gumbel_us":
    two logarithms per draw on the multi-function units, or the other instructions of a
    draw at the fp32 issue rate), not part of the roofline."""
    V, K, bs = cfg["V"], cfg["K"], cfg["bs"]
    clk = peaks["sm_mhz"] * 1e6
    out = {"hbm_us": hbm_bytes(cfg) / (peaks["hbm_gbs"] * 1e9) * 1e6}
    if cfg["top_k"]:
        out["l2_us"] = gathered_bytes(cfg) / (l2_gbs * 1e9) * 1e6
        out["fma_us"] = contraction_flops(cfg) / (2 * FFMA_PER_CLK * sms * clk) * 1e6
    else:
        rb = row_bytes(cfg)
        out["smem_us"] = K * resident_rows * rb / (SMEM_B_PER_CLK * sms * clk) * 1e6
        out["l2_us"] = (K - 1) * (V - resident_rows) * rb / (l2_gbs * 1e9) * 1e6
        if uses_tensor_cores(cfg):
            out["tensor_us"] = contraction_flops(cfg) / (peaks["bf16_tflops"] * 1e12) * 1e6
        else:
            out["fma_us"] = contraction_flops(cfg) / (2 * FFMA_PER_CLK * sms * clk) * 1e6
    return out


# One grid-wide exchange of the walk (every CTA's packed atomicMax, the arrival counter,
# the acquire polling until all 152 CTAs have arrived): ~1.4 us, measured on this GPU with
# a probe kernel doing only that exchange, back to back.
GRID_EXCHANGE_US = 1.4


def chain_floor_us(cfg, fl) -> float:
    """Informational latency floor of the walk: position i + 1's contraction needs
    position i's winner, so the K grid exchanges and the contraction are serial; this is
    K exchanges plus the contraction floor (the top-k walk: K exchanges plus its L2 and
    FMA floors' larger). Not part of the roofline (a chain of latencies, not a resource)."""
    work = max(v for k, v in fl.items() if k in ("tensor_us", "fma_us", "l2_us" if cfg["top_k"] else "tensor_us"))
    return cfg["K"] * GRID_EXCHANGE_US + work


def gumbel_floor_us(cfg, peaks, sms: int) -> float | None:
    """Informational floor of the Gumbel draws of a sampled walk (None when greedy)."""
    if cfg["mode"] != 1:
        return None
    draws = float(cfg["bs"] * cfg["K"] * (cfg["top_k"] or cfg["V"]))
    clk = peaks["sm_mhz"] * 1e6
    return max(2 * draws / (MUFU_PER_CLK * sms * clk), GUMBEL_ALU_PER_DRAW * draws / (FFMA_PER_CLK * sms * clk)) * 1e6


def roofline(cfg, peaks, fl, us, sms: int):
    """The roofline object for the slowest floor: achieved = that resource's algorithmic
    work per walk / measured walk time, against its peak."""
    key = max(fl, key=fl.get)
    clk = peaks["sm_mhz"] * 1e6
    if key == "tensor_us":
        ach = contraction_flops(cfg) / (us * 1e-6) / 1e12
        r = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    elif key == "fma_us":
        peak = 2 * FFMA_PER_CLK * sms * clk / 1e12
        r = {"bound": "fma", "achieved": contraction_flops(cfg) / (us * 1e-6) / 1e12, "peak": peak,
             "unit": "TFLOP/s (fp32 FMA)"}
    elif key == "smem_us":
        r = {"bound": "smem", "achieved": fl[key] / us, "peak": 1.0, "unit": "fraction"}
    elif key == "l2_us":
        r = {"bound": "l2", "achieved": fl[key] / us, "peak": 1.0, "unit": "fraction"}
    else:
        ach = hbm_bytes(cfg) / (us * 1e-6) / 1e9
        r = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    return r


def measure_l2_gbs(dev) -> float:
    """Copy bandwidth of a 32 MB buffer that stays in L2 (read + write bytes)."""
    a = torch.empty(32 * 1024 * 1024, dtype=torch.uint8, device=dev)
    b = torch.empty_like(a)
    for _ in range(5):
        b.copy_(a)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(50):
        b.copy_(a)
    e.record()
    torch.cuda.synchronize()
    return 2.0 * a.numel() * 50 / (s.elapsed_time(e) * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def make_inputs(cfg, dev, seed=0):
    from dspark_markov_draft_gb300 import capi, synth
    inp = synth.make(cfg["V"], cfg["bs"], cfg["K"], seed=seed, peak=cfg["peak"])
    t = dict(w1=inp.w1.to(dev), base=inp.base.to(dev), prev=inp.prev.to(dev),
             seeds=inp.seeds.to(dev), inp=inp)
    w2 = inp.w2.to(dev)
    if cfg["int8"]:
        t["w2q"], t["scales"] = capi.quantize_w2(w2)
        del w2
    else:
        t["w2"] = w2
    return t


def make_walk_args(cfg, t, dev):
    from dspark_markov_draft_gb300 import capi
    bs, K, V = cfg["bs"], cfg["K"], cfg["V"]
    t["tokens"] = torch.empty((bs, K), dtype=torch.int32, device=dev)
    t["logits"] = torch.empty((bs, K, V), dtype=torch.bfloat16, device=dev) if cfg["logits"] else None
    t["ws"] = capi.alloc_workspace(V, bs, K, cfg["top_k"], device=dev)
    return capi.make_args(t["base"], t["w1"], t["prev"], t["tokens"], t["ws"], w2=t.get("w2"),
                          w2q=t.get("w2q"), scales=t.get("scales"), seeds=t["seeds"],
                          mode=cfg["mode"], temperature=cfg["T"], top_k=cfg["top_k"],
                          logits=t["logits"])


def time_walks(cfg, steps, warmup, dev, flush):
    """Per-walk CUDA-event times (ms) of `steps` walks, L2 flushed before each."""
    from dspark_markov_draft_gb300 import capi
    t = make_inputs(cfg, dev)
    args = make_walk_args(cfg, t, dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        st = capi.walk_args_call(args, stream)
        if st:
            raise RuntimeError(f"walk failed: {capi.STATUS.get(st, st)}")
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        flush.zero_()
        s.record(stream)
        capi.walk_args_call(args, stream)
        e.record(stream)
    torch.cuda.synchronize()
    times = [s.elapsed_time(e) for s, e in evs]
    return times, t, args


def time_graph(args, steps, flush, cold=True):
    """The same walk captured once in a CUDA graph and replayed: per-replay CUDA-event
    times (ms), the L2 flushed before each replay (outside the events), as the pages'
    kernel benchmark replays a graph of one walk; cold=False: no flush (warm L2, the
    inputs of the previous replay still cached where they fit)."""
    from dspark_markov_draft_gb300 import capi
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = capi.walk_args_call(args, torch.cuda.current_stream())
    if st:
        raise RuntimeError(f"walk capture failed: {capi.STATUS.get(st, st)}")
    for _ in range(3):
        if cold:
            flush.zero_()
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        if cold:
            flush.zero_()
        s.record(stream)
        g.replay()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def time_verify(dev, flush, peaks, steps, V=151936, K=7, bs=64, T=1.0):
    """Speculative-sampling verification of K drafted tokens per row (dspark_verify) on
    synthetic bf16 logits: draft logits N(0, 3^2), target logits the draft logits plus
    N(0, 0.3^2) noise (so that acceptances and rejections both occur), an independent
    bonus row, draft tokens drawn from softmax(draft / T). Per-call CUDA-event times
    with the L2 flushed before each call; the floor is one read of both logit tensors."""
    from dspark_markov_draft_gb300 import capi
    g = torch.Generator(device=dev).manual_seed(7)
    drf = (torch.randn(bs, K, V, generator=g, device=dev) * 3).to(torch.bfloat16)
    tgt = (torch.cat([drf.float(), torch.randn(bs, 1, V, generator=g, device=dev) * 3], 1)
           + torch.randn(bs, K + 1, V, generator=g, device=dev) * 0.3).to(torch.bfloat16)
    q = torch.softmax(drf.float() / T, -1)
    dtok = torch.stack([torch.multinomial(q[:, i], 1, generator=g)[:, 0] for i in range(K)], 1).to(torch.int32)
    del q
    seeds = torch.arange(bs, device=dev, dtype=torch.int64) * 3 + 1
    acc = torch.empty(bs, dtype=torch.int32, device=dev)
    out = torch.empty((bs, K + 1), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        flush.zero_()
        capi.verify(tgt, drf, dtok, seeds, T, accepted=acc, out_tokens=out, stream=stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in evs:
        flush.zero_()
        s.record(stream)
        capi.verify(tgt, drf, dtok, seeds, T, accepted=acc, out_tokens=out, stream=stream)
        e.record(stream)
    torch.cuda.synchronize()
    us = 1000 * statistics.median([s.elapsed_time(e) for s, e in evs])
    nbytes = (tgt.numel() + drf.numel()) * 2
    floor_us = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    return {"workload": f"verify v{V} k{K} bs{bs} T={T}", "us_per_call": us, "calls": steps,
            "hbm_bytes": nbytes, "floor_us": floor_us, "frac_of_floor": floor_us / us,
            "mean_accepted": float(acc.float().mean()), "kernels_per_call": 3,
            "l2": "flushed before every call"}


LMHEAD_CASES = [(2048, 512, 7), (2048, 4096, 7), (4096, 512, 7), (2048, 512, 16)]


def time_lmhead(dev, flush, peaks, steps, V=151936, K=7, bs=64, d=2048, k=512):
    """The drafter's LM head fused with the top-k selection (dspark_lmhead_topk: sample
    GEMM, pivot, filter GEMM, select) for bs*K hidden rows of width d, then the top-k walk
    on its candidates (sampled, T=1). Per-call CUDA-event times with the L2 flushed before
    each call. Roofline: the dense LM-head product's flops (2 M V d) on the tensor cores;
    the HBM floor is one read of the LM head and the hidden rows."""
    from dspark_markov_draft_gb300 import capi, synth
    M = bs * K
    hidden, head = synth.lmhead(M, d, V, seed=1)
    hidden, head = hidden.to(dev), head.to(dev)
    inp = synth.make(V, bs, K, seed=0)
    w1, w2, prev, seeds = inp.w1.to(dev), inp.w2.to(dev), inp.prev.to(dev), inp.seeds.to(dev)
    cand = torch.empty((M, k), dtype=torch.int32, device=dev)
    cbase = torch.empty((M, k), dtype=torch.float32, device=dev)
    ws = capi.lmhead_workspace(M, V, k, device=dev)
    stats = torch.zeros(2, dtype=torch.int32, device=dev)
    tokens = torch.empty((bs, K), dtype=torch.int32, device=dev)
    wws = capi.alloc_workspace(V, bs, K, k, device=dev)
    wargs = capi.make_args(None, w1, prev, tokens, wws, w2=w2, seeds=seeds, mode=capi.PROBABILISTIC,
                           temperature=1.0, top_k=k, topk_cand=cand.view(bs, K, k),
                           topk_base=cbase.view(bs, K, k), V=V)
    stream = torch.cuda.current_stream()

    def head_call():
        capi.lmhead_topk(hidden, head, k, cand=cand, cand_base=cbase, workspace=ws, stats=stats, stream=stream)

    def timed(fn, n):
        for _ in range(3):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for s_, e_ in evs:
            flush.zero_()
            s_.record(stream)
            fn()
            e_.record(stream)
        torch.cuda.synchronize()
        return 1000 * statistics.median([s_.elapsed_time(e_) for s_, e_ in evs])

    def both():
        head_call()
        st = capi.walk_args_call(wargs, stream, topk=True)
        if st:
            raise RuntimeError(f"top-k walk failed: {capi.STATUS.get(st, st)}")

    us_head = timed(head_call, steps)
    us_both = timed(both, steps)
    flops = 2.0 * M * V * d
    tflops = flops / (us_head * 1e-6) / 1e12
    nbytes = 2.0 * (V * d + M * d)
    return {"workload": f"lmhead d{d} v{V} k{K} bs{bs} top-k {k}", "hidden_rows": M,
            "us_lmhead_topk": us_head, "us_lmhead_topk_plus_walk": us_both,
            "tensor_floor_us": flops / (peaks["bf16_tflops"] * 1e12) * 1e6,
            "hbm_floor_us": nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"]},
            "rows_on_exact_path": int(stats[0].item()), "kernels_per_call": 4 + 2,
            "l2": "flushed before every call"}


def time_e2e(cfg, t, args, steps, dev):
    """Walk through dspark_walk_from_host: per-step H2D of base/prev/seeds from pinned
    host memory, the walk, D2H of the tokens; timed with events around all of it. Two
    sets of device buffers on two streams, steps alternating between them (double
    buffering by the caller), so that one step's copies run while the other's walk runs;
    the copy engine is shared, so the copies themselves stay in sequence."""
    from dspark_markov_draft_gb300 import capi
    inp = t["inp"]
    base_h = inp.base.pin_memory()
    prev_h = inp.prev.pin_memory()
    seeds_h = inp.seeds.pin_memory()
    tok_h = [torch.empty((cfg["bs"], cfg["K"]), dtype=torch.int32).pin_memory() for _ in range(2)]
    t2 = dict(inp=inp, w1=t["w1"], w2=t.get("w2"), w2q=t.get("w2q"), scales=t.get("scales"),
              base=torch.empty_like(t["base"]), prev=torch.empty_like(t["prev"]), seeds=torch.empty_like(t["seeds"]))
    args2 = make_walk_args(cfg, t2, dev)
    arg_sets = [args, args2]
    main = torch.cuda.current_stream()
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    for j in range(2):
        capi.walk_from_host(arg_sets[j], base_h, prev_h, seeds_h, tok_h[j], None, streams[j])
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(main)
    for st in streams:
        st.wait_event(s)
    for j in range(steps):
        capi.walk_from_host(arg_sets[j % 2], base_h, prev_h, seeds_h, tok_h[j % 2], None, streams[j % 2])
    for st in streams:
        ev = torch.cuda.Event()
        ev.record(st)
        main.wait_event(ev)
    e.record(main)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    h2d = base_h.numel() * 2 + prev_h.numel() * 4 + seeds_h.numel() * 8
    d2h = tok_h[0].numel() * 4
    return ms, h2d, d2h


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest replica's time (every rank walks its own batch; the job ends with the
    slowest one)."""
    if dist is None:
        return ms
    x = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return float(x.item())


def job_throughput(ms_max: float, world: int, tokens_per_rank: int) -> float:
    """Draft tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms_max * 1e-3)


def cpu_model() -> str:
    """The host CPU's model name (and architecture), for the oracle baseline."""
    import platform
    name = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                name = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not name:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        name = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return f"{name or 'unknown'} ({platform.machine()})"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleRunner:
    """The CPU oracle (fp64, OpenMP over rows and vocabulary) on `rows` request rows of
    the workload, all K positions, inputs prepared once."""

    def __init__(self, cfg, rows: int):
        from dspark_markov_draft_gb300 import synth
        from oracle import oracle as O
        O.build()
        self.O, self.cfg, self.rows = O, cfg, rows
        inp = synth.make(cfg["V"], rows, cfg["K"], seed=0, peak=cfg["peak"])
        b = inp.bits
        if cfg["int8"]:
            _, q, sc = O.quantize_w2(b(inp.w2))
            self.kw = dict(w2q=q, scales=sc)
        else:
            self.kw = dict(w2_bits=b(inp.w2))
        self.base, self.w1 = b(inp.base), b(inp.w1)
        self.prev = inp.prev.numpy()
        self.seeds = inp.seeds.numpy().astype(np.uint64)

    def parity(self, gpu_tokens, nthreads: int) -> dict:
        """Teacher-forced check of the GPU's tokens of these inputs (every row): at each
        step the GPU token is the oracle's, a near tie (within 1e-3 of the best score),
        a bf16-boundary case, or rejected."""
        c = self.cfg
        follow = np.ascontiguousarray(gpu_tokens, dtype=np.int32)
        r = self.O.walk(self.base, self.w1, self.prev, c["K"], seeds=self.seeds, mode=c["mode"],
                        temperature=c["T"], top_k=c["top_k"], follow=follow, nthreads=nthreads, **self.kw)
        cls = r.follow_class
        return {"steps": int(cls.size), "same": int((cls == self.O.CLASS_SAME).sum()),
                "near_tie": int((cls == self.O.CLASS_NEAR_TIE).sum()),
                "bf16_boundary": int((cls == self.O.CLASS_BF16_BOUNDARY).sum()),
                "rejected": int((cls == self.O.CLASS_REJECTED).sum()), "tie_tol": 1e-3, "bf16_eps": 1e-4}

    def run(self, rows: int, nthreads: int) -> float:
        """Seconds for a walk of the first `rows` rows."""
        c = self.cfg
        t0 = time.perf_counter()
        r = self.O.walk(self.base[:rows], self.w1, self.prev[:rows], c["K"],
                        seeds=self.seeds[:rows], mode=c["mode"], temperature=c["T"],
                        top_k=c["top_k"], nthreads=nthreads, **self.kw)
        dt = time.perf_counter() - t0
        if r.status != 0:
            raise RuntimeError(f"oracle walk status {r.status}")
        return dt


def cpu_baseline(cfg, gpu_tokens=None, target_s: float = 10.0, single_s: float = 3.0):
    """The oracle on the host cores, on a bounded sample of the workload: all cores
    (OpenMP over the vocabulary) on whole request rows (all K positions) for about
    `target_s` seconds, and one core on single rows for about `single_s` seconds. When
    the GPU's tokens of the same inputs are given, the same leg also checks them against
    the oracle, teacher-forced over every row (the parity counts)."""
    cores = host_cores()
    runner = OracleRunner(cfg, cfg["bs"])
    t1 = runner.run(1, cores)
    rows = int(min(cfg["bs"], max(1, target_s / max(t1, 1e-6))))
    reps = 1 if rows < cfg["bs"] else int(min(20, max(1, target_s / max(rows * t1, 1e-6))))
    dt = sum(runner.run(rows, cores) for _ in range(reps))
    toks = reps * rows * cfg["K"]
    out = {"value": toks / dt, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu": cpu_model(),
           "sample": f"{reps} x {rows} of {cfg['bs']} request rows, all {cfg['K']} positions, "
                     f"{dt:.1f} s of oracle time"}
    s1 = runner.run(1, 1)
    reps1 = int(max(1, min(20, single_s / max(s1, 1e-6)))) - 1
    s1 += sum(runner.run(1, 1) for _ in range(reps1))
    out["single_thread"] = {"value": (reps1 + 1) * cfg["K"] / s1, "unit": UNIT, "cores": 1,
                            "sample": f"{reps1 + 1} x 1 request row, all {cfg['K']} positions, {s1:.1f} s"}
    if gpu_tokens is not None:
        out["parity"] = runner.parity(gpu_tokens, cores)
    return out


def reference_arm(a, rank, world):
    """The oracle timed on the host cores as the reference arm: each step walks a bounded
    sample of the main workload's request rows (all K positions)."""
    if rank != 0:
        return 0
    cores = host_cores()
    cfg = MAIN
    runner = OracleRunner(cfg, cfg["bs"])
    t1 = runner.run(1, cores)
    rows = int(min(cfg["bs"], max(1, 2.0 / max(t1, 1e-6))))  # about 2 s per step
    for _ in range(a.warmup):
        runner.run(rows, cores)
    ts = [runner.run(rows, cores) for _ in range(a.steps)]
    value = a.steps * rows * cfg["K"] / sum(ts)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000 * statistics.mean(ts),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": cfg["name"], "V": cfg["V"], "K": cfg["K"], "bs": cfg["bs"],
                   "w2": "int8", "mode": "greedy", "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows} of {cfg['bs']} request rows, all {cfg['K']} positions, per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


KERNEL_SOURCES = {
    "walk_tc_kernel": ["walk_tc.cu", "common.cuh", "walk_params.cuh"],
    "walk_cc_kernel": ["walk_cc.cu", "common.cuh", "walk_params.cuh"],
    "topk_walk_kernel": ["topk.cu", "common.cuh", "walk_params.cuh"],
}


def kernel_name(cfg) -> str:
    if cfg["top_k"]:
        return "topk_walk_kernel"
    return "walk_tc_kernel" if uses_tensor_cores(cfg) else "walk_cc_kernel"


def sources_digest(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "dspark_markov_draft_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(cfg):
    """DRAM bytes per launch from the committed ncu capture of this workload's kernel,
    or None when there is none or the kernel's sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(cfg["name"])
    k = kernel_name(cfg)
    if not rec or rec.get("kernel") != k or rec.get("sources_sha256_16") != sources_digest(k):
        return None
    return float(rec["dram_bytes_per_launch"])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-verify", action="store_true")
    ap.add_argument("--no-lmhead", action="store_true")
    ap.add_argument("--workload", default=MAIN["name"],
                    help="run this workload as the main line (one of the built-in names)")
    a = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if a.impl == "reference":
        return reference_arm(a, rank, world)

    from dspark_markov_draft_gb300 import build, capi
    build.build()
    capi.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 129 MB L2
    by_name = {c["name"]: c for c in [MAIN] + VARIANTS}
    cfg = by_name[a.workload]

    def floors_of(c):
        res = 0
        if not c["top_k"]:
            _, res = capi.query_capacity(local, c["V"], c["int8"], c["bs"])
        fl = floors(c, peaks, sms, res, l2_gbs)
        return fl, res

    def kernels_per_walk(c):
        return 2 if c["top_k"] else 1

    l2_gbs = measure_l2_gbs(dev)
    # untimed warm-up of the whole path, then the timed walks
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        times, t, args = time_walks(cfg, a.steps, a.warmup, dev, flush)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    ms = max_over_ranks(statistics.mean(times), dist, dev)
    toks = cfg["bs"] * cfg["K"]
    value = job_throughput(ms, world, toks)

    e2e_ms, h2d, d2h = (float("nan"), 0, 0) if a.no_e2e else time_e2e(cfg, t, args, max(3, a.steps // 2), dev)
    graph_times = time_graph(args, max(200, a.steps), flush)  # outside the timed region
    graph_warm = time_graph(args, max(200, a.steps), flush, cold=False)
    verify = None if a.no_verify else time_verify(dev, flush, peaks, max(5, a.steps))
    lmhead = [] if a.no_lmhead else [time_lmhead(dev, flush, peaks, max(5, a.steps), K=K_, d=d_, k=k_)
                                     for d_, k_, K_ in LMHEAD_CASES]
    fl, res_rows = floors_of(cfg)
    us = 1000 * ms
    roof = roofline(cfg, peaks, fl, us, sms)
    roof["traffic"] = recorded_traffic(cfg)
    roof["peak_source"] = f"{peaks['src']} (MEASURED_PEAKS.json)" if peaks["src"] == "measured" else "fallback"
    roof["kernel"] = kernel_name(cfg)
    floor_us = max(fl.values())
    floor_rec = {k: round(v, 3) for k, v in fl.items()}
    floor_rec.update({"floor_us": round(floor_us, 3), "floor_sum_us": round(sum(fl.values()), 3),
                      "frac_of_floor": floor_us / us,
                      "resident_w2_rows": res_rows, "l2_gbs_live": round(l2_gbs, 1),
                      "hbm_bytes": hbm_bytes(cfg), "gumbel_us_informational": gumbel_floor_us(cfg, peaks, sms),
                      "chain_us_informational": round(chain_floor_us(cfg, fl), 3)})

    variants = []
    if not a.no_variants:
        for vc in VARIANTS:
            if vc["name"] == cfg["name"]:
                continue
            vt, vtens, _ = time_walks(vc, max(5, a.steps // 2), 3, dev, flush)
            del vtens
            torch.cuda.empty_cache()
            vus = 1000 * statistics.mean(vt)
            vfl, vres = floors_of(vc)
            vfloor = max(vfl.values())
            vr = roofline(vc, peaks, vfl, vus, sms)
            variants.append({"workload": vc["name"], "us_per_walk": vus,
                             "draft_tokens_per_s": vc["bs"] * vc["K"] / (vus * 1e-6),
                             "kernel": kernel_name(vc), "kernels_per_walk": kernels_per_walk(vc),
                             "floor_us": vfloor, "frac_of_floor": vfloor / vus,
                             "bound": vr["bound"], "frac": vr["frac"],
                             "floors_us": {k: round(v, 3) for k, v in vfl.items()},
                             "gumbel_us_informational": gumbel_floor_us(vc, peaks, sms),
                             "chain_us_informational": round(chain_floor_us(vc, vfl), 3)})

    cpu = None
    if rank == 0 and not a.no_cpu_baseline:
        cpu = cpu_baseline(cfg, gpu_tokens=t["tokens"].cpu().numpy())

    if rank == 0:
        tc = uses_tensor_cores(cfg)
        dtype = (("int8 W2 codes as fp16 x fp16 embedding, fp32 accumulate (tcgen05)" if cfg["int8"]
                  else "bf16 x bf16, fp32 accumulate (tcgen05)") if tc else
                 ("int8 x 24-bit integer embedding (dp4a), fp32 epilogue" if cfg["int8"]
                  else "bf16 x bf16, fp32 FMA"))
        parity = (cpu or {}).get("parity")
        if cpu and "parity" in cpu:
            cpu = {k: v for k, v in cpu.items() if k != "parity"}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": {"workload": cfg["name"], "V": cfg["V"], "rank": R, "K": cfg["K"],
                       "bs": cfg["bs"], "w2": "int8" if cfg["int8"] else "bf16",
                       "mode": "greedy" if cfg["mode"] == 0 else f"probabilistic T={cfg['T']}",
                       "top_k": cfg["top_k"], "draft_logits": cfg["logits"],
                       "l2": "flushed before every walk (256 MB write)",
                       "parallelism": f"replicas x{world}"},
            "us_per_walk": us,
            "graph": {"us_per_walk": 1000 * statistics.median(graph_times), "replays": len(graph_times),
                      "l2": "flushed before every replay",
                      "warm_us_per_walk": 1000 * statistics.median(graph_warm),
                      "warm": "no flush between replays"},
            "device": {"name": torch.cuda.get_device_name(dev), "sms_used": sms,
                       "sharing": "one process on the GPU"},
            "roofline": roof,
            "floors": floor_rec,
            "verify": verify,
            "lmhead_topk": lmhead,
            "cpu_baseline": cpu,
            "e2e": {"value": world * toks / (e2e_ms * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipelining": "two buffer sets on two streams, steps alternating"},
            "parity": parity,
            "gpu_launches": a.steps * kernels_per_walk(cfg),
            "clocks": clk.summary(),
            "wall_s_timed": wall,
            "variants": variants,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
