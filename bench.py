"""Benchmark of the Markov draft walk on one GB300 (or N independent replicas).

A step is one full K-position walk over one batch: the timed region holds exactly the
walk kernel(s) of each step, with an L2 flush (a write of a buffer larger than L2)
between steps outside the per-step CUDA events, so every walk starts with a cold L2 as
in the pages' own kernel benchmark. Inputs are seeded synthetic tensors of the
workload's shapes and distributions, resident in HBM before timing starts.

Default workload: V=151936, rank 256, K=7, bs=64, int8 W2 (per-row fp32 scales),
greedy, base logits N(0, 3^2) with one +8 peak per row and position. Further lines of
the same configuration family (bs 1 and 16, probabilistic T=1) are reported under
"variants".

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
VARIANTS = [
    dict(name="v151936_k7_bs1_int8_greedy", V=151936, K=7, bs=1, int8=True, mode=0, T=1.0, top_k=0, peak=8.0, logits=False),
    dict(name="v151936_k7_bs1_int8_prob", V=151936, K=7, bs=1, int8=True, mode=1, T=1.0, top_k=0, peak=8.0, logits=False),
    dict(name="v151936_k7_bs16_int8_greedy", V=151936, K=7, bs=16, int8=True, mode=0, T=1.0, top_k=0, peak=8.0, logits=False),
    dict(name="v151936_k7_bs64_int8_prob", V=151936, K=7, bs=64, int8=True, mode=1, T=1.0, top_k=0, peak=8.0, logits=False),
]


# Further workloads that can be selected with --workload (parity cases, not bench lines).
EXTRA = [
    dict(name="v129280_k5_bs1_bf16_greedy", V=129280, K=5, bs=1, int8=False, mode=0, T=1.0, top_k=0, peak=None, logits=False),
    dict(name="v151936_k16_bs1_bf16_prob_logits", V=151936, K=16, bs=1, int8=False, mode=1, T=0.7, top_k=0, peak=8.0, logits=True),
    dict(name="v151936_k16_bs64_bf16_prob_logits", V=151936, K=16, bs=64, int8=False, mode=1, T=0.7, top_k=0, peak=8.0, logits=True),
    dict(name="v248320_k16_bs1_int8_greedy", V=248320, K=16, bs=1, int8=True, mode=0, T=1.0, top_k=0, peak=None, logits=False),
    dict(name="v248320_k16_bs64_int8_greedy", V=248320, K=16, bs=64, int8=True, mode=0, T=1.0, top_k=0, peak=None, logits=False),
    dict(name="v151936_k7_bs64_topk512_prob", V=151936, K=7, bs=64, int8=False, mode=1, T=1.0, top_k=512, peak=None, logits=False),
    dict(name="v151936_k7_bs64_topk4096_prob", V=151936, K=7, bs=64, int8=False, mode=1, T=1.0, top_k=4096, peak=None, logits=False),
]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), src="measured")
    return dict(hbm_gbs=6800.0, src="fallback")


def hbm_bytes(cfg) -> float:
    """Algorithmic HBM bytes of one walk: W2 (+ scales) once, every base logit once, the
    K embedding rows per request, the tokens, and draft_logits when written."""
    V, K, bs = cfg["V"], cfg["K"], cfg["bs"]
    w2 = V * R * (1 if cfg["int8"] else 2) + (4 * V if cfg["int8"] else 0)
    if cfg["top_k"]:
        w2 = bs * K * cfg["top_k"] * R * 2
    base = bs * K * V * 2
    emb = bs * K * R * 2
    out = bs * K * 4 + (bs * K * V * 2 if cfg["logits"] else 0)
    return float(w2 + base + emb + out)


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


def time_e2e(cfg, t, args, steps, dev):
    """Walk through dspark_walk_from_host: per-step H2D of base/prev/seeds from pinned
    host memory, the walk, D2H of the tokens; timed with events around all of it."""
    from dspark_markov_draft_gb300 import capi
    inp = t["inp"]
    base_h = inp.base.pin_memory()
    prev_h = inp.prev.pin_memory()
    seeds_h = inp.seeds.pin_memory()
    tok_h = torch.empty((cfg["bs"], cfg["K"]), dtype=torch.int32).pin_memory()
    stream = torch.cuda.current_stream()
    for _ in range(2):
        capi.walk_from_host(args, base_h, prev_h, seeds_h, tok_h, None, stream)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        capi.walk_from_host(args, base_h, prev_h, seeds_h, tok_h, None, stream)
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    h2d = base_h.numel() * 2 + prev_h.numel() * 4 + seeds_h.numel() * 8
    d2h = tok_h.numel() * 4
    return ms, h2d, d2h


def oracle_sample(cfg, rows: int, nthreads: int):
    """Time the CPU oracle on `rows` request rows of the workload (all K positions)."""
    from dspark_markov_draft_gb300 import synth
    from oracle import oracle as O
    O.build()
    inp = synth.make(cfg["V"], rows, cfg["K"], seed=0, peak=cfg["peak"])
    b = inp.bits
    kw = {}
    if cfg["int8"]:
        st, q, sc = O.quantize_w2(b(inp.w2))
        kw = dict(w2q=q, scales=sc)
    else:
        kw = dict(w2_bits=b(inp.w2))
    t0 = time.perf_counter()
    O.walk(b(inp.base), b(inp.w1), inp.prev.numpy(), cfg["K"],
           seeds=inp.seeds.numpy().astype(np.uint64), mode=cfg["mode"], temperature=cfg["T"],
           top_k=cfg["top_k"], nthreads=nthreads, **kw)
    dt = time.perf_counter() - t0
    return dt, rows * cfg["K"]


def reference_arm(a, rank, world):
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    cfg = MAIN
    rows = 1
    for _ in range(a.warmup):
        oracle_sample(cfg, rows, cores)
    ts = []
    toks = 0
    for _ in range(a.steps):
        dt, n = oracle_sample(cfg, rows, cores)
        ts.append(dt)
        toks += n
    value = toks / sum(ts)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000 * statistics.mean(ts),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": cfg["name"], "V": cfg["V"], "K": cfg["K"], "bs": cfg["bs"],
                   "w2": "int8", "mode": "greedy", "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows} of {cfg['bs']} request rows, all {cfg['K']} positions, per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
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
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 129 MB L2
    by_name = {c["name"]: c for c in [MAIN] + VARIANTS + EXTRA}
    cfg = by_name[a.workload]
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
    ms = statistics.mean(times)
    if dist:
        x = torch.tensor([ms], device=dev)
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        ms = float(x.item())
    toks = cfg["bs"] * cfg["K"]
    value = world * toks / (ms * 1e-3)

    e2e_ms, h2d, d2h = (float("nan"), 0, 0) if a.no_e2e else time_e2e(cfg, t, args, max(3, a.steps // 2), dev)
    hb = hbm_bytes(cfg)
    achieved = hb / (ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": None,
            "peak_source": peaks["src"], "algorithmic_bytes_per_launch": hb}

    variants = []
    if not a.no_variants:
        for vc in VARIANTS:
            vt, _, _ = time_walks(vc, max(5, a.steps // 2), 2, dev, flush)
            vms = statistics.median(vt)
            vhb = hbm_bytes(vc)
            variants.append({"workload": vc["name"], "us_per_walk": 1000 * vms,
                             "draft_tokens_per_s": vc["bs"] * vc["K"] / (vms * 1e-3),
                             "hbm_gbs": vhb / (vms * 1e-3) / 1e9,
                             "hbm_frac": vhb / (vms * 1e-3) / 1e9 / peaks["hbm_gbs"]})

    cpu = None
    if rank == 0 and not a.no_cpu_baseline:
        cores = os.cpu_count() or 1
        dt, n = oracle_sample(cfg, 1, cores)
        cpu = {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"1 of {cfg['bs']} request rows, all {cfg['K']} positions ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8 x int (dp4a) -> fp32", "data": "synthetic",
            "config": {"workload": cfg["name"], "V": cfg["V"], "rank": R, "K": cfg["K"],
                       "bs": cfg["bs"], "w2": "int8" if cfg["int8"] else "bf16",
                       "mode": "greedy" if cfg["mode"] == 0 else f"probabilistic T={cfg['T']}",
                       "top_k": cfg["top_k"], "draft_logits": cfg["logits"],
                       "l2": "flushed before every walk (256 MB write)",
                       "parallelism": f"replicas x{world}"},
            "us_per_walk": 1000 * ms,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": world * toks / (e2e_ms * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": a.steps,
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
