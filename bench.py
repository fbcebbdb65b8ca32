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
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    sm_mhz=float(d.get("sm_max_mhz", 2070.0)), src="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, sm_mhz=2070.0, src="fallback")


# Per-SM issue rates used for the on-chip floors (nominal Blackwell figures): 128 bytes
# of shared memory per clock, 64 dp4a lanes per clock (half the fp32 lanes), 128 fp32
# FMA lanes per clock.
SMEM_B_PER_CLK = 128
DP4A_PER_CLK = 64
FFMA_PER_CLK = 128


def row_bytes(cfg) -> int:
    return R * (1 if cfg["int8"] else 2)


def hbm_bytes(cfg) -> float:
    """Algorithmic HBM bytes of one walk: W2 (+ scales) once, every base logit once, the
    K embedding rows per request, the tokens, and draft_logits when written."""
    V, K, bs = cfg["V"], cfg["K"], cfg["bs"]
    w2 = V * row_bytes(cfg) + (4 * V if cfg["int8"] else 0)
    if cfg["top_k"]:
        w2 = bs * K * cfg["top_k"] * R * 2
    base = bs * K * V * 2
    emb = bs * K * R * 2
    out = bs * K * 4 + (bs * K * V * 2 if cfg["logits"] else 0)
    return float(w2 + base + emb + out)


def uses_tensor_cores(cfg) -> bool:
    return cfg["top_k"] == 0 and cfg["bs"] >= 3


def floors(cfg, peaks, sms: int, resident_rows: int, l2_gbs: float):
    """Lower bounds (µs) of one walk, per resource. Memory: HBM (W2 once, base logits,
    outputs), shared memory (the resident W2 rows read at every position), L2 (the
    streamed W2 rows at positions 1..K-1). Contraction: 2 V 256 bs K flops on the
    tensor cores (bs >= 3), or the dp4a / fp32 FMA instructions of the CUDA-core
    contraction (bs <= 2). The roofline is the slowest of them."""
    V, K, bs = cfg["V"], cfg["K"], cfg["bs"]
    clk = peaks["sm_mhz"] * 1e6
    out = {"hbm_us": hbm_bytes(cfg) / (peaks["hbm_gbs"] * 1e9) * 1e6}
    if cfg["top_k"]:
        return out
    rb = row_bytes(cfg)
    res_b = resident_rows * rb
    out["smem_us"] = K * res_b / (SMEM_B_PER_CLK * sms * clk) * 1e6
    out["l2_us"] = (K - 1) * (V - resident_rows) * rb / (l2_gbs * 1e9) * 1e6
    if uses_tensor_cores(cfg):
        out["tensor_us"] = 2.0 * V * R * bs * K / (peaks["bf16_tflops"] * 1e12) * 1e6
    else:
        ops, lanes = alu_ops(cfg)  # int8: 3 byte limbs of the embedding, one dp4a per 4 codes each
        out["alu_us"] = ops / (lanes * sms * clk) * 1e6
    return out


def alu_ops(cfg) -> tuple[float, int]:
    """(instructions per walk, lanes per clock per SM) of the CUDA-core contraction."""
    n = float(cfg["V"]) * R * cfg["bs"] * cfg["K"]
    return (3.0 * n / 4, DP4A_PER_CLK) if cfg["int8"] else (n, FFMA_PER_CLK)


def roofline(cfg, peaks, fl, us, sms: int):
    """The roofline object for the slowest floor: achieved = that resource's algorithmic
    work per walk / measured walk time, against its peak."""
    key = max(fl, key=fl.get)
    if key == "tensor_us":
        ach = 2.0 * cfg["V"] * R * cfg["bs"] * cfg["K"] / (us * 1e-6) / 1e12
        r = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    elif key == "alu_us":
        ops, lanes = alu_ops(cfg)
        peak = lanes * sms * peaks["sm_mhz"] * 1e6 / 1e9
        r = {"bound": "alu", "achieved": ops / (us * 1e-6) / 1e9, "peak": peak,
             "unit": "G dp4a/s" if cfg["int8"] else "G FMA/s"}
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


def time_graph(args, steps, flush):
    """The same walk captured once in a CUDA graph and replayed: per-replay CUDA-event
    times (ms), the L2 flushed before each replay (outside the events), as the pages'
    kernel benchmark replays a graph of one walk."""
    from dspark_markov_draft_gb300 import capi
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = capi.walk_args_call(args, torch.cuda.current_stream())
    if st:
        raise RuntimeError(f"walk capture failed: {capi.STATUS.get(st, st)}")
    for _ in range(3):
        flush.zero_()
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
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


def cpu_baseline(cfg, target_s: float = 12.0):
    """Oracle throughput on a bounded sample of the workload: enough request rows (all
    K positions) for about `target_s` seconds of CPU work, capped at the whole batch."""
    cores = host_cores()
    runner = OracleRunner(cfg, cfg["bs"])
    t1 = runner.run(1, cores)
    rows = int(min(cfg["bs"], max(1, target_s / max(t1, 1e-6))))
    reps = 1 if rows < cfg["bs"] else int(min(20, max(1, target_s / max(rows * t1, 1e-6))))
    dt = sum(runner.run(rows, cores) for _ in range(reps))
    toks = reps * rows * cfg["K"]
    return {"value": toks / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} x {rows} of {cfg['bs']} request rows, all {cfg['K']} positions, "
                      f"{dt:.1f} s of oracle time"}


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
    by_name = {c["name"]: c for c in [MAIN] + VARIANTS + EXTRA}
    cfg = by_name[a.workload]

    def floors_of(c):
        res = 0
        if not c["top_k"]:
            _, res = capi.query_capacity(local, c["V"], c["int8"], c["bs"])
        fl = floors(c, peaks, sms, res, l2_gbs)
        return fl, res

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
    graph_times = time_graph(args, max(5, a.steps), flush)  # outside the timed region
    verify = None if a.no_verify else time_verify(dev, flush, peaks, max(5, a.steps))
    fl, res_rows = floors_of(cfg)
    us = 1000 * ms
    roof = roofline(cfg, peaks, fl, us, sms)
    roof["traffic"] = recorded_traffic(cfg)
    roof["peak_source"] = f"{peaks['src']} (MEASURED_PEAKS.json)" if peaks["src"] == "measured" else "fallback"
    roof["kernel"] = kernel_name(cfg)
    floor_us = max(fl.values())
    floor_rec = {k: round(v, 3) for k, v in fl.items()}
    floor_rec.update({"floor_us": round(floor_us, 3), "frac_of_floor": floor_us / us,
                      "resident_w2_rows": res_rows, "l2_gbs_live": round(l2_gbs, 1),
                      "hbm_bytes": hbm_bytes(cfg)})

    variants = []
    if not a.no_variants:
        for vc in VARIANTS:
            vt, _, _ = time_walks(vc, max(5, a.steps // 2), 3, dev, flush)
            vus = 1000 * statistics.mean(vt)
            vfl, vres = floors_of(vc)
            vfloor = max(vfl.values())
            vr = roofline(vc, peaks, vfl, vus, sms)
            variants.append({"workload": vc["name"], "us_per_walk": vus,
                             "draft_tokens_per_s": vc["bs"] * vc["K"] / (vus * 1e-6),
                             "kernel": kernel_name(vc), "floor_us": vfloor,
                             "frac_of_floor": vfloor / vus,
                             "bound": vr["bound"], "frac": vr["frac"],
                             "floors_us": {k: round(v, 3) for k, v in vfl.items()}})

    cpu = None
    if rank == 0 and not a.no_cpu_baseline:
        cpu = cpu_baseline(cfg)

    if rank == 0:
        tc = uses_tensor_cores(cfg)
        dtype = (("int8 W2 codes as fp16 x fp16 embedding, fp32 accumulate (tcgen05)" if cfg["int8"]
                  else "bf16 x bf16, fp32 accumulate (tcgen05)") if tc else
                 ("int8 x 24-bit integer embedding (dp4a), fp32 epilogue" if cfg["int8"]
                  else "bf16 x bf16, fp32 FMA"))
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
                      "l2": "flushed before every replay"},
            "roofline": roof,
            "floors": floor_rec,
            "verify": verify,
            "cpu_baseline": cpu,
            "e2e": {"value": world * toks / (e2e_ms * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": a.steps * (2 if cfg["top_k"] else 1),
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
