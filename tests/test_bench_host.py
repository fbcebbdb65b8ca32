"""Host-side arithmetic of bench.py's report: the algorithmic bytes of a walk counted by
hand, and the roofline object's choice of the slowest floor and its fraction."""
from __future__ import annotations

import pytest

import bench


def test_hbm_bytes_of_the_main_workload_by_hand():
    V, K, bs = 151936, 7, 64
    w2 = V * 256 + 4 * V           # int8 codes + one fp32 scale per row, read once
    base = bs * K * V * 2          # every bf16 base logit once
    emb = bs * K * 256 * 2         # one W1 row per request and position
    tokens = bs * K * 4
    assert bench.hbm_bytes(bench.MAIN) == w2 + base + emb + tokens


def test_hbm_bytes_count_draft_logits_and_top_k_candidates():
    cfg = dict(bench.MAIN, logits=True)
    assert bench.hbm_bytes(cfg) - bench.hbm_bytes(bench.MAIN) == 64 * 7 * 151936 * 2
    tk = dict(bench.MAIN, top_k=512, int8=False)
    # HBM: bf16 W2 at most once and the base logits; the gathered candidate rows are L2 work
    assert bench.hbm_bytes(tk) == 151936 * 512 + 64 * 7 * 151936 * 2 + 64 * 7 * 256 * 2 + 64 * 7 * 4
    assert bench.gathered_bytes(tk) == 64 * 7 * 512 * 512


PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, sm_mhz=2000.0, src="fallback")


def test_roofline_takes_the_slowest_floor_and_its_fraction():
    cfg = bench.MAIN
    fl = bench.floors(cfg, PEAKS, sms=152, resident_rows=100_000, l2_gbs=20_000.0)
    assert set(fl) == {"hbm_us", "smem_us", "l2_us", "tensor_us"}
    slowest = max(fl, key=fl.get)
    us = 4 * fl[slowest]
    r = bench.roofline(cfg, PEAKS, fl, us, sms=152)
    assert r["frac"] == pytest.approx(fl[slowest] / us)  # a quarter of the floor's speed
    if slowest == "hbm_us":
        assert r["bound"] == "hbm" and r["unit"] == "GB/s"
        assert r["achieved"] * 1e9 * us * 1e-6 == pytest.approx(bench.hbm_bytes(cfg))


def test_small_batches_take_the_fp32_contraction_floor():
    """bs <= 2: the method's multiply-adds at the fp32 FMA pipe's peak (128 lanes per SM
    and clock, two flops each) -- not the implementation's byte limbs."""
    cfg = dict(bench.MAIN, bs=1)
    fl = bench.floors(cfg, PEAKS, sms=152, resident_rows=150_000, l2_gbs=20_000.0)
    assert "fma_us" in fl and "tensor_us" not in fl
    flops = 2.0 * 151936 * 256 * 7
    assert bench.contraction_flops(cfg) == flops
    assert fl["fma_us"] == pytest.approx(flops / (2 * 128 * 152 * 2000e6) * 1e6)
    r = bench.roofline(cfg, PEAKS, {"fma_us": fl["fma_us"]}, 2 * fl["fma_us"], sms=152)
    assert r["bound"] == "fma" and r["frac"] == pytest.approx(0.5)


def test_top_k_floors_put_gathered_rows_on_l2():
    tk = dict(bench.MAIN, top_k=4096, int8=False, mode=1)
    fl = bench.floors(tk, PEAKS, sms=152, resident_rows=0, l2_gbs=8_000.0)
    assert fl["l2_us"] == pytest.approx(64 * 7 * 4096 * 512 / 8e12 * 1e6)
    assert fl["hbm_us"] == pytest.approx(bench.hbm_bytes(tk) / 6.8e12 * 1e6)
    assert bench.gumbel_floor_us(tk, PEAKS, 152) > 0
    assert bench.gumbel_floor_us(bench.MAIN, PEAKS, 152) is None


def test_variants_cover_every_configuration():
    names = {c["name"] for c in bench.VARIANTS} | {bench.MAIN["name"]}
    assert len(names) == len(bench.VARIANTS) + 1
    vs = [bench.MAIN] + bench.VARIANTS
    assert any(c["V"] == 129280 and c["K"] == 5 and c["bs"] == 1 and not c["int8"] for c in vs)
    assert {c["bs"] for c in vs if c["V"] == 151936 and c["K"] == 7 and c["int8"]} == {1, 16, 64}
    assert {c["bs"] for c in vs if c["V"] == 151936 and c["K"] == 16 and c["logits"]} == {1, 64}
    assert {c["bs"] for c in vs if c["V"] == 248320} == {1, 16, 64}
    assert {c["top_k"] for c in vs if c["top_k"]} == {512, 4096}


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores (no GPU) and prints
    one JSON line with the keys the two arms share, plus its sample description."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["config"]["workload"] == bench.MAIN["name"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_chain_floor_adds_the_grid_exchanges_to_the_contraction():
    """K serial grid exchanges plus the contraction floor (informational)."""
    cfg = dict(bench.MAIN, bs=1)
    fl = bench.floors(cfg, PEAKS, sms=152, resident_rows=150_000, l2_gbs=20_000.0)
    assert bench.chain_floor_us(cfg, fl) == pytest.approx(7 * bench.GRID_EXCHANGE_US + fl["fma_us"])
    tc = dict(bench.MAIN)
    fl = bench.floors(tc, PEAKS, sms=152, resident_rows=100_000, l2_gbs=20_000.0)
    assert bench.chain_floor_us(tc, fl) == pytest.approx(7 * bench.GRID_EXCHANGE_US + fl["tensor_us"])
    tk = dict(bench.MAIN, top_k=4096, int8=False, mode=1)
    fl = bench.floors(tk, PEAKS, sms=152, resident_rows=0, l2_gbs=8_000.0)
    assert bench.chain_floor_us(tk, fl) == pytest.approx(7 * bench.GRID_EXCHANGE_US + max(fl["l2_us"], fl["fma_us"]))
