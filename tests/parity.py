"""Comparison rules between the CUDA walk and the CPU oracle.

* int8 codes, scales, Philox words: bit-exact (checked by the callers).
* Draft tokens: the oracle walks each checked row step by step. At every step the
  GPU's token must be the oracle's argmax, or lie within 1e-3 of the oracle's best
  score (a near tie), or -- in probabilistic mode only -- be explained by one bf16
  rounding of a logit lying within 1e-4 of a bf16 rounding midpoint. When the token
  is acceptable the oracle continues from it, so one allowed divergence does not
  cascade; a rejected token fails the test.
* Logits: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| where the oracle is finite; -inf,
  +inf and NaN positions must match exactly.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import numpy as np
import torch

TIE_TOL = 1e-3
BF16_EPS = 1e-4
ATOL, RTOL = 2e-2, 1e-2
# Tokens that differ from the oracle's (near ties, bf16-boundary cases) must stay rare:
# at most this fraction of the checked steps (and at least one step allowed per case).
MAX_DIFFERENT_FRACTION = 0.01

# Parity counts of every checked case in this test session, by label (printed in the
# terminal summary by conftest.py).
REPORT: dict = {}


@dataclass
class ParityStats:
    steps: int
    same: int
    near_tie: int
    bf16_boundary: int
    max_abs_err: float = 0.0


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def nthreads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def check_walk(O, inp, gpu_tokens: torch.Tensor, *, mode: int, T: float = 1.0, top_k: int = 0,
               q=None, sc=None, gpu_logits: torch.Tensor | None = None, rows=None,
               base_bits=None, label: str | None = "small and special cases",
               base_f64_all=None) -> ParityStats:
    """Validate GPU tokens (and optional bf16 logits) of the rows `rows` (default all).
    base_f64_all: fp64 [bs, K, V] base logits for the oracle (the LM-head output) instead
    of the bf16 base logits of `inp`."""
    toks = gpu_tokens.detach().cpu().numpy().astype(np.int32)
    bs, K = toks.shape
    rows = np.arange(bs) if rows is None else np.asarray(rows)
    kw = dict(w2q=q, scales=sc) if q is not None else dict(w2_bits=bits(inp.w2))
    if base_f64_all is not None:
        base_rows = None
        kw["base_f64"] = np.ascontiguousarray(base_f64_all[rows])
    else:
        base_rows = (bits(inp.base) if base_bits is None else base_bits)[rows]
    res = O.walk(base_rows, bits(inp.w1), inp.prev.numpy()[rows], K, slot=rows.astype(np.int32),
                 seeds=inp.seeds.numpy().astype(np.uint64)[rows], mode=mode, temperature=T,
                 top_k=top_k, follow=toks[rows], tie_tol=TIE_TOL, bf16_eps=BF16_EPS,
                 nthreads=nthreads(), want_logits=gpu_logits is not None, **kw)
    assert res.status == 0, res.status
    cls = res.follow_class
    bad = np.argwhere(cls == O.CLASS_REJECTED)
    assert bad.size == 0, (
        f"GPU tokens rejected at (row, step) {bad[:5].tolist()}: gpu "
        f"{[int(toks[rows[r], i]) for r, i in bad[:5]]} oracle "
        f"{[int(res.tokens[r, i]) for r, i in bad[:5]]} gap {[float(res.gap[r, i]) for r, i in bad[:5]]}")
    st = ParityStats(int(cls.size), int((cls == 0).sum()), int((cls == 1).sum()), int((cls == 2).sum()))
    different = st.near_tie + st.bf16_boundary
    assert different <= max(1, MAX_DIFFERENT_FRACTION * st.steps), (
        f"{different} of {st.steps} tokens differ from the oracle's (near ties {st.near_tie}, "
        f"bf16-boundary {st.bf16_boundary})")
    if gpu_logits is not None:
        g = gpu_logits.detach()[torch.as_tensor(rows, device=gpu_logits.device)].cpu().double().numpy()
        r = res.logits
        fin = np.isfinite(r)
        assert np.array_equal(np.isnan(g), np.isnan(r)), "NaN positions differ"
        assert np.array_equal(np.isposinf(g), np.isposinf(r)), "+inf positions differ"
        assert np.array_equal(np.isneginf(g), np.isneginf(r)), "-inf positions differ"
        err = np.abs(g[fin] - r[fin])
        lim = ATOL + RTOL * np.abs(r[fin])
        worst = int(np.argmax(err - lim)) if err.size else 0
        assert np.all(err <= lim), f"logit error {err[worst]} > {lim[worst]}"
        st.max_abs_err = float(err.max()) if err.size else 0.0
    return record(label, st) if label else st


def record(label: str, st: ParityStats) -> ParityStats:
    """Add a case's counts to the session report."""
    tot = REPORT.setdefault(label, ParityStats(0, 0, 0, 0))
    tot.steps += st.steps
    tot.same += st.same
    tot.near_tie += st.near_tie
    tot.bf16_boundary += st.bf16_boundary
    tot.max_abs_err = max(tot.max_abs_err, st.max_abs_err)
    return st


def check_walk_rows(O, inp, gpu_tokens, *, label: str, chunk: int = 8, rows_subset=None, **kw) -> ParityStats:
    """check_walk over every row (or the rows of `rows_subset`), a few rows at a time
    (bounded fp64 logit buffers), with the summed counts recorded under `label`."""
    all_rows = list(range(gpu_tokens.shape[0])) if rows_subset is None else list(rows_subset)
    tot = ParityStats(0, 0, 0, 0)
    for r0 in range(0, len(all_rows), chunk):
        st = check_walk(O, inp, gpu_tokens, rows=all_rows[r0:r0 + chunk], label=None, **kw)
        tot.steps += st.steps
        tot.same += st.same
        tot.near_tie += st.near_tie
        tot.bf16_boundary += st.bf16_boundary
        tot.max_abs_err = max(tot.max_abs_err, st.max_abs_err)
    different = tot.near_tie + tot.bf16_boundary
    assert different <= max(1, MAX_DIFFERENT_FRACTION * tot.steps), (label, tot)
    return record(label, tot)
