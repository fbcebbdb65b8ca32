"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one part of the oracle to a fact fixed by the pages or by
mathematics: hand-derived golden values, library routines on special cases,
closed forms, brute force on tiny inputs, an independent Philox implementation
and the Gumbel-max sampling theorem. None of them needs a GPU.
"""
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns of a list of floats (or 'nan', 'inf', '-inf', '-0')."""
    f = np.array([float(v) for v in values], dtype=np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _eval_expr(s: str) -> float:
    return float(eval(s.replace("^", "**"), {"__builtins__": {}}, {}))


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_golden(oracle):
    cases = json.load(open(os.path.join(GOLDEN, "bf16_rounding.json")))["cases"]
    for c in cases:
        x = -0.0 if c["x"] == "-0.0" else _eval_expr(c["x"])
        assert oracle.round_bf16(x) == int(c["bits"], 16), c


def test_round_bf16_matches_torch_on_fp32_values(oracle):
    # For inputs that are already fp32, torch's fp32 -> bf16 conversion is a single
    # round-to-nearest-even step, so it must agree with the oracle bit for bit.
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * 10,
        (rng.standard_normal(500) * 1e-39).astype(np.float32),   # subnormals
        np.float32(1.0) + rng.integers(0, 2**16, 500).astype(np.float32) * np.float32(2**-16),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)


# ---------------------------------------------------------------- Philox / Gumbel

_TRITON_SCRIPT = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def k(c_ptr, out_ptr, seed, N: tl.constexpr):
    offs = tl.arange(0, N)
    c0 = tl.load(c_ptr + offs * 4 + 0).to(tl.uint32)
    c1 = tl.load(c_ptr + offs * 4 + 1).to(tl.uint32)
    c2 = tl.load(c_ptr + offs * 4 + 2).to(tl.uint32)
    c3 = tl.load(c_ptr + offs * 4 + 3).to(tl.uint32)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + offs * 4 + 0, a)
    tl.store(out_ptr + offs * 4 + 1, b)
    tl.store(out_ptr + offs * 4 + 2, c)
    tl.store(out_ptr + offs * 4 + 3, d)

req = json.loads(sys.stdin.read())
res = []
for seed, ctrs in req:
    c = torch.tensor(np.array(ctrs, dtype=np.uint32).view(np.int32))
    out = torch.zeros_like(c)
    k[(1,)](c, out, seed, N=c.shape[0])
    res.append(out.numpy().view(np.uint32).tolist())
print(json.dumps(res))
"""


def test_philox_matches_independent_implementation(oracle):
    """Philox4x32-10 against triton's own implementation, run by its CPU interpreter."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(1)
    seeds = [0, 1, 0x123456789ABCDEF0, 2**64 - 1, 42]
    req = []
    for s in seeds:
        ctrs = rng.integers(0, 2**32, size=(16, 4), dtype=np.uint64)
        ctrs[0] = [0, 0, 0, 0]
        ctrs[1] = [0xFFFFFFFF] * 4
        req.append([s, ctrs.astype(np.uint32).tolist()])
    p = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(req),
                       capture_output=True, text=True, timeout=300)
    if p.returncode != 0:
        pytest.skip(f"triton interpreter unavailable: {p.stderr[-300:]}")
    res = json.loads(p.stdout.strip().splitlines()[-1])
    for (s, ctrs), outs in zip(req, res):
        key = [s & 0xFFFFFFFF, s >> 32]
        for c, o in zip(ctrs, outs):
            np.testing.assert_array_equal(oracle.philox4x32_10(c, key), np.array(o, np.uint32))


def test_philox_distinct_and_uniform(oracle):
    words, u, g = oracle.gumbel_block(np.array([7, 8], np.uint64), K=3, V=4096)
    w = words.reshape(-1)
    # 24576 outputs of a bijection on distinct counters and keys: collisions of 32-bit
    # words are possible but essentially never more than a handful.
    assert len(np.unique(w)) > len(w) - 5
    # chi-square uniformity of the top 6 bits
    hist = np.bincount((w >> 26).astype(np.int64), minlength=64)
    exp = len(w) / 64
    chi2 = ((hist - exp) ** 2 / exp).sum()
    assert chi2 < 130, chi2  # 63 dof; p ~ 1e-6


def test_uniform_and_gumbel_closed_form(oracle):
    words, u, g = oracle.gumbel_block(np.array([3], np.uint64), K=2, V=2000)
    u64 = u.astype(np.float64)
    assert np.all(u64 > 0) and np.all(u64 < 1)
    m = u64 * 2.0**24
    assert np.all(m == np.round(m)) and np.all(np.round(m) % 2 == 1)   # odd multiples of 2^-24
    # g inverts the Gumbel CDF F(g) = exp(-exp(-g)) at u
    np.testing.assert_allclose(np.exp(-np.exp(-g)), u64, rtol=1e-12, atol=0)
    # monotone in the word's top 23 bits
    order = np.argsort(words.reshape(-1) >> 9, kind="stable")
    assert np.all(np.diff(u64.reshape(-1)[order]) >= 0)


# ---------------------------------------------------------------- quantizer

def test_quantize_golden_rows(oracle):
    spec = json.load(open(os.path.join(GOLDEN, "quantize_rows.json")))
    w = np.stack([bf16_bits(r["w"]) for r in spec["rows"]])
    st, q, sc = oracle.quantize_w2(w)
    assert st == 0
    for r, qq, s in zip(spec["rows"], q, sc):
        assert s == np.float32(r["scale"]), r
        np.testing.assert_array_equal(qq, np.array(r["q"], np.int8), err_msg=r["why"])


def test_quantize_matches_torch(oracle):
    # torch on CPU: fp32 abs-max, fp32 division and torch.round (half to even).
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(300, 256, generator=g) / 16).to(torch.bfloat16)
    w[7] = 0
    w[9, 3] = -w[9].abs().max() * 1.5  # negative row maximum
    wf = w.float()
    scale = wf.abs().amax(dim=1) / 127
    ref_q = torch.where(scale[:, None] == 0, torch.zeros_like(wf),
                        torch.round(wf / scale[:, None]).clamp(-127, 127)).to(torch.int8)
    st, q, sc = oracle.quantize_w2(w.view(torch.int16).numpy().view(np.uint16))
    assert st == 0
    np.testing.assert_array_equal(sc, scale.numpy())
    np.testing.assert_array_equal(q, ref_q.numpy())


def test_quantize_nonfinite_status(oracle):
    w = bf16_bits([1, 2, "inf", 4] + [0] * 4).reshape(1, 8)
    st, _, _ = oracle.quantize_w2(w)
    assert st == 7


# ---------------------------------------------------------------- walk: closed forms

def _int_bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_single_step_integer_inputs_exact(oracle):
    """K = 1 with small integers: logits = base + W2 @ W1[prev] exactly (integer matmul)."""
    rng = np.random.default_rng(2)
    V, R, bs = 37, 16, 5
    w1 = rng.integers(-3, 4, size=(V, R))
    w2 = rng.integers(-4, 5, size=(V, R))
    base = rng.integers(-20, 21, size=(bs, 1, V))
    prev = rng.integers(0, V, size=bs).astype(np.int32)
    res = oracle.walk(_int_bf16(base), _int_bf16(w1), prev, 1, w2_bits=_int_bf16(w2),
                      want_logits=True)
    exp = base[:, 0, :] + (w2 @ w1[prev].T).T
    np.testing.assert_array_equal(res.logits[:, 0, :], exp.astype(np.float64))
    np.testing.assert_array_equal(res.tokens[:, 0], np.argmax(exp, axis=1))


def test_single_step_int8_closed_form(oracle):
    """int8 W2: bias = scale_v * sum_k q[v,k] e_k, exact with power-of-two scales."""
    rng = np.random.default_rng(3)
    V, R, bs = 50, 32, 3
    q = rng.integers(-127, 128, size=(V, R)).astype(np.int8)
    scales = (2.0 ** rng.integers(-9, -4, size=V)).astype(np.float32)
    w1 = rng.integers(-5, 6, size=(V, R))
    base = rng.integers(-8, 9, size=(bs, 1, V))
    prev = rng.integers(0, V, size=bs).astype(np.int32)
    res = oracle.walk(_int_bf16(base), _int_bf16(w1), prev, 1, w2q=q, scales=scales,
                      want_logits=True)
    exp = base[:, 0, :] + scales[None, :].astype(np.float64) * (q.astype(np.int64) @ w1[prev].T).T
    np.testing.assert_array_equal(res.logits[:, 0, :], exp)


def test_rank1_and_onehot_closed_forms(oracle):
    rng = np.random.default_rng(4)
    V, R = 40, 16
    a = rng.integers(-7, 8, size=V)
    c = rng.integers(-7, 8, size=R)
    w2 = np.outer(a, c)                       # |entries| <= 49: exact in bf16
    w1 = rng.integers(-3, 4, size=(V, R))
    base = np.zeros((2, 1, V))
    prev = np.array([3, 11], np.int32)
    res = oracle.walk(_int_bf16(base), _int_bf16(w1), prev, 1, w2_bits=_int_bf16(w2),
                      want_logits=True)
    for r, p in enumerate(prev):
        np.testing.assert_array_equal(res.logits[r, 0], a * float(c @ w1[p]))
    # one-hot embedding row: the bias is one column of W2
    w1h = np.zeros((V, R))
    w1h[5, 9] = 1.0
    res = oracle.walk(_int_bf16(base[:1]), _int_bf16(w1h), np.array([5], np.int32), 1,
                      w2_bits=_int_bf16(w2), want_logits=True)
    np.testing.assert_array_equal(res.logits[0, 0], w2[:, 9].astype(np.float64))


def test_greedy_chain_brute_force(oracle):
    """Exactly one of V^K token sequences satisfies every step's argmax condition."""
    import itertools
    rng = np.random.default_rng(6)
    V, R, K = 5, 8, 3
    for trial in range(6):
        w1 = torch.randn(V, R, generator=torch.Generator().manual_seed(trial)).to(torch.bfloat16)
        w2 = (torch.randn(V, R, generator=torch.Generator().manual_seed(100 + trial))).to(torch.bfloat16)
        base = (torch.randn(1, K, V, generator=torch.Generator().manual_seed(200 + trial)) * 3).to(torch.bfloat16)
        prev = int(rng.integers(0, V))
        W1 = w1.double().numpy(); W2 = w2.double().numpy(); B = base.double().numpy()[0]
        valid = []
        for seq in itertools.product(range(V), repeat=K):
            p, ok = prev, True
            for i, t in enumerate(seq):
                logits = B[i] + W2 @ W1[p]
                if int(np.argmax(logits)) != t:
                    ok = False
                    break
                p = t
            if ok:
                valid.append(seq)
        assert len(valid) == 1
        res = oracle.walk(WalkBits(base), WalkBits(w1), np.array([prev], np.int32), K,
                          w2_bits=WalkBits(w2))
        assert tuple(res.tokens[0]) == valid[0]


def WalkBits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- ties and NaN

def test_argmax_rules_golden(oracle):
    spec = json.load(open(os.path.join(GOLDEN, "argmax_rules.json")))
    V, R = 6, 4
    w1 = np.zeros((V, R), np.uint16)
    w2 = np.zeros((V, R), np.uint16)
    for c in spec["cases"]:
        base = bf16_bits(c["base"]).reshape(1, 1, V)
        res = oracle.walk(base, w1, np.array([0], np.int32), 1, w2_bits=w2, want_scores=True)
        assert res.tokens[0, 0] == c["token"], c
        # torch.argmax on the same scores agrees
        assert int(torch.argmax(torch.from_numpy(res.scores[0, 0]))) == c["token"], c


def test_identical_rows_tie_by_index(oracle):
    rng = np.random.default_rng(8)
    V, R = 64, 32
    w2 = torch.randn(V, R, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    w1 = torch.randn(V, R, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    w2[41] = w2[17]
    base = torch.full((1, 1, V), -30.0).to(torch.bfloat16)
    base[0, 0, 17] = base[0, 0, 41] = 20.0
    for int8 in (False, True):
        kw = {}
        if int8:
            st, q, sc = oracle.quantize_w2(WalkBits(w2))
            kw = dict(w2q=q, scales=sc)
        else:
            kw = dict(w2_bits=WalkBits(w2))
        res = oracle.walk(WalkBits(base), WalkBits(w1), np.array([3], np.int32), 1, **kw)
        assert res.tokens[0, 0] == 17 and res.gap[0, 0] == 0.0


# ---------------------------------------------------------------- Gumbel-max sampling

def _chi2(counts, probs):
    exp = probs * counts.sum()
    return float(((counts - exp) ** 2 / exp).sum())


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_gumbel_sampler_matches_softmax(oracle, T):
    """Over many seeds the sampled token follows softmax(bf16(l) / T) (Gumbel-max theorem)."""
    V, R, N = 5, 4, 20000
    l = np.array([0.5, 1.0, -0.25, 2.0, 0.0])          # exact in bf16
    base = np.broadcast_to(_int_bf16(l), (N, 1, V)).copy()
    res = oracle.walk(base, np.zeros((V, R), np.uint16), np.zeros(N, np.int32), 1,
                      w2_bits=np.zeros((V, R), np.uint16), seeds=np.arange(N, dtype=np.uint64),
                      slot=np.zeros(N, np.int32), mode=oracle.PROBABILISTIC, temperature=T)
    counts = np.bincount(res.tokens[:, 0], minlength=V)
    p = np.exp(l / T) / np.exp(l / T).sum()
    assert _chi2(counts, p) < 25.0  # 4 dof, p ~ 5e-5


def test_gumbel_path_probability(oracle):
    """Two-step paths are drawn with probability softmax(l0)[t0] * softmax(l1(t0))[t1]."""
    V, R, N = 3, 2, 30000
    w1 = np.array([[1, 0], [0, 1], [1, 1]], float)
    w2 = np.array([[0.5, -0.5], [-1.0, 0.25], [0.0, 1.0]])
    base = np.array([[0.0, 0.5, -0.5], [0.25, 0.0, 0.5]])
    prev = 2
    bias = lambda p: w2 @ w1[p]
    sm = lambda x: np.exp(x) / np.exp(x).sum()
    probs = np.zeros((V, V))
    p0 = sm(base[0] + bias(prev))
    for t0 in range(V):
        probs[t0] = p0[t0] * sm(base[1] + bias(t0))
    res = oracle.walk(np.broadcast_to(_int_bf16(base), (N, 2, V)).copy(), _int_bf16(w1),
                      np.full(N, prev, np.int32), 2, w2_bits=_int_bf16(w2),
                      seeds=np.arange(N, dtype=np.uint64) + 1000, mode=oracle.PROBABILISTIC)
    idx = res.tokens[:, 0] * V + res.tokens[:, 1]
    counts = np.bincount(idx, minlength=V * V)
    assert _chi2(counts, probs.reshape(-1)) < 35.0  # 8 dof


# ---------------------------------------------------------------- top-k

def test_topk_matches_torch_topk(oracle):
    rng = np.random.default_rng(9)
    x = (torch.randn(6, 3000, generator=torch.Generator().manual_seed(3)) * 3).to(torch.bfloat16)
    for k in (1, 17, 512):
        cand = oracle.topk_select(WalkBits(x), k)
        for r in range(x.shape[0]):
            xf = x[r].float()
            thr = float(torch.topk(xf, k).values[-1])
            above = torch.nonzero(xf > thr).flatten().tolist()
            at = torch.nonzero(xf == thr).flatten().tolist()
            exp = sorted(above + at[: k - len(above)])
            assert cand[r].tolist() == exp


def test_topk_nan_and_boundary_ties(oracle):
    row = bf16_bits([1, "nan", 5, 5, 5, 2, "nan", 5])[None, :]
    np.testing.assert_array_equal(oracle.topk_select(row, 3), [[1, 2, 6]])
    np.testing.assert_array_equal(oracle.topk_select(row, 4), [[1, 2, 3, 6]])
    row = bf16_bits([0, "-0", 0, -1])[None, :]
    np.testing.assert_array_equal(oracle.topk_select(row, 2), [[0, 1]])


def test_topk_full_vocab_equals_dense(oracle):
    V, R, K, bs = 300, 16, 4, 3
    w1 = torch.randn(V, R, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    w2 = (torch.randn(V, R, generator=torch.Generator().manual_seed(2)) / 4).to(torch.bfloat16)
    base = (torch.randn(bs, K, V, generator=torch.Generator().manual_seed(3)) * 3).to(torch.bfloat16)
    kw = dict(w2_bits=WalkBits(w2), seeds=np.arange(bs, dtype=np.uint64),
              mode=oracle.PROBABILISTIC, temperature=0.8, want_scores=True)
    prev = np.array([1, 2, 3], np.int32)
    dense = oracle.walk(WalkBits(base), WalkBits(w1), prev, K, **kw)
    full = oracle.walk(WalkBits(base), WalkBits(w1), prev, K, top_k=V, **kw)
    np.testing.assert_array_equal(dense.tokens, full.tokens)
    np.testing.assert_array_equal(dense.scores, full.scores)
    part = oracle.walk(WalkBits(base), WalkBits(w1), prev, K, top_k=7, want_logits=True,
                       want_cand=True, **kw)
    for r in range(bs):
        for i in range(K):
            mask = np.zeros(V, bool)
            mask[part.cand[r, i]] = True
            assert np.all(np.isneginf(part.logits[r, i][~mask]))
            assert np.all(np.isfinite(part.logits[r, i][mask]))
            assert mask[part.tokens[r, i]]


def test_topk_full_vocab_equals_dense_int8(oracle):
    """int8 W2 in the top-k walk: the candidates' bias is the dense int8 walk's, so
    k = V reproduces the dense int8 walk and every other k scores only candidates."""
    V, R, K, bs = 300, 16, 4, 3
    g = torch.Generator().manual_seed(4)
    w1 = torch.randn(V, R, generator=g).to(torch.bfloat16)
    q = torch.randint(-127, 128, (V, R), generator=g, dtype=torch.int64).to(torch.int8).numpy()
    sc = (torch.rand(V, generator=g) / 64).numpy().astype(np.float32)
    base = (torch.randn(bs, K, V, generator=g) * 3).to(torch.bfloat16)
    prev = np.array([4, 5, 6], np.int32)
    for mode in (oracle.GREEDY, oracle.PROBABILISTIC):
        kw = dict(w2q=q, scales=sc, seeds=np.arange(bs, dtype=np.uint64), mode=mode,
                  temperature=0.9, want_logits=True)
        dense = oracle.walk(WalkBits(base), WalkBits(w1), prev, K, **kw)
        full = oracle.walk(WalkBits(base), WalkBits(w1), prev, K, top_k=V, **kw)
        assert dense.status == 0 and full.status == 0
        np.testing.assert_array_equal(dense.tokens, full.tokens)
        np.testing.assert_array_equal(dense.logits, full.logits)
        part = oracle.walk(WalkBits(base), WalkBits(w1), prev, K, top_k=5, want_cand=True, **kw)
        for r in range(bs):
            for i in range(K):
                mask = np.zeros(V, bool)
                mask[part.cand[r, i]] = True
                assert np.all(np.isneginf(part.logits[r, i][~mask])) and mask[part.tokens[r, i]]


# ---------------------------------------------------------------- errors and follow classes

def test_bad_token_and_invalid_args(oracle):
    V, R = 10, 4
    z = np.zeros((V, R), np.uint16)
    res = oracle.walk(np.zeros((2, 3, V), np.uint16), z, np.array([1, 10], np.int32), 3, w2_bits=z)
    assert res.status == 6 and list(res.tokens[1]) == [-1, -1, -1] and res.tokens[0, 0] == 0
    res = oracle.walk(np.zeros((1, 1, V), np.uint16), z, np.array([1], np.int32), 1, w2_bits=z,
                      mode=oracle.PROBABILISTIC, seeds=np.zeros(1, np.uint64), temperature=0.0)
    assert res.status == 1


def test_follow_classification(oracle):
    V, R = 6, 4
    z = np.zeros((V, R), np.uint16)
    base = bf16_bits([1.0, 3.0, 2.9990234375, -1, 0, 3.0]).reshape(1, 1, V)
    res = oracle.walk(base, z, np.array([0], np.int32), 1, w2_bits=z, follow=np.array([[5]]))
    assert res.tokens[0, 0] == 1 and res.follow_class[0, 0] == oracle.CLASS_NEAR_TIE
    res = oracle.walk(base, z, np.array([0], np.int32), 1, w2_bits=z, follow=np.array([[0]]))
    assert res.follow_class[0, 0] == oracle.CLASS_REJECTED


# The bf16-boundary class: in probabilistic mode a GPU token that differs from the
# oracle's is accepted when one logit lies within bf16_eps (1e-4, in logit units) of a
# bf16 rounding midpoint and rounding it the other way makes the GPU token come within
# tie_tol of the best score. The cases below are built exactly: V = 6, R = 4, the
# embedding W1[0] = e_0, so the bias of entry v is its W2 entry x_v and the fp64 logit
# is base_v + x_v (bf16 values summed exactly in fp64; x_v = a_v + b_v over two
# embedding components where x_v itself needs more than 8 significant bits). The Gumbel noise g comes
# from the separately pinned Philox generator. T = 0.5 makes logit units and score
# units differ by a factor of 2, so a window applied in score units fails case A.
_BF16_MID = 4.015625          # midpoint between the bf16 values 4.0 and 4.03125
_STEP = 2.0 ** -14            # bf16 spacing of the W2 entries near 2^-6


def _boundary_row(oracle, follow_logit_x, tok_logit, tok_x=0.0, follow_base=4.0, seed=None):
    """Walk one probabilistic step over V = 6 and return (oracle token, follow class) of
    the follow token 0, for the first seed whose noise admits the construction."""
    V, R, T = 6, 4, 0.5
    w1 = np.zeros((V, R), np.uint16)
    w1[0] = bf16_bits([1.0, 1.0, 0, 0])
    seeds = [seed] if seed is not None else range(200)
    for sd in seeds:
        _, _, g = oracle.gumbel_block(np.array([sd], np.uint64), 1, V)
        g = g[0, 0]
        base = np.full(V, -30.0)
        base[0] = follow_base
        b1 = tok_logit(g)  # the oracle's token (entry 1): a bf16 base value, or None
        if b1 is None:
            continue
        base[1] = b1
        xa, xb = np.zeros(V), np.zeros(V)  # x_v = xa_v + xb_v, each bf16-exact
        xa[0], xb[0] = follow_logit_x if isinstance(follow_logit_x, tuple) else (follow_logit_x, 0.0)
        xa[1], xb[1] = tok_x if isinstance(tok_x, tuple) else (tok_x, 0.0)
        w2 = np.zeros((V, R), np.uint16)
        w2[:, 0] = bf16_bits(xa)
        w2[:, 1] = bf16_bits(xb)
        assert np.array_equal(bf16_bits(xa).view(np.int16), torch.tensor(xa, dtype=torch.float64)
                              .to(torch.bfloat16).view(torch.int16).numpy()), "bias parts must be bf16-exact"
        res = oracle.walk(bf16_bits(base).reshape(1, 1, V), w1, np.array([0], np.int32), 1, w2_bits=w2,
                          seeds=np.array([sd], np.uint64), mode=oracle.PROBABILISTIC, temperature=T,
                          follow=np.array([[0]], np.int32), want_logits=True, want_scores=True)
        return sd, res
    raise AssertionError("no seed admits the construction")


def _tok_for_up_case(g):
    """bf16 base logit b1 of entry 1 with 2 b1 + g_1 between the follow token's score under
    round-to-nearest (2 * 4.0 + g_0) and under the upward rounding (2 * 4.03125 + g_0),
    each with a margin beyond tie_tol = 1e-3."""
    lo, hi = 8.0 + g[0] + 0.004, 8.0625 + g[0] - 0.004
    target = 0.5 * ((lo + hi) / 2 - g[1])
    b1 = float(torch.tensor(target, dtype=torch.float32).to(torch.bfloat16).float())
    s1 = 2 * b1 + g[1]
    return b1 if lo < s1 < hi else None


def test_bf16_boundary_class_upward_rounding(oracle):
    """Case A: the follow token's logit lies 2^-14 (6.1e-5 < 1e-4) below the midpoint, so
    rounding it up gives it the best score: CLASS_BF16_BOUNDARY. Case B: 2^-13 (1.2e-4)
    below, outside the window: CLASS_REJECTED. Both with the oracle's token kept by
    round-to-nearest (no near tie)."""
    for x0, want in ((0.015625 - _STEP, oracle.CLASS_BF16_BOUNDARY),
                     (0.015625 - 2 * _STEP, oracle.CLASS_REJECTED)):
        sd, res = _boundary_row(oracle, x0, _tok_for_up_case)
        assert res.status == 0
        assert abs(res.logits[0, 0, 0] - _BF16_MID) in (_STEP, 2 * _STEP)
        assert res.tokens[0, 0] == 1, (sd, res.tokens)
        assert res.scores[0, 0, 1] - res.scores[0, 0, 0] > 1e-3  # not a near tie
        assert res.follow_class[0, 0] == want, (x0, sd, res.follow_class)


def test_bf16_boundary_class_downward_rounding(oracle):
    """Case C: the oracle's token's logit lies 2^-14 ABOVE a midpoint (rounded up by
    round-to-nearest); rounding it down instead lets the follow token (bf16-exact logit)
    come within tie_tol: CLASS_BF16_BOUNDARY. The same token 2^-13 above: rejected."""
    # entry 1's logit = 4.0 + 0.015625 + x1: bf16 4.03125 by round-to-nearest, 4.0 when
    # rounded down; entry 0 (bf16-exact base b0, no bias) scores between the two.
    for x1, want in ((_STEP, oracle.CLASS_BF16_BOUNDARY), (2 * _STEP, oracle.CLASS_REJECTED)):
        V = 6
        found = None
        for sd in range(400):
            _, _, g = oracle.gumbel_block(np.array([sd], np.uint64), 1, V)
            g = g[0, 0]
            lo, hi = 8.0 + g[1] - 1e-3 + 0.004, 8.0625 + g[1] - 1e-3 - 0.004  # s0 window
            target = 0.5 * ((lo + hi) / 2 - g[0])
            b0 = float(torch.tensor(target, dtype=torch.float32).to(torch.bfloat16).float())
            if lo < 2 * b0 + g[0] < hi:
                found = (sd, b0)
                break
        assert found is not None
        sd, b0 = found
        _, res = _boundary_row(oracle, 0.0, lambda g: 4.0, tok_x=(0.015625, x1), follow_base=b0, seed=sd)
        assert res.status == 0
        assert res.logits[0, 0, 1] - _BF16_MID == x1
        assert res.tokens[0, 0] == 1, (sd, res.tokens)
        assert res.scores[0, 0, 1] - res.scores[0, 0, 0] > 1e-3
        assert res.follow_class[0, 0] == want, (x1, sd, res.follow_class)


def _mutated_oracle(tmp_path, edits):
    """A copy of the oracle with planted mistakes (each an (old, new) source edit), built
    into tmp_path on the CPU and bound like the real one."""
    import ctypes as C
    from oracle import oracle as O
    src = open(O.SRC).read()
    for old, new in edits:
        assert old in src
        src = src.replace(old, new)
    path = tmp_path / "mutant.cpp"
    path.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
                    "-shared", str(path), "-o", str(so)], check=True)
    return O.bind(C.CDLL(str(so)))


@pytest.mark.parametrize("edits", [
    # the up / down choices of the alternative rounding swapped
    [("const double pick = up ? std::max(lb, hi) : std::min(lb, lo);",
      "const double pick = up ? std::min(lb, lo) : std::max(lb, hi);")],
    # the window applied in score units (logit units times T) instead of logit units
    [("const double lo = bf16_bits_to_double(round_to_bf16(l[v] - a->bf16_eps));",
      "const double lo = bf16_bits_to_double(round_to_bf16(l[v] - a->bf16_eps * T));"),
     ("const double hi = bf16_bits_to_double(round_to_bf16(l[v] + a->bf16_eps));",
      "const double hi = bf16_bits_to_double(round_to_bf16(l[v] + a->bf16_eps * T));")],
], ids=["up_down_swapped", "window_in_score_units"])
def test_bf16_boundary_pins_catch_planted_mistakes(oracle, tmp_path, monkeypatch, edits):
    """Each planted mistake in the bf16-boundary classification makes one of the pins
    above fail."""
    monkeypatch.setattr(oracle, "_lib", _mutated_oracle(tmp_path, edits))
    failed = 0
    for pin in (test_bf16_boundary_class_upward_rounding, test_bf16_boundary_class_downward_rounding):
        try:
            pin(oracle)
        except AssertionError:
            failed += 1
    assert failed >= 1


def test_prob_score_uses_bf16_logit(oracle):
    """The sampled score is bf16(l)/T + g: subtracting the (separately pinned) Gumbel
    noise and undoing T leaves exactly the bf16-rounded logit, not the fp64 one."""
    V, R, K, bs, T = 200, 16, 2, 2, 0.7
    w1 = torch.randn(V, R, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    w2 = (torch.randn(V, R, generator=torch.Generator().manual_seed(5)) / 4).to(torch.bfloat16)
    base = (torch.randn(bs, K, V, generator=torch.Generator().manual_seed(6)) * 3).to(torch.bfloat16)
    seeds = np.array([11, 12], np.uint64)
    res = oracle.walk(WalkBits(base), WalkBits(w1), np.array([4, 9], np.int32), K,
                      w2_bits=WalkBits(w2), seeds=seeds, mode=oracle.PROBABILISTIC,
                      temperature=T, want_scores=True, want_logits=True, want_logits_bf16=True)
    _, _, g = oracle.gumbel_block(seeds, K, V)
    lb = torch.from_numpy(res.logits_bf16.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_allclose((res.scores - g) * np.float64(np.float32(T)), lb, rtol=0, atol=1e-12)
    # and that rounding did change some logits (the inputs are not bf16-exact)
    assert np.mean(lb != res.logits) > 0.9


# ---------------------------------------------------------------- the drafter's LM head

def test_lmhead_logits_exact_on_integer_inputs(oracle):
    """Small-integer hidden states and LM-head weights: every product and sum is exact,
    so the fp64 logits equal the integer matrix product (numpy int64)."""
    g = np.random.default_rng(9)
    M, d, V = 5, 96, 301
    h = g.integers(-6, 7, size=(M, d))
    w = g.integers(-9, 10, size=(V, d))
    out = oracle.lmhead_logits(bf16_bits(h.ravel()).reshape(M, d), bf16_bits(w.ravel()).reshape(V, d))
    np.testing.assert_array_equal(out, (h.astype(np.int64) @ w.T.astype(np.int64)).astype(np.float64))


def test_lmhead_one_hot_hidden_selects_a_column(oracle):
    """A one-hot hidden state e_j gives, for every vocabulary entry, the LM head's entry
    in column j (bf16 values, exact)."""
    g = np.random.default_rng(10)
    d, V = 64, 257
    w = bf16_bits(g.normal(0, 1, V * d)).reshape(V, d)
    for j in (0, 17, 63):
        h = np.zeros((1, d), np.uint16)
        h[0, j] = bf16_bits([1.0])[0]
        out = oracle.lmhead_logits(h, w)
        col = torch.from_numpy(w[:, j].view(np.int16)).view(torch.bfloat16).double().numpy()
        np.testing.assert_array_equal(out[0], col)


def test_walk_on_fp64_base_equals_walk_on_the_same_bf16_values(oracle):
    """The walk fed unrounded fp64 base logits that happen to be bf16 values behaves like
    the walk fed those bf16 values (dense and top-k)."""
    V, R, K, bs = 120, 8, 3, 2
    g = torch.Generator().manual_seed(11)
    base = (torch.randn(bs, K, V, generator=g) * 3).to(torch.bfloat16)
    w1 = torch.randn(V, R, generator=g).to(torch.bfloat16)
    w2 = (torch.randn(V, R, generator=g) / 3).to(torch.bfloat16)
    bb = base.view(torch.int16).numpy().view(np.uint16)
    kw = dict(w2_bits=w2.view(torch.int16).numpy().view(np.uint16), seeds=np.array([3, 4], np.uint64),
              mode=oracle.PROBABILISTIC, temperature=0.8, want_logits=True)
    w1b = w1.view(torch.int16).numpy().view(np.uint16)
    for top_k in (0, 7):
        a = oracle.walk(bb, w1b, np.array([5, 9], np.int32), K, top_k=top_k, **kw)
        b = oracle.walk(None, w1b, np.array([5, 9], np.int32), K, top_k=top_k, base_f64=base.double().numpy(), **kw)
        np.testing.assert_array_equal(a.tokens, b.tokens)
        np.testing.assert_array_equal(a.logits, b.logits)
