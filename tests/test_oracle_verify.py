"""Pins of the oracle's speculative-sampling verification against what the method
guarantees, independently of the implementation:

* unbiasedness (Leviathan et al. 2023, Theorem 1 / Chen et al. 2023): whatever the
  draft distribution q, every emitted token is distributed by the target distribution
  of its position -- checked by chi-square on many seeded trials at a small vocabulary;
* the acceptance probability of a draft token drawn from q is sum_v min(p_v, q_v);
* special cases: q == p accepts every draft; a draft token the target gives zero
  probability is always rejected; one with q = 0 and p > 0 always accepted.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch
from scipy import stats

from oracle import oracle as O


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def _probs(bits_row: np.ndarray, T: float) -> np.ndarray:
    x = torch.from_numpy(bits_row.view(np.int16)).view(torch.bfloat16).double().numpy() / T
    e = np.exp(x - x.max())
    return e / e.sum()


def _trials(K, V, n, T, seed):
    """n independent trials sharing one set of target / draft logits: the draft tokens
    are drawn from q with numpy's generator, the verifier's randomness from its seeds."""
    g = torch.Generator().manual_seed(seed)
    tgt = torch.randn(1, K + 1, V, generator=g) * 1.5
    drf = torch.randn(1, K, V, generator=g) * 1.5
    tb, db = _bits(tgt), _bits(drf)
    q = np.stack([_probs(db[0, i], T) for i in range(K)])
    p = np.stack([_probs(tb[0, i], T) for i in range(K + 1)])
    rng = np.random.default_rng(seed)
    dtok = np.stack([rng.choice(V, size=n, p=q[i]) for i in range(K)], axis=1).astype(np.int32)
    res = O.verify(np.repeat(tb, n, 0), np.repeat(db, n, 0), dtok,
                   np.arange(n, dtype=np.uint64) + 1000 * seed, T)
    assert res.status == 0
    return p, q, dtok, res


@pytest.mark.parametrize("K,T", [(1, 1.0), (3, 0.7)])
def test_emitted_tokens_follow_the_target(oracle, K, T):
    V, n = 6, 20000
    p, q, dtok, res = _trials(K, V, n, T, seed=K)
    for j in range(K + 1):
        have = res.accepted >= j  # token j is emitted iff the first j drafts were accepted
        if have.sum() < 500:
            continue
        counts = np.bincount(res.out_tokens[have, j], minlength=V)
        chi = stats.chisquare(counts, p[j] * counts.sum())
        assert chi.pvalue > 1e-4, (j, counts, p[j] * counts.sum())
    # and the drafts alone are not: q differs from p, so emitting d unchecked would fail
    counts = np.bincount(dtok[:, 0], minlength=V)
    assert stats.chisquare(counts, p[0] * n).pvalue < 1e-6


def test_acceptance_rate_is_sum_of_minima(oracle):
    V, n, T = 6, 20000, 1.0
    p, q, dtok, res = _trials(1, V, n, T, seed=7)
    rate = np.mean(res.accepted >= 1)
    expect = np.minimum(p[0], q[0]).sum()
    assert abs(rate - expect) < 4 * np.sqrt(expect * (1 - expect) / n), (rate, expect)


def test_special_cases(oracle):
    V, K, T = 5, 2, 1.0
    g = torch.Generator().manual_seed(3)
    logits = torch.randn(1, K + 1, V, generator=g)
    tb = _bits(logits)
    # q == p: every draft accepted, then the bonus
    db = tb[:, :K].copy()
    dtok = np.array([[1, 3]], np.int32)
    res = O.verify(tb, db, dtok, np.array([5], np.uint64), T)
    assert res.accepted[0] == K and list(res.out_tokens[0, :K]) == [1, 3]
    # target -inf at the draft token: rejected at once, the sample is not that token
    tz = tb.copy()
    tz[0, 0, 1] = 0xFF80
    res = O.verify(tz, db, dtok, np.array([5], np.uint64), T)
    assert res.accepted[0] == 0 and res.out_tokens[0, 0] != 1 and list(res.out_tokens[0, 1:]) == [-1, -1]
    # draft -inf (q = 0) at a token the target allows: accepted
    dz = db.copy()
    dz[0, 0, 1] = 0xFF80
    res = O.verify(tb, dz, dtok, np.array([5], np.uint64), T)
    assert res.accepted[0] >= 1 and res.out_tokens[0, 0] == 1


def test_random_draws_follow_the_documented_counters(oracle):
    """The verifier's randomness, recomputed from the Philox core (itself pinned against
    an independent implementation) and the documented layout: u_i from counter
    (0, i, b, 1), word 0; the sample noise of position n from counter (v >> 2, n, b, 2),
    word v & 3, g = -log(-log u). The bonus scores are target / T + g, the residual
    scores log(p - q) + g where p > q; the probabilities are softmax(row / T)."""
    bs, K, V, T = 3, 2, 37, 0.8
    g = torch.Generator().manual_seed(11)
    tgt = torch.randn(bs, K + 1, V, generator=g) * 2
    drf = torch.randn(bs, K, V, generator=g) * 2
    tb, db = _bits(tgt), _bits(drf)
    dtok = np.array([[1, 5], [36, 0], [7, 7]], np.int32)
    seeds = np.array([5, 2**40 + 3, 2**64 - 7], np.uint64)
    res = O.verify(tb, db, dtok, seeds, T, want_probs=True)
    assert res.status == 0
    T = float(np.float32(T))  # the temperature is an fp32 argument

    def u_of(w):
        return (2.0 * (int(w) >> 9) + 1.0) * 2.0**-24

    for r in range(bs):
        key = [int(seeds[r]) & 0xFFFFFFFF, int(seeds[r]) >> 32]
        for i in range(K):
            w = O.philox4x32_10([0, i, r, 1], key)[0]
            assert res.u[r, i] == u_of(w)
        for n in range(K + 1):
            p = _probs(tb[r, n], T)
            np.testing.assert_allclose(res.p[r, n], p, rtol=1e-12, atol=1e-300)
            x = torch.from_numpy(tb[r, n].view(np.int16)).view(torch.bfloat16).double().numpy()
            noise = np.array([-np.log(-np.log(u_of(O.philox4x32_10([v >> 2, n, r, 2], key)[v & 3])))
                              for v in range(V)])
            if n == K:
                want = x / T + noise
            else:
                rv = p - _probs(db[r, n], T)
                want = np.where(rv > 0, np.log(np.where(rv > 0, rv, 1.0)) + noise, -np.inf)
            np.testing.assert_allclose(res.scores[r, n], want, rtol=1e-9, atol=1e-9)
            assert res.y[r, n] == int(np.argmax(want))
