"""Speculative-sampling verification on the GPU (dspark_verify) against the oracle and
against what the method guarantees (every emitted token follows the target)."""
from __future__ import annotations

import numpy as np
import pytest
import torch
from scipy import stats

from dspark_markov_draft_gb300 import capi, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def check_verify(O, tgt, drf, dtok, seeds, T, acc_g, out_g):
    """The GPU's accepted counts and emitted tokens against the oracle's. A different
    acceptance decision is allowed only at the boundary |u q(d) - p(d)| <= 1e-5 max(.)
    (fp32 against fp64 probabilities; the row is not compared further); a different
    sample only within the oracle's score gap 1e-3, widened for residual samples by the
    conditioning of log(p - q) (1e-5 (p + q) / |p - q| for both tokens)."""
    tb, db = _bits(tgt), _bits(drf)
    res = O.verify(tb, db, dtok.cpu().numpy(), seeds.cpu().numpy().astype(np.uint64), T, want_probs=True)
    assert res.status == 0
    acc_g = acc_g.cpu().numpy()
    out_g = out_g.cpu().numpy()
    bs, K1 = out_g.shape
    K = K1 - 1
    dt = dtok.cpu().numpy()
    boundary = 0
    for r in range(bs):
        n_o, n_g = int(res.accepted[r]), int(acc_g[r])
        assert 0 <= n_g <= K
        if n_o != n_g:
            m = min(n_o, n_g)
            u, pd, qd = res.u[r, m], res.p_d[r, m], res.q_d[r, m]
            assert abs(u * qd - pd) <= 1e-5 * max(pd, u * qd) + 1e-30, (r, m, u, pd, qd)
            boundary += 1
            continue
        n = n_o
        assert list(out_g[r, :n]) == list(dt[r, :n]) and all(out_g[r, n + 1:] == -1), r
        y_g, y_o = int(out_g[r, n]), int(res.y[r, n])
        if y_g != y_o:
            s = res.scores[r, n]
            tol = 1e-3
            if n < K:
                for v in (y_g, y_o):
                    p, q = res.p[r, n, v], res.q[r, n, v]
                    tol += 1e-5 * (p + q) / max(abs(p - q), 1e-300)
            assert s[y_o] - s[y_g] <= tol, (r, n, y_g, y_o, s[y_o] - s[y_g], tol)
    return boundary


@pytest.mark.parametrize("reuse_norms", [True, False])
@pytest.mark.parametrize("V,K,bs,T", [(5003, 4, 8, 1.0), (3001, 2, 16, 0.7), (130, 7, 5, 1.3)])
def test_verify_matches_oracle(oracle, V, K, bs, T, reuse_norms):
    """Both ways to the sample pass's normalisers (the acceptance pass's, through the
    norms scratch, or recomputed by the sample pass) match the oracle."""
    g = torch.Generator().manual_seed(V + K)
    drf = (torch.randn(bs, K, V, generator=g) * 3).to(torch.bfloat16)
    # targets near the drafts so that acceptances and rejections both occur
    tgt = (torch.cat([drf.float(), torch.randn(bs, 1, V, generator=g) * 3], 1)
           + torch.randn(bs, K + 1, V, generator=g) * 0.7).to(torch.bfloat16)
    q = torch.softmax(drf.float() / T, -1)
    dtok = torch.stack([torch.multinomial(q[:, i], 1, generator=g)[:, 0] for i in range(K)], 1).to(torch.int32)
    seeds = torch.arange(bs, dtype=torch.int64) * 7 + 3
    acc, out = capi.verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), seeds.to(DEV), T, reuse_norms=reuse_norms)
    torch.cuda.synchronize()
    check_verify(oracle, tgt, drf, dtok, seeds, T, acc, out)
    assert 0 < int(acc.sum()) < bs * K  # both outcomes exercised


def test_verify_after_the_walk(oracle):
    """The pipeline: a probabilistic walk drafts K tokens and keeps its draft_logits;
    the verifier takes them with target logits near the drafter's."""
    V, K, bs, T = 6000, 5, 6, 0.8
    inp = synth.make(V, bs, K, seed=12)
    w1, w2, base, prev, seeds = (inp.w1.to(DEV), inp.w2.to(DEV), inp.base.to(DEV), inp.prev.to(DEV),
                                 inp.seeds.to(DEV))
    tokens, lg = capi.walk(base, w1, prev, w2=w2, seeds=seeds, mode=capi.PROBABILISTIC, temperature=T,
                           want_logits=True)
    g = torch.Generator().manual_seed(5)
    tgt = torch.cat([lg.float().cpu(), torch.randn(bs, 1, V, generator=g) * 3], 1)
    tgt = (tgt + torch.randn(bs, K + 1, V, generator=g) * 0.5).to(torch.bfloat16)
    vseeds = seeds + 1000
    acc, out = capi.verify(tgt.to(DEV), lg, tokens, vseeds, T)
    torch.cuda.synchronize()
    check_verify(oracle, tgt, lg.cpu(), tokens.cpu(), vseeds.cpu(), T, acc, out)


@pytest.mark.parametrize("K,T", [(1, 1.0), (2, 0.7)])
def test_emitted_tokens_follow_the_target(K, T):
    """Whatever q, the first emitted token is distributed by p_0, and the second (when
    the first draft was accepted) by p_1: chi-square over 64 rows x 160 launches."""
    V, bs, launches = 6, 64, 160
    g = torch.Generator().manual_seed(40 + K)
    tgt1 = (torch.randn(1, K + 1, V, generator=g) * 1.5).to(torch.bfloat16)
    drf1 = (torch.randn(1, K, V, generator=g) * 1.5).to(torch.bfloat16)
    p = torch.softmax(tgt1.double() / T, -1)[0].numpy()
    q = torch.softmax(drf1.float() / T, -1)[0]
    tgt = tgt1.expand(bs, K + 1, V).contiguous().to(DEV)
    drf = drf1.expand(bs, K, V).contiguous().to(DEV)
    outs, accs = [], []
    for l in range(launches):
        dtok = torch.stack([torch.multinomial(q[i], bs, replacement=True, generator=g) for i in range(K)], 1)
        seeds = torch.arange(bs, dtype=torch.int64, device=DEV) + bs * l + 100000 * K
        acc, out = capi.verify(tgt, drf, dtok.to(torch.int32).to(DEV), seeds, T)
        outs.append(out)
        accs.append(acc)
    out = torch.cat(outs).cpu().numpy()
    acc = torch.cat(accs).cpu().numpy()
    for j in range(K + 1):
        have = acc >= j
        if have.sum() < 500:
            continue
        counts = np.bincount(out[have, j], minlength=V)
        assert stats.chisquare(counts, p[j] * counts.sum()).pvalue > 1e-4, (j, counts)


def test_verify_special_cases():
    V, K, bs = 100, 3, 3
    g = torch.Generator().manual_seed(9)
    tgt = (torch.randn(bs, K + 1, V, generator=g) * 2).to(torch.bfloat16)
    drf = tgt[:, :K].clone()  # q == p: every draft accepted, then the bonus
    dtok = torch.tensor([[1, 2, 3], [4, 5, 6], [7, 8, V + 5]], dtype=torch.int32)  # last: out of range
    seeds = torch.tensor([1, 2, 3], dtype=torch.int64)
    acc, out = capi.verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), seeds.to(DEV), 1.0)
    torch.cuda.synchronize()
    acc, out = acc.cpu().tolist(), out.cpu().numpy()
    assert acc == [3, 3, 2]
    assert list(out[0, :3]) == [1, 2, 3] and 0 <= out[0, 3] < V
    assert list(out[2, :2]) == [7, 8] and 0 <= out[2, 2] < V and out[2, 3] == -1


def test_verify_captured_in_cuda_graph():
    """The verifier captured in a CUDA graph (the sample pass a programmatic dependent of
    the acceptance pass) and replayed equals an eager call on the same buffers."""
    V, K, bs, T = 4001, 4, 8, 1.0
    g0 = torch.Generator().manual_seed(5)
    drf = (torch.randn(bs, K, V, generator=g0) * 3).to(torch.bfloat16)
    tgt = (torch.cat([drf.float(), torch.randn(bs, 1, V, generator=g0) * 3], 1)
           + torch.randn(bs, K + 1, V, generator=g0) * 0.7).to(torch.bfloat16)
    dtok = torch.randint(0, V, (bs, K), generator=g0, dtype=torch.int32)
    seeds = torch.arange(bs, dtype=torch.int64) * 11 + 1
    tgt, drf, dtok, seeds = tgt.to(DEV), drf.to(DEV), dtok.to(DEV), seeds.to(DEV)
    acc = torch.empty(bs, dtype=torch.int32, device=DEV)
    out = torch.empty((bs, K + 1), dtype=torch.int32, device=DEV)
    capi.verify(tgt, drf, dtok, seeds, T, accepted=acc, out_tokens=out)  # eager first
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        capi.verify(tgt, drf, dtok, seeds, T, accepted=acc, out_tokens=out,
                    stream=torch.cuda.current_stream())
    for step in range(2):
        out.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        ra, ro = capi.verify(tgt, drf, dtok, seeds, T)
        torch.cuda.synchronize()
        assert torch.equal(acc, ra) and torch.equal(out, ro), step
