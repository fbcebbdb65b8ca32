"""The drafter's LM head fused with the top-k selection (dspark_lmhead_topk) against the
CPU oracle, and the top-k walk fed its candidates.

Candidate sets must equal the oracle's top-k of the fp64 LM-head logits (order: NaN
first, larger value, smaller index), except that at the k-th value entries whose oracle
logits lie within the fp32-versus-fp64 rounding window of it may be exchanged; their
fp32 logits must match the oracle's within that window. Integer-valued inputs make the
fp32 logits exact, so ties at the k-th value must resolve to the smaller indices exactly.
"""
import numpy as np
import pytest
import torch

from dspark_markov_draft_gb300 import capi, synth

from parity import bits, check_walk_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
VAL_TOL = 2e-4  # |fp32 tensor-core logit - fp64 oracle logit| (d <= 2048, logits ~ N(0, 9))


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dspark_markov_draft_gb300 import build
    build.build()
    capi.lib()


def topk_ref(row: np.ndarray, k: int) -> np.ndarray:
    """Oracle order on an fp64 row: NaN first (by index), larger value, smaller index."""
    idx = np.arange(row.size)
    key = np.where(np.isnan(row), np.inf, row)
    order = np.lexsort((idx, -key, ~np.isnan(row)))
    return order[:k]


def check_sets(ref_logits: np.ndarray, cand: np.ndarray, cand_base: np.ndarray, k: int, tol: float):
    for m in range(ref_logits.shape[0]):
        row = ref_logits[m]
        want = topk_ref(row, k)
        got = cand[m]
        assert len(set(got.tolist())) == k, "duplicate candidates"
        assert np.all((got >= 0) & (got < row.size))
        kth = row[want[-1]]
        diff = set(got.tolist()) ^ set(want.tolist())
        for v in diff:  # only exchanges at the k-th value, within the rounding window
            assert abs(row[v] - kth) <= tol, (m, v, row[v], kth)
        np.testing.assert_allclose(cand_base[m], row[got], rtol=0, atol=tol)


@pytest.mark.parametrize("M,d,V,k", [(6, 128, 3001, 1), (6, 128, 3001, 17), (6, 128, 3001, 300),
                                     (300, 64, 2000, 40), (600, 64, 2000, 40), (5, 2048, 5000, 700)])
@pytest.mark.parametrize("exact", [False, True])
def test_lmhead_topk_matches_oracle(oracle, M, d, V, k, exact):
    hidden, head = synth.lmhead(M, d, V, seed=M + V + k)
    stats = torch.zeros(2, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cand, cbase = capi.lmhead_topk(hidden.to(DEV), head.to(DEV), k, stats=stats, status=status, exact=exact)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.lmhead_logits(bits(hidden), bits(head), nthreads=16)
    check_sets(ref, cand.cpu().numpy(), cbase.cpu().double().numpy(), k, VAL_TOL)
    if exact:
        assert int(stats[0]) == M
    else:
        assert int(stats[0]) == 0 and int(stats[1]) == 0  # every row served by its pivot


def test_lmhead_ties_resolve_to_smaller_indices(oracle):
    """Integer inputs: exact fp32 logits with many equal values; the k-th value is shared
    by more entries than fit, and the smallest indices must be taken (fast and exact
    paths alike)."""
    g = np.random.default_rng(5)
    M, d, V, k = 4, 64, 4096, 100
    h = torch.from_numpy(g.integers(-1, 2, size=(M, d)).astype(np.float32)).bfloat16()
    w = torch.from_numpy(g.integers(-1, 2, size=(V, d)).astype(np.float32)).bfloat16()
    ref = oracle.lmhead_logits(bits(h), bits(w))
    for exact in (False, True):
        cand, cbase = capi.lmhead_topk(h.to(DEV), w.to(DEV), k, exact=exact)
        torch.cuda.synchronize()
        for m in range(M):
            want = set(topk_ref(ref[m], k).tolist())
            assert set(cand[m].cpu().tolist()) == want
            np.testing.assert_array_equal(cbase[m].cpu().double().numpy(), ref[m][cand[m].cpu().numpy()])


@pytest.mark.parametrize("M,d,V,k", [(1, 64, 50, 10), (2, 64, 1000, 1000), (513, 64, 300, 5), (7, 192, 129, 128)])
def test_lmhead_edge_shapes(oracle, M, d, V, k):
    """A single hidden row and a vocabulary smaller than one 128-row tile; k = V (every
    entry is a candidate); 513 hidden rows (a second 512-row chunk of one row); a
    vocabulary one row past a tile with k one below it. Sets and values as above."""
    hidden, head = synth.lmhead(M, d, V, seed=M + d + V + k)
    cand, cbase = capi.lmhead_topk(hidden.to(DEV), head.to(DEV), k)
    torch.cuda.synchronize()
    ref = oracle.lmhead_logits(bits(hidden), bits(head), nthreads=16)
    check_sets(ref, cand.cpu().numpy(), cbase.cpu().double().numpy(), k, VAL_TOL)
    if k == V:
        for m in range(M):
            assert sorted(cand[m].cpu().tolist()) == list(range(V))


def test_lmhead_all_equal_logits_overflow_to_the_exact_path(oracle):
    """Zero hidden states: every logit is 0, every entry reaches the pivot, each row's
    list overflows (V > 3k + 1024) and the exact path must return the k smallest indices
    with value 0 (equal values in index order)."""
    M, d, V, k = 3, 128, 5000, 100
    hidden = torch.zeros((M, d), dtype=torch.bfloat16)
    _, head = synth.lmhead(M, d, V, seed=11)
    stats = torch.zeros(2, dtype=torch.int32, device=DEV)
    cand, cbase = capi.lmhead_topk(hidden.to(DEV), head.to(DEV), k, stats=stats)
    torch.cuda.synchronize()
    assert int(stats[0]) == M and int(stats[1]) == M  # every row: exact path, by overflow
    ref = oracle.lmhead_logits(bits(hidden), bits(head))
    assert np.all(ref == 0.0)
    for m in range(M):
        assert sorted(cand[m].cpu().tolist()) == list(range(k))
    assert np.all(cbase.cpu().numpy() == 0.0)


def test_lmhead_nan_row_takes_the_smallest_indices(oracle):
    """A NaN in one hidden row makes all its logits NaN: NaN counts as the largest value,
    so its candidates are the k smallest indices, with NaN logits; the other rows are
    unaffected."""
    M, d, V, k = 4, 128, 3001, 64
    hidden, head = synth.lmhead(M, d, V, seed=12)
    hidden[2, 5] = float("nan")
    cand, cbase = capi.lmhead_topk(hidden.to(DEV), head.to(DEV), k)
    torch.cuda.synchronize()
    ref = oracle.lmhead_logits(bits(hidden), bits(head))
    assert np.all(np.isnan(ref[2]))
    assert sorted(cand[2].cpu().tolist()) == list(range(k))
    assert np.all(np.isnan(cbase[2].cpu().numpy()))
    rows = [0, 1, 3]
    check_sets(ref[rows], cand.cpu().numpy()[rows], cbase.cpu().double().numpy()[rows], k, VAL_TOL)


@pytest.mark.parametrize("mode,T", [(capi.GREEDY, 1.0), (capi.PROBABILISTIC, 1.0), (capi.PROBABILISTIC, 0.7)])
def test_walk_on_fused_candidates(oracle, mode, T):
    """LM head -> top-k candidates -> the top-k walk on them (no dense base logits):
    tokens and draft_logits against the oracle walk on the fp64 LM-head logits."""
    V, K, bs, d, k = 3001, 3, 4, 128, 50
    inp = synth.make(V, bs, K, seed=77)
    hidden, head = synth.lmhead(bs * K, d, V, seed=78)
    cand, cbase = capi.lmhead_topk(hidden.to(DEV), head.to(DEV), k)
    w1, w2, prev, seeds = inp.w1.to(DEV), inp.w2.to(DEV), inp.prev.to(DEV), inp.seeds.to(DEV)
    tokens, lg = capi.walk(None, w1, prev, w2=w2, seeds=seeds, mode=mode, temperature=T, top_k=k,
                           topk_cand=cand.view(bs, K, k), topk_base=cbase.view(bs, K, k), V=V, want_logits=True)
    torch.cuda.synchronize()
    base64 = oracle.lmhead_logits(bits(hidden), bits(head), nthreads=16).reshape(bs, K, V)
    check_walk_rows(oracle, inp, tokens, label=f"lmhead top-k {k} small", mode=mode, T=T, top_k=k,
                    gpu_logits=lg, base_f64_all=base64)


@pytest.mark.parametrize("d,k,K", [(2048, 512, 7), (2048, 4096, 7), (4096, 512, 7), (2048, 512, 16)])
def test_full_size_lmhead_topk_walk(oracle, d, k, K):
    """d in {2048, 4096}, V = 151936, bs = 64, K = 7 (448 hidden rows) or K = 16 (1024
    hidden rows: two 512-row chunks per LM-head tile): the fused selection served by the
    pivot on every row; candidate sets, values and the walk's tokens checked on sampled
    request rows (all their positions) against the oracle."""
    V, bs = 151936, 64
    inp = synth.make(V, bs, K, seed=0)
    hidden, head = synth.lmhead(bs * K, d, V, seed=1)
    stats = torch.zeros(2, dtype=torch.int32, device=DEV)
    cand, cbase = capi.lmhead_topk(hidden.to(DEV), head.to(DEV), k, stats=stats)
    w1, w2, prev, seeds = inp.w1.to(DEV), inp.w2.to(DEV), inp.prev.to(DEV), inp.seeds.to(DEV)
    tokens, lg = capi.walk(None, w1, prev, w2=w2, seeds=seeds, mode=capi.PROBABILISTIC, top_k=k,
                           topk_cand=cand.view(bs, K, k), topk_base=cbase.view(bs, K, k), V=V)
    torch.cuda.synchronize()
    assert int(stats[0]) == 0 and int(stats[1]) == 0
    rows_b = [0, 37, 63]
    hrows = [b * K + i for b in rows_b for i in range(K)]
    ref = oracle.lmhead_logits(bits(hidden)[hrows], bits(head), nthreads=16)
    check_sets(ref, cand.cpu().numpy()[hrows], cbase.cpu().double().numpy()[hrows], k, VAL_TOL)
    base64 = np.zeros((bs, K, V))
    base64[rows_b] = ref.reshape(len(rows_b), K, V)
    check_walk_rows(oracle, inp, tokens, label=f"V=151936 K={K} bs=64 lmhead d={d} top-k {k} (rows {rows_b})",
                    mode=capi.PROBABILISTIC, top_k=k, base_f64_all=base64, rows_subset=rows_b)


def test_lmhead_topk_captured_in_cuda_graph():
    """The fused LM head captured in a CUDA graph (its passes chained as programmatic
    dependents) and replayed: every replay gives the candidate sets and logits of an eager
    call on the hidden rows the graph's buffer holds at replay time."""
    M, d, V, k = 40, 256, 7000, 64
    g0 = torch.Generator().manual_seed(77)
    hidden = torch.randn(M, d, generator=g0).to(torch.bfloat16).to(DEV)
    head = (torch.randn(V, d, generator=g0) * (3.0 / d ** 0.5)).to(torch.bfloat16).to(DEV)
    cand = torch.empty((M, k), dtype=torch.int32, device=DEV)
    cbase = torch.empty((M, k), dtype=torch.float32, device=DEV)
    ws = capi.lmhead_workspace(M, V, k, device=DEV)
    capi.lmhead_topk(hidden, head, k, cand=cand, cand_base=cbase, workspace=ws)  # eager first
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        capi.lmhead_topk(hidden, head, k, cand=cand, cand_base=cbase, workspace=ws,
                         stream=torch.cuda.current_stream())
    for step in range(3):
        if step == 1:  # new hidden rows in the captured buffer
            hidden.copy_(torch.randn(M, d, generator=g0).to(torch.bfloat16).to(DEV))
        cand.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        rc, rb = capi.lmhead_topk(hidden, head, k)
        torch.cuda.synchronize()
        # the same candidate sets with the same logits (a row's candidates come in any order)
        o1, o2 = torch.argsort(cand, dim=1), torch.argsort(rc, dim=1)
        assert torch.equal(torch.gather(cand, 1, o1), torch.gather(rc, 1, o2)), step
        assert torch.equal(torch.gather(cbase, 1, o1).view(torch.int32),
                           torch.gather(rb, 1, o2).view(torch.int32)), step
