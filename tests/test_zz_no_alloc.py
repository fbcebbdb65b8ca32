"""dspark_walk_noalloc against dspark_walk.

The allocation-free entry point serves callers that cannot call cudaMalloc (a plugin
enqueue hook, or a server whose device memory is all pre-reserved): its scratch is a
static device array inside the library instead of a caller-provided workspace. Here it
runs through the C ABI twice in a row on the same inputs, and each result must match the regular
entry point's within the parity tolerances (tokens identical, logits within
2e-2 + 1e-2 |x|). A call after one whose wait timed out (leaving the array dirty) must
match as well. This file is collected last so that a failure here cannot stop the rest
of the suite.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from dspark_markov_draft_gb300 import capi, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dspark_markov_draft_gb300 import build
    build.build()
    capi.lib()


@pytest.mark.parametrize("int8,mode,T,bs,K", [(True, capi.GREEDY, 1.0, 3, 5),
                                              (False, capi.PROBABILISTIC, 0.7, 2, 4)])
def test_noalloc_matches_walk_twice(int8, mode, T, bs, K):
    V = 20011
    inp = synth.make(V, bs, K, seed=41, peak=8.0)
    dev = "cuda"
    w1, w2 = inp.w1.to(dev), inp.w2.to(dev)
    base, prev, seeds = inp.base.to(dev), inp.prev.to(dev), inp.seeds.to(dev)
    kw = dict(w2=w2)
    if int8:
        q, sc = capi.quantize_w2(w2)
        kw = dict(w2q=q, scales=sc)
    ref_tok, ref_lg = capi.walk(base, w1, prev, seeds=seeds, mode=mode, temperature=T,
                                want_logits=True, **kw)
    torch.cuda.synchronize()
    unused_ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    for _ in range(2):
        tok = torch.full((bs, K), -7, dtype=torch.int32, device=dev)
        lg = torch.zeros((bs, K, V), dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        args = capi.make_args(base, w1, prev, tok, unused_ws, seeds=seeds, mode=mode,
                              temperature=T, logits=lg, status=status, **kw)
        st = capi.lib().dspark_walk_noalloc(C.byref(args), torch.cuda.current_stream().cuda_stream)
        assert st == 0, capi.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(tok, ref_tok)
        g = lg.float().cpu().double().numpy()
        r = ref_lg.float().cpu().double().numpy()
        fin = np.isfinite(r)
        assert np.array_equal(np.isfinite(g), fin)
        assert np.all(np.abs(g[fin] - r[fin]) <= 2e-2 + 1e-2 * np.abs(r[fin]))


def test_noalloc_recovers_after_a_timed_out_call():
    """A call whose grid barrier gives up (CTA 0 skips its first arrival, a 20 ms limit)
    leaves the static array dirty; the next call clears it first and must then match the
    regular entry point."""
    V, bs, K = 6007, 2, 3
    inp = synth.make(V, bs, K, seed=43)
    dev = "cuda"
    w1, w2 = inp.w1.to(dev), inp.w2.to(dev)
    base, prev = inp.base.to(dev), inp.prev.to(dev)
    ref_tok, _ = capi.walk(base, w1, prev, w2=w2)
    torch.cuda.synchronize()
    unused_ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    tok = torch.full((bs, K), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    args = capi.make_args(base, w1, prev, tok, unused_ws, w2=w2, status=status,
                          flags=capi.FLAG_SKIP_ARRIVAL_CTA0, timeout_us=20000)
    assert capi.walk_noalloc(args) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 5  # TIMEOUT
    status.zero_()
    args = capi.make_args(base, w1, prev, tok, unused_ws, w2=w2, status=status)
    assert capi.walk_noalloc(args) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(tok, ref_tok)


def test_noalloc_rejects_topk():
    fake = 1 << 20
    a = capi.WalkArgs()
    a.base_logits = a.w1 = a.w2 = a.prev_tokens = a.draft_tokens = fake
    a.V, a.rank, a.bs, a.K, a.top_k = 1000, 256, 1, 2, 5
    assert capi.lib().dspark_walk_noalloc(C.byref(a), None) == 2
