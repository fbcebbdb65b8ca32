"""GPU parity tests: the C ABI (libdspark.so) against the CPU oracle.

Small cases span several vocabulary slices per CTA, ragged tails and both the
shared-memory-resident and the streamed W2 rows; full-size cases run the benchmark
workloads and check sampled rows. All inputs are seeded and synthetic.
"""
import numpy as np
import pytest
import torch

from dspark_markov_draft_gb300 import capi, synth

from parity import bits, check_walk, check_walk_rows, nthreads, record

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dspark_markov_draft_gb300 import build
    build.build()
    capi.lib()


def to_dev(inp):
    return (inp.w1.to(DEV), inp.w2.to(DEV), inp.base.to(DEV), inp.prev.to(DEV),
            inp.seeds.to(DEV))


# ------------------------------------------------------------------ quantizer / noise

@pytest.mark.parametrize("V", [1, 7, 5000, 151936])
def test_quantize_bit_exact(oracle, V):
    w1, w2 = synth.weights(V, seed=V)
    w2[0, :] = 0
    if V > 3:
        w2[1, 5] = -w2[1].abs().max().float() * 2
        w2[2, :8] = torch.tensor([127, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5])
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, sc = capi.quantize_w2(w2.to(DEV), status=status)
    torch.cuda.synchronize()
    st, q_ref, sc_ref = oracle.quantize_w2(bits(w2))
    assert st == 0 and int(status.item()) == 0
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)


def test_quantize_nonfinite_reported():
    w = torch.zeros(4, 256, dtype=torch.bfloat16)
    w[2, 7] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    capi.quantize_w2(w.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 7


def test_philox_words_bit_exact(oracle):
    seeds = torch.tensor([0, 1, 0x123456789ABCDEF, -1], dtype=torch.int64)
    K, V = 3, 1001
    words, g = capi.gumbel_noise(seeds.to(DEV), K, V)
    torch.cuda.synchronize()
    w_ref, u_ref, g_ref = oracle.gumbel_block(seeds.numpy().astype(np.uint64), K, V)
    np.testing.assert_array_equal(words.cpu().numpy().view(np.uint32), w_ref)
    gg = g.cpu().double().numpy()
    assert np.all(np.abs(gg - g_ref) <= 4e-6 * np.maximum(1.0, np.abs(g_ref)))


# ------------------------------------------------------------------ dense walk, small

CASES = [
    # (int8, mode, T, bs, logits)
    (True, capi.GREEDY, 1.0, 1, False),
    (True, capi.GREEDY, 1.0, 3, True),
    (True, capi.PROBABILISTIC, 1.0, 3, True),
    (True, capi.PROBABILISTIC, 0.7, 16, False),
    (False, capi.GREEDY, 1.0, 1, True),
    (False, capi.GREEDY, 1.0, 16, False),
    (False, capi.PROBABILISTIC, 0.7, 3, True),
    (False, capi.PROBABILISTIC, 1.0, 1, False),
]


@pytest.mark.parametrize("int8,mode,T,bs,logits", CASES)
@pytest.mark.parametrize("cap", [-1, 0])
def test_walk_small_parity(oracle, int8, mode, T, bs, logits, cap):
    V, K = 5003, 5
    inp = synth.make(V, bs, K, seed=11 + bs, peak=8.0)
    w1, w2, base, prev, seeds = to_dev(inp)
    q = sc = q_ref = sc_ref = None
    wk = dict(w2=w2)
    if int8:
        q, sc = capi.quantize_w2(w2)
        _, q_ref, sc_ref = oracle.quantize_w2(bits(inp.w2))
        wk = dict(w2q=q, scales=sc)
    tokens, lg = capi.walk(base, w1, prev, seeds=seeds, mode=mode, temperature=T,
                           want_logits=logits, resident_rows_cap=cap, **wk)
    torch.cuda.synchronize()
    check_walk(oracle, inp, tokens, mode=mode, T=T, q=q_ref, sc=sc_ref, gpu_logits=lg)


PATH_FLAGS = {"cuda_cores": capi.FLAG_FORCE_CUDA_CORES, "tensor_cores": capi.FLAG_FORCE_TENSOR_CORES}


@pytest.mark.parametrize("path", ["cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("bs", [1, 5, 20, 40, 64])
@pytest.mark.parametrize("int8,mode,T,logits", [(True, capi.GREEDY, 1.0, True),
                                                (False, capi.PROBABILISTIC, 0.7, True),
                                                (True, capi.PROBABILISTIC, 1.0, False)])
def test_both_contraction_paths_match_oracle(oracle, path, bs, int8, mode, T, logits):
    """Each contraction path (CUDA cores, tcgen05 tensor cores with N = 16/32/64) on
    its own, for several batch sizes, against the oracle."""
    V, K = 5003, 3
    inp = synth.make(V, bs, K, seed=50 + bs, peak=8.0)
    w1, w2, base, prev, seeds = to_dev(inp)
    q_ref = sc_ref = None
    wk = dict(w2=w2)
    if int8:
        q, sc = capi.quantize_w2(w2)
        _, q_ref, sc_ref = oracle.quantize_w2(bits(inp.w2))
        wk = dict(w2q=q, scales=sc)
    rows = list(range(bs)) if bs <= 8 else [0, bs // 2, bs - 1]
    tokens, lg = capi.walk(base, w1, prev, seeds=seeds, mode=mode, temperature=T,
                           want_logits=logits, flags=PATH_FLAGS[path], **wk)
    torch.cuda.synchronize()
    check_walk(oracle, inp, tokens, mode=mode, T=T, q=q_ref, sc=sc_ref, gpu_logits=lg, rows=rows)


@pytest.mark.parametrize("int8", [True, False])
def test_resident_split_does_not_change_results(int8):
    V, K, bs = 20011, 4, 2
    inp = synth.make(V, bs, K, seed=5)
    w1, w2, base, prev, seeds = to_dev(inp)
    wk = dict(w2=w2)
    if int8:
        q, sc = capi.quantize_w2(w2)
        wk = dict(w2q=q, scales=sc)
    for flags in (capi.FLAG_FORCE_CUDA_CORES, capi.FLAG_FORCE_TENSOR_CORES):
        outs = []
        for cap in (0, 32, 64, -1):
            t, lg = capi.walk(base, w1, prev, seeds=seeds, mode=capi.PROBABILISTIC,
                              temperature=0.9, want_logits=True, resident_rows_cap=cap,
                              flags=flags, **wk)
            outs.append((t.cpu(), lg.cpu()))
        for t, lg in outs[1:]:
            assert torch.equal(t, outs[0][0])
            assert torch.equal(lg.view(torch.int16), outs[0][1].view(torch.int16))


def test_integer_inputs_bit_exact_logits(oracle):
    """Small-integer inputs make every bias exact in fp32: GPU logits equal the oracle's."""
    rng = np.random.default_rng(0)
    V, K, bs = 3001, 3, 2
    inp = synth.make(V, bs, K, seed=1)
    inp.w1 = torch.from_numpy(rng.integers(-3, 4, size=(V, 256)).astype(np.float32)).bfloat16()
    inp.w2 = torch.from_numpy(rng.integers(-4, 5, size=(V, 256)).astype(np.float32)).bfloat16()
    inp.base = torch.from_numpy(rng.integers(-30, 31, size=(bs, K, V)).astype(np.float32)).bfloat16()
    w1, w2, base, prev, seeds = to_dev(inp)
    tokens, lg = capi.walk(base, w1, prev, w2=w2, want_logits=True)
    torch.cuda.synchronize()
    res = oracle.walk(bits(inp.base), bits(inp.w1), inp.prev.numpy(), K, w2_bits=bits(inp.w2),
                      want_logits=True)
    np.testing.assert_array_equal(tokens.cpu().numpy(), res.tokens)
    np.testing.assert_array_equal(lg.cpu().float().double().numpy(),
                                  torch.from_numpy(res.logits).bfloat16().double().numpy())
    # int8 with power-of-two scales: exact as well
    q = torch.from_numpy(rng.integers(-127, 128, size=(V, 256)).astype(np.int8))
    sc = torch.from_numpy((2.0 ** rng.integers(-8, -3, size=V)).astype(np.float32))
    tokens, lg = capi.walk(base, w1, prev, w2q=q.to(DEV), scales=sc.to(DEV), want_logits=True)
    torch.cuda.synchronize()
    res = oracle.walk(bits(inp.base), bits(inp.w1), inp.prev.numpy(), K, w2q=q.numpy(),
                      scales=sc.numpy(), want_logits=True)
    np.testing.assert_array_equal(tokens.cpu().numpy(), res.tokens)
    np.testing.assert_array_equal(lg.cpu().float().double().numpy(),
                                  torch.from_numpy(res.logits).bfloat16().double().numpy())


@pytest.mark.parametrize("int8", [True, False])
def test_ties_nan_and_signed_zero(oracle, int8):
    """Hand-built ties across CTA slices, planted NaNs, all -inf rows and -0/+0."""
    V, K, bs = 9000, 1, 5
    inp = synth.make(V, bs, K, seed=3)
    inp.w2[8500] = inp.w2[40]                       # identical rows in different slices
    base = torch.full((bs, K, V), -40.0)
    base[0, 0, 40] = base[0, 0, 8500] = 30.0         # tie -> 40
    base[1, 0, 7000] = float("nan")
    base[1, 0, 100] = float("nan")                  # first NaN -> 100
    base[2] = float("-inf")                         # every logit -inf -> 0
    base[3, 0, 6000] = 0.0
    base[3, 0, 5000] = -0.0
    inp.base = base.bfloat16()
    inp.w1[inp.prev[3]] = 0                         # zero bias: -0 and +0 tie -> 5000
    inp.w1[inp.prev[0]] = 0
    inp.w1[inp.prev[0], 0] = 1.0
    w1, w2, basedev, prev, seeds = to_dev(inp)
    wk, okw = dict(w2=w2), {}
    if int8:
        q, sc = capi.quantize_w2(w2)
        _, q_ref, sc_ref = oracle.quantize_w2(bits(inp.w2))
        wk, okw = dict(w2q=q, scales=sc), dict(q=q_ref, sc=sc_ref)
    for mode in (capi.GREEDY, capi.PROBABILISTIC):
        tokens, lg = capi.walk(basedev, w1, prev, seeds=seeds, mode=mode, want_logits=True, **wk)
        torch.cuda.synchronize()
        t = tokens.cpu().numpy()[:, 0]
        if mode == capi.GREEDY:
            assert t[0] == 40 and t[1] == 100 and t[2] == 0 and t[3] == 5000, t
        else:
            assert t[1] == 100 and t[2] == 0, t
        check_walk(oracle, inp, tokens, mode=mode, gpu_logits=lg, **okw)


@pytest.mark.parametrize("bs", [2, 3])
def test_bad_token_reported(bs):
    """An out-of-range previous token: BAD_TOKEN, that row's tokens are -1, the other
    rows walk on (bs = 2: CUDA cores; bs = 3: tensor cores)."""
    V, K = 4000, 3
    inp = synth.make(V, bs, K, seed=2)
    inp.prev[1] = V
    w1, w2, base, prev, seeds = to_dev(inp)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tokens, _ = capi.walk(base, w1, prev, w2=w2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6
    t = tokens.cpu().numpy()
    live = [r for r in range(bs) if r != 1]
    assert list(t[1]) == [-1] * K and np.all(t[live] >= 0)


@pytest.mark.parametrize("bs", [1, 2, 4, 20])
def test_vocabulary_smaller_than_grid(oracle, bs):
    """V below the number of CTAs: CTAs without vocabulary rows still take part in every
    position's exchange (bs <= 2: CUDA-core walk, else tensor cores)."""
    V, K = 100, 4
    inp = synth.make(V, bs, K, seed=60 + bs, peak=8.0)
    w1, w2, base, prev, seeds = to_dev(inp)
    q, sc = capi.quantize_w2(w2)
    _, q_ref, sc_ref = oracle.quantize_w2(bits(inp.w2))
    for mode in (capi.GREEDY, capi.PROBABILISTIC):
        tokens, lg = capi.walk(base, w1, prev, seeds=seeds, mode=mode, want_logits=True, w2q=q, scales=sc)
        torch.cuda.synchronize()
        check_walk(oracle, inp, tokens, mode=mode, q=q_ref, sc=sc_ref, gpu_logits=lg)


@pytest.mark.parametrize("flags", [capi.FLAG_FORCE_CUDA_CORES, capi.FLAG_FORCE_TENSOR_CORES])
def test_small_shared_memory_plan_keeps_one_cta_per_sm(oracle, flags):
    """Both walks allocate all of tensor memory, so a second CTA on an SM would wait in
    the allocation until the first exits. With a tiny vocabulary and no resident rows the
    shared-memory request alone would allow several CTAs per SM; the launch raises it so
    that one fits, and the walk completes correctly."""
    V, K, bs = 64, 3, 2
    inp = synth.make(V, bs, K, seed=66)
    w1, w2, base, prev, seeds = to_dev(inp)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tokens, _ = capi.walk(base, w1, prev, w2=w2, resident_rows_cap=0, flags=flags,
                          status=status, timeout_us=200000)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_walk(oracle, inp, tokens, mode=capi.GREEDY)


@pytest.mark.parametrize("bs", [1, 8])
def test_timeout_returns_status_and_context_survives(bs):
    """CTA 0 skips its first arrival: every wait gives up after 20 ms and reports
    TIMEOUT; after re-zeroing the workspace the next walk is correct."""
    V, K = 4000, 3
    inp = synth.make(V, bs, K, seed=4)
    w1, w2, base, prev, seeds = to_dev(inp)
    ws = capi.alloc_workspace(V, bs, K)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    capi.walk(base, w1, prev, w2=w2, workspace=ws, status=status,
              flags=capi.FLAG_SKIP_ARRIVAL_CTA0, timeout_us=20000)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    ws.zero_()
    status.zero_()
    t1, _ = capi.walk(base, w1, prev, w2=w2, workspace=ws, status=status)
    t2, _ = capi.walk(base, w1, prev, w2=w2)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.equal(t1, t2)


@pytest.mark.parametrize("bs", [1, 2, 4, 8])
def test_workspace_left_zeroed_and_reusable(bs):
    V, K = 7000, 6
    inp = synth.make(V, bs, K, seed=8)
    w1, w2, base, prev, seeds = to_dev(inp)
    ws = capi.alloc_workspace(V, bs, K)
    ref = None
    for _ in range(4):
        t, _ = capi.walk(base, w1, prev, w2=w2, seeds=seeds, mode=capi.PROBABILISTIC,
                         workspace=ws)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero()) == 0
        ref = t.clone() if ref is None else ref
        assert torch.equal(t, ref)


@pytest.mark.parametrize("bs,path", [(2, "default"), (6, "default"), (40, "default"),
                                     (6, "cuda_cores"), (2, "tensor_cores")])
@pytest.mark.parametrize("int8", [True, False])
def test_per_row_modes_and_temperatures(oracle, bs, path, int8):
    """Per-request mode and temperature in one walk: every group of rows with the same
    (mode, T) matches the oracle run with that mode and T, and every row equals the same
    row of a walk that gives all rows its settings (bit for bit: tokens and logits)."""
    V, K = 5003, 4
    inp = synth.make(V, bs, K, seed=70 + bs, peak=8.0)
    w1, w2, base, prev, seeds = to_dev(inp)
    okw, wk = {}, dict(w2=w2)
    if int8:
        q, sc = capi.quantize_w2(w2)
        _, q_ref, sc_ref = oracle.quantize_w2(bits(inp.w2))
        wk, okw = dict(w2q=q, scales=sc), dict(q=q_ref, sc=sc_ref)
    Ts = [0.5, 1.0, 0.7, 1.3]
    sampled = [b % 3 != 0 for b in range(bs)]
    T_row = [Ts[b % 4] for b in range(bs)]
    modes = torch.tensor([1 if s else 0 for s in sampled], dtype=torch.int32, device=DEV)
    temps = torch.tensor(T_row, dtype=torch.float32, device=DEV)
    flags = PATH_FLAGS.get(path, 0)
    tokens, lg = capi.walk(base, w1, prev, seeds=seeds, temperatures=temps, row_modes=modes,
                           want_logits=True, flags=flags, **wk)
    torch.cuda.synchronize()
    greedy_rows = [b for b in range(bs) if not sampled[b]]
    check_walk(oracle, inp, tokens, mode=capi.GREEDY, gpu_logits=lg, rows=greedy_rows, **okw)
    t_ref, l_ref = capi.walk(base, w1, prev, seeds=seeds, want_logits=True, flags=flags, **wk)
    torch.cuda.synchronize()
    assert torch.equal(tokens[greedy_rows], t_ref[greedy_rows])
    assert torch.equal(lg[greedy_rows].view(torch.int16), l_ref[greedy_rows].view(torch.int16))
    for T in Ts:
        rows = [b for b in range(bs) if sampled[b] and T_row[b] == T]
        if not rows:
            continue
        check_walk(oracle, inp, tokens, mode=capi.PROBABILISTIC, T=T, gpu_logits=lg, rows=rows, **okw)
        t_ref, _ = capi.walk(base, w1, prev, seeds=seeds, mode=capi.PROBABILISTIC, temperature=T,
                             flags=flags, **wk)
        torch.cuda.synchronize()
        assert torch.equal(tokens[rows], t_ref[rows]), T


@pytest.mark.parametrize("bs", [3, 40])
def test_per_row_settings_topk(oracle, bs):
    """The top-k walk with per-request mode and temperature equals, row by row, top-k
    walks that give every row those settings."""
    V, K, k = 3001, 3, 17
    inp = synth.make(V, bs, K, seed=80 + bs)
    w1, w2, base, prev, seeds = to_dev(inp)
    sampled = [b % 2 == 1 for b in range(bs)]
    T_row = [0.7 if b % 4 == 1 else 1.0 for b in range(bs)]
    modes = torch.tensor([1 if s else 0 for s in sampled], dtype=torch.int32, device=DEV)
    temps = torch.tensor(T_row, dtype=torch.float32, device=DEV)
    tokens, _ = capi.walk(base, w1, prev, w2=w2, seeds=seeds, top_k=k, temperatures=temps,
                          row_modes=modes)
    torch.cuda.synchronize()
    for mode, T in ((capi.GREEDY, 1.0), (capi.PROBABILISTIC, 1.0), (capi.PROBABILISTIC, 0.7)):
        rows = [b for b in range(bs) if sampled[b] == (mode == capi.PROBABILISTIC)
                and (mode == capi.GREEDY or T_row[b] == T)]
        if not rows:
            continue
        t_ref, _ = capi.walk(base, w1, prev, w2=w2, seeds=seeds, top_k=k, mode=mode, temperature=T)
        torch.cuda.synchronize()
        assert torch.equal(tokens[rows], t_ref[rows]), (mode, T)
        check_walk(oracle, inp, tokens, mode=mode, T=T, top_k=k, rows=rows)


@pytest.mark.parametrize("bs", [2, 5])
def test_invalid_per_row_settings_reported(bs):
    """An unknown per-row mode, or a sampled row with T <= 0 or NaN: INVALID_ARG, that
    row's tokens are -1, the other rows (a greedy row with T = 0 among them) walk on."""
    V, K = 4000, 3
    inp = synth.make(V, bs, K, seed=5)
    w1, w2, base, prev, seeds = to_dev(inp)
    m = [0, 7] + [1] * (bs - 2)
    T = [0.0, 1.0] + [float("nan") if b == 2 else 0.8 for b in range(2, bs)]
    modes = torch.tensor(m, dtype=torch.int32, device=DEV)
    temps = torch.tensor(T, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tokens, _ = capi.walk(base, w1, prev, w2=w2, seeds=seeds, temperatures=temps, row_modes=modes,
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    t = tokens.cpu().numpy()
    bad = [1] + ([2] if bs > 2 else [])
    assert all(list(t[r]) == [-1] * K for r in bad)
    assert all(np.all(t[r] >= 0) for r in range(bs) if r not in bad)


@pytest.mark.parametrize("bs,top_k", [(1, 0), (5, 0), (40, 0), (3, 17)])
def test_walk_captured_in_cuda_graph(bs, top_k):
    """The walk captured in a CUDA graph and replayed: every replay equals an eager walk
    on the inputs the graph's buffers hold at replay time (the workspace returns to zero
    after each replay)."""
    V, K = 6000, 4
    inp = synth.make(V, bs, K, seed=90 + bs)
    w1, w2, base, prev, seeds = to_dev(inp)
    tokens = torch.empty((bs, K), dtype=torch.int32, device=DEV)
    logits = torch.empty((bs, K, V), dtype=torch.bfloat16, device=DEV)
    ws = capi.alloc_workspace(V, bs, K, top_k)
    a = capi.make_args(base, w1, prev, tokens, ws, w2=w2, seeds=seeds, mode=capi.PROBABILISTIC,
                       temperature=0.8, top_k=top_k, logits=logits)
    assert capi.walk_args_call(a) == 0  # eager first: device query and kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert capi.walk_args_call(a, torch.cuda.current_stream()) == 0
    other = synth.make(V, bs, K, seed=190 + bs)
    for step in range(3):
        if step == 1:  # new inputs in the captured buffers
            base.copy_(other.base.to(DEV))
            prev.copy_(other.prev.to(DEV))
        tokens.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        ref, lref = capi.walk(base, w1, prev, w2=w2, seeds=seeds, mode=capi.PROBABILISTIC,
                              temperature=0.8, top_k=top_k, want_logits=True)
        torch.cuda.synchronize()
        assert torch.equal(tokens, ref), step
        assert torch.equal(logits.view(torch.int16), lref.view(torch.int16)), step
        if top_k == 0:  # (the top-k candidate lists stay in the workspace)
            assert int(ws.count_nonzero()) == 0


def test_walk_from_host_matches_device_walk():
    V, K, bs = 6000, 4, 3
    inp = synth.make(V, bs, K, seed=9)
    w1, w2, base, prev, seeds = to_dev(inp)
    ref, lref = capi.walk(base, w1, prev, w2=w2, seeds=seeds, mode=capi.PROBABILISTIC,
                          want_logits=True)
    base_h = inp.base.pin_memory()
    prev_h = inp.prev.pin_memory()
    seeds_h = inp.seeds.pin_memory()
    tok_h = torch.zeros((bs, K), dtype=torch.int32).pin_memory()
    lg_h = torch.zeros((bs, K, V), dtype=torch.bfloat16).pin_memory()
    base_d = torch.empty_like(base)
    prev_d = torch.empty_like(prev)
    seeds_d = torch.empty_like(seeds)
    tok_d = torch.empty((bs, K), dtype=torch.int32, device=DEV)
    lg_d = torch.empty((bs, K, V), dtype=torch.bfloat16, device=DEV)
    ws = capi.alloc_workspace(V, bs, K)
    args = capi.make_args(base_d, w1, prev_d, tok_d, ws, w2=w2, seeds=seeds_d,
                          mode=capi.PROBABILISTIC, logits=lg_d)
    capi.walk_from_host(args, base_h, prev_h, seeds_h, tok_h, lg_h)
    torch.cuda.synchronize()
    assert torch.equal(tok_h, ref.cpu())
    assert torch.equal(lg_h.view(torch.int16), lref.cpu().view(torch.int16))


# ------------------------------------------------------------------ top-k walk

@pytest.mark.parametrize("k", [1, 17, 300])
@pytest.mark.parametrize("mode,T", [(capi.GREEDY, 1.0), (capi.PROBABILISTIC, 1.0),
                                    (capi.PROBABILISTIC, 0.7)])
@pytest.mark.parametrize("int8", [False, True])
def test_topk_small_parity(oracle, k, mode, T, int8):
    V, K, bs = 3001, 3, 5
    inp = synth.make(V, bs, K, seed=20 + k)
    w1, w2, base, prev, seeds = to_dev(inp)
    wk, okw = dict(w2=w2), {}
    if int8:  # int8 codes with per-row scales: 256-byte gathered rows
        q, sc = capi.quantize_w2(w2)
        _, q_ref, sc_ref = oracle.quantize_w2(bits(inp.w2))
        wk, okw = dict(w2q=q, scales=sc), dict(q=q_ref, sc=sc_ref)
    tokens, lg = capi.walk(base, w1, prev, seeds=seeds, mode=mode, temperature=T,
                           top_k=k, want_logits=True, **wk)
    torch.cuda.synchronize()
    check_walk(oracle, inp, tokens, mode=mode, T=T, top_k=k, gpu_logits=lg, **okw)


@pytest.mark.parametrize("case", ["sampled", "ranked_ties", "wide_tie", "overflow"])
def test_topk_select_paths(oracle, case):
    """Every path of the candidate selection gives the oracle's candidate set (draft_logits
    are -inf exactly off the candidates) and tokens: a list collected above a sampled
    pivot; a boundary tie ranked by index; a tie too wide to rank and a list too long
    for shared memory, both taking the exact whole-row selection."""
    V, K, bs = 20000, 2, 2  # V a multiple of 8: 16-byte row loads
    inp = synth.make(V, bs, K, seed=41)
    g = torch.Generator().manual_seed(7)
    base = inp.base.float()
    k = 300
    if case == "ranked_ties":  # 500 equal top keys, 300 of them taken by index
        base[:, :, torch.randperm(V, generator=g)[:500]] = 12.0
    elif case == "wide_tie":  # 3000 equal top keys, 1000 taken
        base[:, :, torch.randperm(V, generator=g)[:3000]] = 12.0
        k = 1000
    elif case == "overflow":  # every key equal
        base[:] = 1.0
    inp.base = base.bfloat16()
    w1, w2, basedev, prev, seeds = to_dev(inp)
    for mode in (capi.GREEDY, capi.PROBABILISTIC):
        tokens, lg = capi.walk(basedev, w1, prev, w2=w2, seeds=seeds, mode=mode, top_k=k,
                               want_logits=True)
        torch.cuda.synchronize()
        check_walk(oracle, inp, tokens, mode=mode, top_k=k, gpu_logits=lg)


def test_topk_full_vocab_equals_dense():
    V, K, bs = 2003, 4, 3
    inp = synth.make(V, bs, K, seed=31)
    w1, w2, base, prev, seeds = to_dev(inp)
    for mode in (capi.GREEDY, capi.PROBABILISTIC):
        td, ld = capi.walk(base, w1, prev, w2=w2, seeds=seeds, mode=mode, want_logits=True)
        tk, lk = capi.walk(base, w1, prev, w2=w2, seeds=seeds, mode=mode, top_k=V,
                           want_logits=True)
        torch.cuda.synchronize()
        assert torch.equal(td, tk)
        # the same bias in both walks (fp32 sums of the same products, in possibly
        # different orders): bf16 logits within the parity tolerance of each other
        a, b = ld.float().double().cpu().numpy(), lk.float().double().cpu().numpy()
        assert np.all(np.abs(a - b) <= 2e-2 + 1e-2 * np.abs(b))


def test_topk_boundary_ties_and_all_neg_inf(oracle):
    V, K, bs = 1000, 2, 3
    inp = synth.make(V, bs, K, seed=5)
    base = torch.full((bs, K, V), -5.0)
    base[0, :, 10:20] = 3.0          # ten-way tie at the top, k = 4 takes 10..13
    base[1] = float("-inf")          # all -inf -> token 0
    base[2, :, 500] = float("nan")   # NaN is the largest candidate
    inp.base = base.bfloat16()
    w1, w2, bd, prev, seeds = to_dev(inp)
    tokens, lg = capi.walk(bd, w1, prev, w2=w2, seeds=seeds, mode=capi.GREEDY, top_k=4,
                           want_logits=True)
    torch.cuda.synchronize()
    t = tokens.cpu().numpy()
    assert np.all(t[1] == 0) and np.all(t[2] == 500)
    check_walk(oracle, inp, tokens, mode=capi.GREEDY, top_k=4, gpu_logits=lg)


# ------------------------------------------------------------------ full-size workloads

def _full_case(oracle, V, K, bs, int8, mode, T, peak, logits, top_k=0):
    inp = synth.make(V, bs, K, seed=0, peak=peak)
    w1, w2, base, prev, seeds = to_dev(inp)
    q_ref = sc_ref = None
    wk = dict(w2=w2)
    if int8:
        q, sc = capi.quantize_w2(w2)
        _, q_ref, sc_ref = oracle.quantize_w2(bits(inp.w2))
        torch.cuda.synchronize()
        assert np.array_equal(q.cpu().numpy(), q_ref)
        wk = dict(w2q=q, scales=sc)
    tokens, lg = capi.walk(base, w1, prev, seeds=seeds, mode=mode, temperature=T, top_k=top_k,
                           want_logits=logits, **wk)
    torch.cuda.synchronize()
    assert int(tokens.min()) >= 0
    label = (f"V={V} K={K} bs={bs} {'int8' if int8 else 'bf16'} "
             f"{'greedy' if mode == capi.GREEDY else f'prob T={T}'}{f' top-k {top_k}' if top_k else ''}"
             f"{' +logits' if logits else ''}")
    return check_walk_rows(oracle, inp, tokens, label=label, mode=mode, T=T, top_k=top_k, q=q_ref, sc=sc_ref,
                           gpu_logits=lg)


FULL = [
    # V, K, bs, int8, mode, T, peak, logits -- every row checked
    (129280, 5, 1, False, capi.GREEDY, 1.0, None, False),
    (151936, 7, 1, True, capi.GREEDY, 1.0, 8.0, False),
    (151936, 7, 1, True, capi.PROBABILISTIC, 1.0, 8.0, True),
    (151936, 7, 16, True, capi.GREEDY, 1.0, 8.0, False),
    (151936, 7, 16, True, capi.PROBABILISTIC, 1.0, 8.0, False),
    (151936, 7, 64, True, capi.GREEDY, 1.0, 8.0, False),
    (151936, 7, 64, True, capi.PROBABILISTIC, 1.0, 8.0, True),
    (151936, 16, 1, False, capi.PROBABILISTIC, 0.7, 8.0, True),
    (151936, 16, 64, False, capi.PROBABILISTIC, 0.7, 8.0, True),
    (248320, 16, 1, True, capi.GREEDY, 1.0, None, False),
    (248320, 16, 16, True, capi.GREEDY, 1.0, None, False),
    (248320, 16, 64, True, capi.GREEDY, 1.0, None, False),
]


@pytest.mark.parametrize("V,K,bs,int8,mode,T,peak,logits", FULL)
def test_full_size_every_row(oracle, V, K, bs, int8, mode, T, peak, logits):
    _full_case(oracle, V, K, bs, int8, mode, T, peak, logits)


@pytest.mark.parametrize("k", [512, 4096])
def test_full_size_topk_every_row(oracle, k):
    _full_case(oracle, 151936, 7, 64, False, capi.PROBABILISTIC, 1.0, None, True, top_k=k)
