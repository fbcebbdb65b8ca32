"""Host-side checks of the C ABI that need no GPU: the library builds for sm_103a,
loads, exports every entry point the public header declares, and rejects bad
arguments before touching the device."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from dspark_markov_draft_gb300 import build, capi
    build.build()
    return capi.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dspark.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("dspark_quantize_w2", "dspark_walk", "dspark_walk_topk",
                     "dspark_walk_workspace_size", "dspark_query_capacity",
                     "dspark_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    from dspark_markov_draft_gb300 import capi
    for code in capi.STATUS:
        s = L.dspark_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.dspark_status_string(999).decode() == "unknown status"


def test_workspace_size_grows_with_shape(L):
    from dspark_markov_draft_gb300 import capi
    a = capi.workspace_size(151936, 1, 7)
    b = capi.workspace_size(151936, 64, 7)
    c = capi.workspace_size(151936, 64, 7, 4096)
    assert 0 < a < b < c
    # a top-k walk keeps the candidate ids (int32) and their base logits (fp32) that the
    # selection writes for the walk: 8 bytes per (row, position, candidate)
    assert c - b >= 64 * 7 * 4096 * 8
    assert capi.workspace_size(10, 0, 1) == 0


def test_invalid_arguments_rejected_on_host(L):
    from dspark_markov_draft_gb300 import capi
    assert L.dspark_walk(None, None) == 1
    a = capi.WalkArgs()
    assert L.dspark_walk(C.byref(a), None) == 1          # null pointers
    # plausible non-null (never dereferenced) pointers with a bad rank / size / mode
    fake = 1 << 20
    def args(**kw):
        d = dict(base_logits=fake, w1=fake, w2=fake, prev_tokens=fake, draft_tokens=fake,
                 workspace=fake, workspace_bytes=1 << 20, V=1000, rank=256, bs=1, K=2,
                 mode=0, temperature=1.0, top_k=0, resident_rows_cap=-1)
        d.update(kw)
        x = capi.WalkArgs()
        for k, v in d.items():
            setattr(x, k, v)
        return x
    for bad in (dict(rank=128), dict(bs=0), dict(bs=65), dict(K=0), dict(K=33), dict(V=0),
                dict(mode=2), dict(mode=1, seeds=fake, temperature=0.0),
                dict(mode=1, seeds=None), dict(w2q=fake), dict(top_k=1001),
                dict(row_modes=fake, seeds=None),                      # per-row modes need seeds
                dict(row_modes=fake, seeds=fake, temperature=0.0)):    # ... and a valid scalar T
        assert L.dspark_walk(C.byref(args(**bad)), None) == 1, bad
    for bad in (dict(w2q=fake, w2=None),                       # int8 W2 without its scales
                dict(w1=fake + 8), dict(w2=fake + 4),            # rows not 16-byte aligned
                dict(V=(1 << 31)), dict(top_k=-1),
                dict(mode=1, seeds=fake, temperature=float("inf")),
                dict(mode=1, seeds=fake, temperature=float("nan"))):
        assert L.dspark_walk(C.byref(args(**bad)), None) == 1, bad
    # the top-k and allocation-free entry points apply the same checks first (the latter
    # before it looks up its scratch on the device, so here, with no GPU, too)
    for f in (L.dspark_walk_topk, L.dspark_walk_noalloc):
        assert f(None, None) == 1
        for bad in (dict(rank=128), dict(bs=65), dict(K=33), dict(mode=1, seeds=None)):
            assert f(C.byref(args(**bad)), None) == 1, (f, bad)
    assert L.dspark_walk_topk(C.byref(args(top_k=0)), None) == 1      # k >= 1 required
    assert L.dspark_walk_noalloc(C.byref(args(top_k=5)), None) == 2   # full vocabulary only
    assert L.dspark_walk_noalloc(C.byref(args(top_k=-1)), None) == 1  # invalid before unsupported
    assert L.dspark_walk(C.byref(args(workspace_bytes=16)), None) == 8
    assert L.dspark_walk(C.byref(args(workspace=None)), None) == 8
    assert L.dspark_walk(C.byref(args(workspace=fake + 128)), None) == 8   # not 256-byte aligned
    assert L.dspark_quantize_w2(None, 10, 256, None, None, None, None) == 1
    assert L.dspark_quantize_w2(fake, 10, 255, fake, fake, None, None) == 1
    assert L.dspark_gumbel_noise(None, 1, 1, 10, None, None, None) == 1
    v = capi.VerifyArgs()
    assert L.dspark_verify(C.byref(v), None) == 1                     # null pointers
    for bad in (dict(V=0), dict(bs=0), dict(bs=65), dict(K=0), dict(K=33), dict(temperature=0.0),
                dict(temperature=float("nan"))):
        d = dict(target_logits=fake, draft_logits=fake, draft_tokens=fake, seeds=fake, V=100,
                 bs=2, K=3, temperature=1.0, accepted=fake, out_tokens=fake)
        d.update(bad)
        x = capi.VerifyArgs()
        for k, val in d.items():
            setattr(x, k, val)
        assert L.dspark_verify(C.byref(x), None) == 1, bad
    # the optional normaliser scratch must be 16-byte aligned
    d = dict(target_logits=fake, draft_logits=fake, draft_tokens=fake, seeds=fake, V=100,
             bs=2, K=3, temperature=1.0, accepted=fake, out_tokens=fake, norms=fake + 4)
    x = capi.VerifyArgs()
    for k, val in d.items():
        setattr(x, k, val)
    assert L.dspark_verify(C.byref(x), None) == 1


def test_verify_binding_refuses_mismatched_buffers():
    """The binding checks shapes, dtypes and contiguity before any pointer reaches the
    kernels (which index the buffers by bs, K and V): CPU tensors suffice to see it."""
    import torch
    from dspark_markov_draft_gb300 import capi
    bs, K, V = 3, 2, 10
    good = dict(t=torch.zeros(bs, K + 1, V, dtype=torch.bfloat16), d=torch.zeros(bs, K, V, dtype=torch.bfloat16),
                k=torch.zeros(bs, K, dtype=torch.int32), s=torch.zeros(bs, dtype=torch.int64))
    bad = [dict(d=torch.zeros(bs, K + 1, V, dtype=torch.bfloat16)),          # K mismatch
           dict(d=torch.zeros(bs, K, V, dtype=torch.float32)),               # dtype
           dict(k=torch.zeros(bs, K, dtype=torch.int64)),
           dict(s=torch.zeros(bs + 1, dtype=torch.int64)),
           dict(t=torch.zeros(bs, V, K + 1, dtype=torch.bfloat16).transpose(1, 2))]  # not contiguous
    for over in bad:
        a = dict(good, **over)
        with pytest.raises(ValueError, match="expected a contiguous"):
            capi.verify(a["t"], a["d"], a["k"], a["s"], 1.0)
    with pytest.raises(ValueError, match="CUDA tensor"):  # well-formed, but on the host
        capi.verify(good["t"], good["d"], good["k"], good["s"], 1.0,
                    accepted=torch.zeros(bs, dtype=torch.int32), out_tokens=torch.zeros(bs, K + 1, dtype=torch.int32))


def test_lmhead_arguments_rejected_on_host(L):
    """dspark_lmhead_topk refuses bad shapes, unaligned rows and a short workspace before
    any CUDA call; the workspace size grows with every dimension."""
    from dspark_markov_draft_gb300 import capi
    fake = 1 << 20
    ws = int(L.dspark_lmhead_workspace_size(448, 151936, 512))
    assert ws > 0
    assert int(L.dspark_lmhead_workspace_size(448, 151936, 4096)) > ws
    assert int(L.dspark_lmhead_workspace_size(0, 151936, 512)) == 0
    assert int(L.dspark_lmhead_workspace_size(448, 151936, 0)) == 0

    def args(**kw):
        d = dict(hidden=fake, lm_head=fake, V=151936, M=448, d=2048, top_k=512, cand=fake, cand_base=fake,
                 workspace=fake, workspace_bytes=ws)
        d.update(kw)
        x = capi.LmheadArgs()
        for k, v in d.items():
            setattr(x, k, v)
        return x
    assert L.dspark_lmhead_topk(None, None) == 1
    for bad in (dict(hidden=None), dict(lm_head=None), dict(cand=None), dict(cand_base=None),
                dict(M=0), dict(V=0), dict(d=32), dict(d=2000), dict(d=16384 + 64),
                dict(top_k=0), dict(top_k=8193), dict(V=100, top_k=101),
                dict(hidden=fake + 8), dict(lm_head=fake + 2)):
        assert L.dspark_lmhead_topk(C.byref(args(**bad)), None) == 1, bad
    for bad in (dict(workspace=None), dict(workspace=fake + 64), dict(workspace_bytes=ws - 1)):
        assert L.dspark_lmhead_topk(C.byref(args(**bad)), None) == 8, bad
