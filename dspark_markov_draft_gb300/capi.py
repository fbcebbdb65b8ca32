"""Python binding of libdspark.so (ctypes): argument marshalling only.

Every function here forwards torch CUDA tensors to the C ABI in include/dspark.h as raw
device pointers plus the current CUDA stream. Nothing is computed in Python and there
is no fallback: if the library is missing or the call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdspark.so")

GREEDY, PROBABILISTIC = 0, 1
FLAG_SKIP_ARRIVAL_CTA0 = 0x1
FLAG_FORCE_CUDA_CORES = 0x2
FLAG_FORCE_TENSOR_CORES = 0x4
RANK = 256
MAX_BS = 64
MAX_K = 32

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "COOP_TOO_LARGE",
          5: "TIMEOUT", 6: "BAD_TOKEN", 7: "NONFINITE_W2", 8: "WORKSPACE"}


class DsparkError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == 3:
            detail = ": " + lib().dspark_last_cuda_error().decode()
        super().__init__(f"{what} failed with {STATUS.get(status, status)}{detail}")


class WalkArgs(C.Structure):
    _fields_ = [
        ("base_logits", C.c_void_p), ("w1", C.c_void_p), ("w2", C.c_void_p),
        ("w2q", C.c_void_p), ("w2_scales", C.c_void_p), ("prev_tokens", C.c_void_p),
        ("seeds", C.c_void_p), ("V", C.c_int64), ("rank", C.c_int32), ("bs", C.c_int32),
        ("K", C.c_int32), ("mode", C.c_int32), ("temperature", C.c_float),
        ("top_k", C.c_int32), ("draft_tokens", C.c_void_p), ("draft_logits", C.c_void_p),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
        ("status_dev", C.c_void_p), ("flags", C.c_uint32), ("resident_rows_cap", C.c_int32),
        ("timeout_us", C.c_uint32), ("temperatures", C.c_void_p), ("row_modes", C.c_void_p),
        ("topk_cand", C.c_void_p), ("topk_base", C.c_void_p),
    ]


class LmheadArgs(C.Structure):
    _fields_ = [
        ("hidden", C.c_void_p), ("lm_head", C.c_void_p), ("V", C.c_int64), ("M", C.c_int32),
        ("d", C.c_int32), ("top_k", C.c_int32), ("cand", C.c_void_p), ("cand_base", C.c_void_p),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t), ("status_dev", C.c_void_p),
        ("stats_dev", C.c_void_p), ("flags", C.c_uint32), ("timeout_us", C.c_uint32),
    ]


LMHEAD_FLAG_EXACT = 0x1


class VerifyArgs(C.Structure):
    _fields_ = [
        ("target_logits", C.c_void_p), ("draft_logits", C.c_void_p), ("draft_tokens", C.c_void_p),
        ("seeds", C.c_void_p), ("V", C.c_int64), ("bs", C.c_int32), ("K", C.c_int32),
        ("temperature", C.c_float), ("accepted", C.c_void_p), ("out_tokens", C.c_void_p),
        ("norms", C.c_void_p),
    ]


_lib = None


def lib():
    """Load libdspark.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "dspark_markov_draft_gb300.build.build() (nvcc, sm_103a)")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        L.dspark_quantize_w2.argtypes = [vp, i64, i32, vp, vp, vp, vp]
        L.dspark_walk.argtypes = [C.POINTER(WalkArgs), vp]
        L.dspark_walk_topk.argtypes = [C.POINTER(WalkArgs), vp]
        L.dspark_walk_noalloc.argtypes = [C.POINTER(WalkArgs), vp]
        L.dspark_walk_from_host.argtypes = [C.POINTER(WalkArgs), vp, vp, vp, vp, vp, vp]
        L.dspark_walk_workspace_size.argtypes = [i64, i32, i32, i32]
        L.dspark_walk_workspace_size.restype = C.c_size_t
        L.dspark_query_capacity.argtypes = [i32, i64, i32, i32, C.POINTER(C.c_int32),
                                            C.POINTER(C.c_int64)]
        L.dspark_gumbel_noise.argtypes = [vp, i32, i32, i64, vp, vp, vp]
        L.dspark_verify.argtypes = [C.POINTER(VerifyArgs), vp]
        L.dspark_lmhead_topk.argtypes = [C.POINTER(LmheadArgs), vp]
        L.dspark_lmhead_workspace_size.argtypes = [i32, i64, i32]
        L.dspark_lmhead_workspace_size.restype = C.c_size_t
        L.dspark_status_string.argtypes = [i32]
        L.dspark_status_string.restype = C.c_char_p
        L.dspark_last_cuda_error.argtypes = []
        L.dspark_last_cuda_error.restype = C.c_char_p
        for f in ("dspark_quantize_w2", "dspark_walk", "dspark_walk_topk", "dspark_walk_noalloc",
                  "dspark_walk_from_host", "dspark_query_capacity", "dspark_gumbel_noise",
                  "dspark_verify", "dspark_lmhead_topk"):
            getattr(L, f).restype = C.c_int32
        _lib = L
    return _lib


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdspark must be contiguous")
    return t.data_ptr()


def _dev_ptr(t: torch.Tensor | None):
    if t is not None and not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return _ptr(t)


def _expect(t: torch.Tensor, shape, dtypes, name: str, device):
    """A contiguous tensor of this shape and one of these dtypes on `device`."""
    if tuple(t.shape) != tuple(shape) or t.dtype not in dtypes or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous {'/'.join(map(str, dtypes))} tensor of shape "
                         f"{tuple(shape)}, got {t.dtype} {tuple(t.shape)}"
                         f"{'' if t.is_contiguous() else ' (not contiguous)'}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise DsparkError(status, what)


def workspace_size(V: int, bs: int, K: int, top_k: int = 0) -> int:
    return int(lib().dspark_walk_workspace_size(V, bs, K, top_k))


def alloc_workspace(V: int, bs: int, K: int, top_k: int = 0, device=None) -> torch.Tensor:
    """A zeroed workspace tensor (uint8) of the size the walk needs."""
    n = workspace_size(V, bs, K, top_k)
    return torch.zeros(n + 256, dtype=torch.uint8, device=device or "cuda")


def _ws_view(ws: torch.Tensor):
    """(pointer aligned to 256 bytes, usable bytes)."""
    p = ws.data_ptr()
    off = (-p) % 256
    return p + off, ws.numel() - off


def query_capacity(device: int, V: int, int8: bool, bs: int):
    g, r = C.c_int32(), C.c_int64()
    _check(lib().dspark_query_capacity(device, V, int(int8), bs, C.byref(g), C.byref(r)),
           "dspark_query_capacity")
    return g.value, r.value


def quantize_w2(w2: torch.Tensor, q: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                status: torch.Tensor | None = None, stream=None):
    """bf16 [V, 256] -> (int8 [V, 256], fp32 [V]) via dspark_quantize_w2."""
    V = w2.shape[0]
    q = q if q is not None else torch.empty((V, RANK), dtype=torch.int8, device=w2.device)
    scales = scales if scales is not None else torch.empty(V, dtype=torch.float32, device=w2.device)
    _check(lib().dspark_quantize_w2(_dev_ptr(w2), V, w2.shape[1], _dev_ptr(q), _dev_ptr(scales),
                                    _dev_ptr(status), _stream(stream)), "dspark_quantize_w2")
    return q, scales


def make_args(base, w1, prev, tokens, workspace, *, w2=None, w2q=None, scales=None, seeds=None,
              mode=GREEDY, temperature=1.0, top_k=0, logits=None, status=None, flags=0,
              resident_rows_cap=-1, timeout_us=0, temperatures=None, row_modes=None,
              topk_cand=None, topk_base=None, V=None) -> WalkArgs:
    """temperatures (fp32 [bs]) and row_modes (int32 [bs]), device tensors, override the
    scalar temperature and mode row by row. topk_cand (int32 [bs, K, top_k]) and
    topk_base (fp32, same shape): candidates chosen elsewhere (base may then be None,
    with V given)."""
    if base is not None:
        bs, K, V = base.shape
    else:
        bs, K = tokens.shape
        if V is None or topk_cand is None:
            raise ValueError("without base logits: topk_cand, topk_base and V are required")
    for t, name, dt in ((topk_cand, "topk_cand", torch.int32), (topk_base, "topk_base", torch.float32)):
        if t is not None:
            _expect(t, (bs, K, top_k), (dt,), name, tokens.device)
    wsp, wsn = _ws_view(workspace)
    return WalkArgs(
        _dev_ptr(base), _dev_ptr(w1), _dev_ptr(w2), _dev_ptr(w2q), _dev_ptr(scales),
        _dev_ptr(prev), _dev_ptr(seeds), V, w1.shape[1], bs, K, mode, temperature, top_k,
        _dev_ptr(tokens), _dev_ptr(logits), wsp, wsn, _dev_ptr(status), flags,
        resident_rows_cap, timeout_us, _dev_ptr(temperatures), _dev_ptr(row_modes),
        _dev_ptr(topk_cand), _dev_ptr(topk_base))


def walk(base, w1, prev, *, w2=None, w2q=None, scales=None, seeds=None, mode=GREEDY,
         temperature=1.0, top_k=0, tokens=None, logits=None, want_logits=False, workspace=None,
         status=None, flags=0, resident_rows_cap=-1, timeout_us=0, stream=None,
         temperatures=None, row_modes=None, topk_cand=None, topk_base=None, V=None):
    """Run dspark_walk (or dspark_walk_topk when top_k > 0). Returns (tokens, logits).
    With topk_cand / topk_base (e.g. from lmhead_topk) base may be None and V given."""
    if base is not None:
        bs, K, V = base.shape
        dev = base.device
    else:
        bs, K = topk_cand.shape[:2]
        dev = topk_cand.device
    if tokens is None:
        tokens = torch.empty((bs, K), dtype=torch.int32, device=dev)
    if want_logits and logits is None:
        logits = torch.empty((bs, K, V), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = alloc_workspace(V, bs, K, top_k, device=dev)
    a = make_args(base, w1, prev, tokens, workspace, w2=w2, w2q=w2q, scales=scales,
                  seeds=seeds, mode=mode, temperature=temperature, top_k=top_k, logits=logits,
                  status=status, flags=flags, resident_rows_cap=resident_rows_cap,
                  timeout_us=timeout_us, temperatures=temperatures, row_modes=row_modes,
                  topk_cand=topk_cand, topk_base=topk_base, V=V)
    _check(lib().dspark_walk(C.byref(a), _stream(stream)), "dspark_walk")
    return tokens, logits


def lmhead_workspace(M: int, V: int, top_k: int, device=None) -> torch.Tensor:
    n = int(lib().dspark_lmhead_workspace_size(M, V, top_k))
    if n == 0:
        raise ValueError("invalid sizes for dspark_lmhead_workspace_size")
    return torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")


def lmhead_topk(hidden, lm_head, top_k: int, *, cand=None, cand_base=None, workspace=None, status=None,
                stats=None, exact=False, timeout_us=0, stream=None):
    """dspark_lmhead_topk: the top_k largest LM-head logits of every hidden row without the
    dense logits. hidden bf16 [M, d], lm_head bf16 [V, d]. Returns (cand int32 [M, top_k],
    cand_base fp32 [M, top_k])."""
    M, d = hidden.shape
    V = lm_head.shape[0]
    dev = hidden.device
    _expect(hidden, (M, d), (torch.bfloat16,), "hidden", dev)
    _expect(lm_head, (V, d), (torch.bfloat16,), "lm_head", dev)
    if cand is None:
        cand = torch.empty((M, top_k), dtype=torch.int32, device=dev)
    if cand_base is None:
        cand_base = torch.empty((M, top_k), dtype=torch.float32, device=dev)
    _expect(cand, (M, top_k), (torch.int32,), "cand", dev)
    _expect(cand_base, (M, top_k), (torch.float32,), "cand_base", dev)
    if workspace is None:
        workspace = lmhead_workspace(M, V, top_k, device=dev)
    wsp, wsn = _ws_view(workspace)
    a = LmheadArgs(_dev_ptr(hidden), _dev_ptr(lm_head), V, M, d, top_k, _dev_ptr(cand), _dev_ptr(cand_base),
                   wsp, wsn, _dev_ptr(status), _dev_ptr(stats), LMHEAD_FLAG_EXACT if exact else 0, timeout_us)
    _check(lib().dspark_lmhead_topk(C.byref(a), _stream(stream)), "dspark_lmhead_topk")
    return cand, cand_base


def walk_args_call(args: WalkArgs, stream=None, topk: bool = False) -> int:
    """Call dspark_walk / dspark_walk_topk on prepared arguments; returns the status."""
    f = lib().dspark_walk_topk if topk else lib().dspark_walk
    return int(f(C.byref(args), _stream(stream)))


def walk_noalloc(args: WalkArgs, stream=None) -> int:
    """Call dspark_walk_noalloc (scratch from the library's static array); returns the status."""
    return int(lib().dspark_walk_noalloc(C.byref(args), _stream(stream)))


def walk_from_host(args: WalkArgs, base_host, prev_host, seeds_host, tokens_host,
                   logits_host=None, stream=None):
    _check(lib().dspark_walk_from_host(C.byref(args), _ptr(base_host), _ptr(prev_host),
                                       _ptr(seeds_host), _ptr(tokens_host), _ptr(logits_host),
                                       _stream(stream)), "dspark_walk_from_host")


def verify(target_logits, draft_logits, draft_tokens, seeds, temperature=1.0, *, accepted=None,
           out_tokens=None, reuse_norms=True, stream=None):
    """dspark_verify: speculative-sampling verification. target_logits bf16 [bs, K+1, V],
    draft_logits bf16 [bs, K, V], draft_tokens int32 [bs, K], seeds [bs]. reuse_norms:
    pass the normaliser scratch (the sample pass reuses the acceptance pass's softmax
    normalisers); False: NULL, recomputed.
    Returns (accepted int32 [bs], out_tokens int32 [bs, K+1])."""
    bs, K1, V = target_logits.shape
    dev = target_logits.device
    # the kernels index these buffers by (bs, K, V): refuse a mismatch here rather than
    # read past a buffer on the device
    _expect(target_logits, (bs, K1, V), (torch.bfloat16,), "target_logits", dev)
    _expect(draft_logits, (bs, K1 - 1, V), (torch.bfloat16,), "draft_logits", dev)
    _expect(draft_tokens, (bs, K1 - 1), (torch.int32,), "draft_tokens", dev)
    _expect(seeds, (bs,), (torch.int64, getattr(torch, "uint64", torch.int64)), "seeds", dev)
    if accepted is None:
        accepted = torch.empty(bs, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((bs, K1), dtype=torch.int32, device=dev)
    _expect(accepted, (bs,), (torch.int32,), "accepted", dev)
    _expect(out_tokens, (bs, K1), (torch.int32,), "out_tokens", dev)
    norms = torch.empty((bs, K1 - 1, 4), dtype=torch.float32, device=dev) if reuse_norms else None
    a = VerifyArgs(_dev_ptr(target_logits), _dev_ptr(draft_logits), _dev_ptr(draft_tokens),
                   _dev_ptr(seeds), V, bs, K1 - 1, temperature, _dev_ptr(accepted),
                   _dev_ptr(out_tokens), _dev_ptr(norms) if norms is not None else None)
    _check(lib().dspark_verify(C.byref(a), _stream(stream)), "dspark_verify")
    return accepted, out_tokens


def gumbel_noise(seeds: torch.Tensor, K: int, V: int, stream=None):
    """(words uint32 as int32, gumbel fp32), each [bs, K, V]."""
    bs = seeds.shape[0]
    words = torch.empty((bs, K, V), dtype=torch.int32, device=seeds.device)
    g = torch.empty((bs, K, V), dtype=torch.float32, device=seeds.device)
    _check(lib().dspark_gumbel_noise(_dev_ptr(seeds), bs, K, V, _dev_ptr(words), _dev_ptr(g),
                                     _stream(stream)), "dspark_gumbel_noise")
    return words, g
