"""ctypes binding of the CPU oracle (dspark_oracle.cpp).

TEST INFRASTRUCTURE ONLY: the test suite, the package's smoke check and the
benchmark's CPU-baseline leg are the only callers. Nothing on the product path
imports this module.

`build()` compiles the oracle with g++ (-O2 -ffp-contract=off, no fast-math,
OpenMP) into ``oracle/libdspark_oracle.so`` next to the source.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dspark_oracle.cpp")
LIB = os.path.join(HERE, "libdspark_oracle.so")

GREEDY, PROBABILISTIC = 0, 1
CLASS_SAME, CLASS_NEAR_TIE, CLASS_BF16_BOUNDARY, CLASS_REJECTED = 0, 1, 2, 255


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


class _WalkArgs(C.Structure):
    _fields_ = [
        ("base", C.c_void_p), ("w1", C.c_void_p), ("w2", C.c_void_p), ("w2q", C.c_void_p),
        ("w2_scales", C.c_void_p), ("prev", C.c_void_p), ("seeds", C.c_void_p),
        ("slot", C.c_void_p),
        ("V", C.c_int64), ("R", C.c_int32), ("bs", C.c_int32), ("K", C.c_int32),
        ("mode", C.c_int32), ("temperature", C.c_float), ("top_k", C.c_int32),
        ("follow", C.c_void_p), ("tie_tol", C.c_double), ("bf16_eps", C.c_double),
        ("nthreads", C.c_int32),
        ("tokens", C.c_void_p), ("gap", C.c_void_p), ("best_score", C.c_void_p),
        ("follow_class", C.c_void_p), ("logits", C.c_void_p), ("logits_bf16", C.c_void_p),
        ("scores", C.c_void_p), ("cand", C.c_void_p), ("base_f64", C.c_void_p),
    ]


_lib = None


def bind(L):
    """Declare the C signatures of an oracle library handle (also used by the tests
    that build copies of the oracle with planted mistakes)."""
    L.oracle_bf16_to_double.restype = C.c_double
    L.oracle_bf16_to_double.argtypes = [C.c_uint16]
    L.oracle_round_bf16.restype = C.c_uint16
    L.oracle_round_bf16.argtypes = [C.c_double]
    L.oracle_philox4x32_10.restype = None
    L.oracle_philox4x32_10.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
    L.oracle_gumbel_block.restype = None
    L.oracle_gumbel_block.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_int64,
                                      C.c_void_p, C.c_void_p, C.c_void_p]
    L.oracle_quantize_w2.restype = C.c_int32
    L.oracle_quantize_w2.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_void_p,
                                     C.c_void_p]
    L.oracle_topk_select.restype = C.c_int32
    L.oracle_topk_select.argtypes = [C.c_void_p, C.c_int32, C.c_int64, C.c_int32,
                                     C.c_void_p]
    L.oracle_walk.restype = C.c_int32
    L.oracle_walk.argtypes = [C.POINTER(_WalkArgs)]
    L.oracle_lmhead_logits.restype = C.c_int32
    L.oracle_lmhead_logits.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int64,
                                       C.c_void_p, C.c_int32]
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = bind(C.CDLL(build()))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def round_bf16(x: float) -> int:
    return int(lib().oracle_round_bf16(float(x)))


def bf16_to_double(h: int) -> float:
    return float(lib().oracle_bf16_to_double(int(h)))


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def gumbel_block(seeds, K: int, V: int):
    """(words uint32, u float32, g float64), each [bs, K, V]."""
    s = _c(seeds, np.uint64)
    bs = s.shape[0]
    words = np.zeros((bs, K, V), dtype=np.uint32)
    u = np.zeros((bs, K, V), dtype=np.float32)
    g = np.zeros((bs, K, V), dtype=np.float64)
    lib().oracle_gumbel_block(s.ctypes.data, bs, K, V, words.ctypes.data, u.ctypes.data,
                              g.ctypes.data)
    return words, u, g


def quantize_w2(w2_bits: np.ndarray):
    """(status, q int8 [V, R], scales fp32 [V]) from a bf16 bit-pattern array."""
    w = _c(w2_bits, np.uint16)
    V, R = w.shape
    q = np.zeros((V, R), dtype=np.int8)
    sc = np.zeros(V, dtype=np.float32)
    st = lib().oracle_quantize_w2(w.ctypes.data, V, R, q.ctypes.data, sc.ctypes.data)
    return int(st), q, sc


def topk_select(base_bits: np.ndarray, k: int):
    b = _c(base_bits, np.uint16)
    V = b.shape[-1]
    rows = int(np.prod(b.shape[:-1]))
    cand = np.zeros(b.shape[:-1] + (k,), dtype=np.int32)
    st = lib().oracle_topk_select(b.ctypes.data, rows, V, k, cand.ctypes.data)
    if st != 0:
        raise ValueError(f"oracle_topk_select status {st}")
    return cand


@dataclass
class WalkResult:
    status: int
    tokens: np.ndarray
    gap: np.ndarray
    best_score: np.ndarray
    follow_class: np.ndarray | None
    logits: np.ndarray | None
    logits_bf16: np.ndarray | None
    scores: np.ndarray | None
    cand: np.ndarray | None


def lmhead_logits(hidden_bits, lm_head_bits, nthreads: int = 1) -> np.ndarray:
    """fp64 LM-head logits [M, V] of bf16 hidden states [M, d] and LM head [V, d]."""
    h = _c(hidden_bits, np.uint16)
    w = _c(lm_head_bits, np.uint16)
    M, d = h.shape
    V = w.shape[0]
    assert w.shape[1] == d
    out = np.zeros((M, V), dtype=np.float64)
    st = lib().oracle_lmhead_logits(_ptr(h), _ptr(w), M, d, V, _ptr(out), nthreads)
    assert st == 0, st
    return out


def walk(base_bits, w1_bits, prev, K: int, *, w2_bits=None, w2q=None, scales=None, seeds=None,
         slot=None, mode: int = GREEDY, temperature: float = 1.0, top_k: int = 0, follow=None,
         tie_tol: float = 1e-3, bf16_eps: float = 1e-4, nthreads: int = 1,
         want_logits: bool = False, want_logits_bf16: bool = False, want_scores: bool = False,
         want_cand: bool = False, base_f64=None) -> WalkResult:
    """base_bits: bf16 [bs, K, V] base logits, or None with base_f64: fp64 [bs, K, V]
    unrounded base logits (the LM-head output)."""
    b64 = _c(base_f64, np.float64)
    base = _c(base_bits, np.uint16) if base_bits is not None else None
    w1 = _c(w1_bits, np.uint16)
    w2 = _c(w2_bits, np.uint16)
    q = _c(w2q, np.int8)
    sc = _c(scales, np.float32)
    pv = _c(prev, np.int32)
    sd = _c(seeds, np.uint64)
    sl = _c(slot, np.int32)
    fo = _c(follow, np.int32)
    bs = pv.shape[0]
    V = (base if base is not None else b64).shape[-1]
    R = w1.shape[1]
    assert (base if base is not None else b64).shape == (bs, K, V), (bs, K, V)
    tokens = np.zeros((bs, K), dtype=np.int32)
    gap = np.zeros((bs, K), dtype=np.float64)
    best = np.zeros((bs, K), dtype=np.float64)
    fcls = np.zeros((bs, K), dtype=np.uint8) if fo is not None else None
    logits = np.zeros((bs, K, V), dtype=np.float64) if want_logits else None
    lbf = np.zeros((bs, K, V), dtype=np.uint16) if want_logits_bf16 else None
    scores = np.zeros((bs, K, V), dtype=np.float64) if want_scores else None
    cand = np.zeros((bs, K, top_k), dtype=np.int32) if (want_cand and top_k > 0) else None
    args = _WalkArgs(
        _ptr(base), _ptr(w1), _ptr(w2), _ptr(q), _ptr(sc), _ptr(pv), _ptr(sd), _ptr(sl),
        V, R, bs, K, mode, temperature, top_k, _ptr(fo), tie_tol, bf16_eps, nthreads,
        _ptr(tokens), _ptr(gap), _ptr(best), _ptr(fcls), _ptr(logits), _ptr(lbf), _ptr(scores),
        _ptr(cand), _ptr(b64))
    st = lib().oracle_walk(C.byref(args))
    return WalkResult(int(st), tokens, gap, best, fcls, logits, lbf, scores, cand)


class _VerifyArgs(C.Structure):
    _fields_ = [
        ("target", C.c_void_p), ("draft", C.c_void_p), ("dtok", C.c_void_p), ("seeds", C.c_void_p),
        ("slot", C.c_void_p), ("V", C.c_int64), ("bs", C.c_int32), ("K", C.c_int32),
        ("temperature", C.c_float), ("accepted", C.c_void_p), ("out_tokens", C.c_void_p),
        ("p_out", C.c_void_p), ("q_out", C.c_void_p), ("u_out", C.c_void_p),
        ("ratio_out", C.c_void_p), ("qd_out", C.c_void_p), ("y_out", C.c_void_p),
        ("gap_out", C.c_void_p), ("score_out", C.c_void_p),
    ]


@dataclass
class VerifyResult:
    status: int
    accepted: np.ndarray      # [bs]
    out_tokens: np.ndarray    # [bs, K+1]
    u: np.ndarray             # [bs, K] acceptance uniforms
    p_d: np.ndarray           # [bs, K] target probability of each draft token
    q_d: np.ndarray           # [bs, K] draft probability of each draft token
    y: np.ndarray             # [bs, K+1] sample of every position (residual, or bonus at K)
    gap: np.ndarray           # [bs, K+1] its top-2 score gap
    p: np.ndarray | None      # [bs, K+1, V]
    q: np.ndarray | None      # [bs, K, V]
    scores: np.ndarray | None  # [bs, K+1, V]


def verify(target_bits, draft_bits, dtok, seeds, temperature: float, *, slot=None,
           want_probs: bool = False) -> VerifyResult:
    """Speculative-sampling verification of the draft tokens (see oracle_verify)."""
    t = _c(target_bits, np.uint16)
    d = _c(draft_bits, np.uint16)
    tk = _c(dtok, np.int32)
    sd = _c(seeds, np.uint64)
    sl = _c(slot, np.int32)
    bs, K1, V = t.shape
    K = K1 - 1
    assert d.shape == (bs, K, V) and tk.shape == (bs, K)
    acc = np.zeros(bs, np.int32)
    out = np.zeros((bs, K + 1), np.int32)
    u = np.zeros((bs, K)); pd = np.zeros((bs, K)); qd = np.zeros((bs, K))
    y = np.zeros((bs, K + 1), np.int32); gap = np.zeros((bs, K + 1))
    p = np.zeros((bs, K + 1, V)) if want_probs else None
    q = np.zeros((bs, K, V)) if want_probs else None
    sc = np.zeros((bs, K + 1, V)) if want_probs else None
    a = _VerifyArgs(_ptr(t), _ptr(d), _ptr(tk), _ptr(sd), _ptr(sl), V, bs, K, temperature,
                    _ptr(acc), _ptr(out), _ptr(p), _ptr(q), _ptr(u), _ptr(pd), _ptr(qd), _ptr(y),
                    _ptr(gap), _ptr(sc))
    st = lib().oracle_verify(C.byref(a))
    return VerifyResult(int(st), acc, out, u, pd, qd, y, gap, p, q, sc)
