"""The merge step of a vocabulary-sharded walk, on two gloo ranks (CPU).

In a walk sharded over the vocabulary, rank r holds W2 rows [v0_r, v1_r) and, at every
draft position, scores only its shard. The ranks then agree on each request row's token
with ONE 8-byte all-reduce-max per row: the word packs the orderable 32-bit key of the
rank's best score in the high half and the complement of its (global) vocabulary index
in the low half, so the integer maximum is the largest score and, among equal scores,
the smallest index -- torch.argmax order across shard boundaries, with the first NaN
winning. The all-reduce is also the step's barrier: no rank gathers the next embedding
before it has the winner.

The packing here is restated independently of the GPU code (numpy on the host). The
check: for random and hand-built rows (ties across the shard boundary, NaN in either
shard, -0 against +0, all -inf), the merged word decodes to torch.argmax of the whole
row. Signed 64-bit all-reduce keeps the unsigned order after flipping the top bit.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

TOP = np.uint64(1) << np.uint64(63)


def order_key(x: np.ndarray) -> np.ndarray:
    """Monotone uint32 key of fp32 scores: NaN above every number, -0 equal to +0."""
    u = x.astype(np.float32).view(np.uint32).copy()
    nan = np.isnan(x)
    u[(u & 0x7FFFFFFF) == 0] = 0
    neg = (u & 0x80000000) != 0
    key = np.where(neg, ~u, u | np.uint32(0x80000000)).astype(np.uint32)
    key[nan] = 0xFFFFFFFF
    return key


def shard_word(scores: np.ndarray, v0: int) -> np.ndarray:
    """Per row: max over the shard of (key << 32 | (2^32 - 1 - global index))."""
    key = order_key(scores).astype(np.uint64)
    idx = (np.arange(scores.shape[1], dtype=np.uint64) + np.uint64(v0))
    words = (key << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - idx)
    return words.max(axis=1)


def unpack(word: np.ndarray) -> np.ndarray:
    return (np.uint64(0xFFFFFFFF) - (word & np.uint64(0xFFFFFFFF))).astype(np.int64)


def rows_under_test(V: int) -> np.ndarray:
    g = np.random.default_rng(3)
    rows = [g.normal(0, 3, V).astype(np.float32) for _ in range(6)]
    half = V // 2
    r = np.full(V, -5.0, np.float32); r[half - 1] = r[half + 2] = 7.0; rows.append(r)   # tie across shards
    r = np.full(V, -5.0, np.float32); r[half + 3] = np.nan; r[2] = 9.0; rows.append(r)   # NaN in shard 1
    r = np.full(V, -5.0, np.float32); r[1] = np.nan; r[half + 1] = np.nan; rows.append(r)  # first NaN wins
    r = np.full(V, -5.0, np.float32); r[half] = 0.0; r[3] = -0.0; rows.append(r)         # -0 == +0
    rows.append(np.full(V, -np.inf, np.float32))                                        # all -inf -> 0
    return np.stack(rows)


def _rank(rank: int, world: int, port: int, V: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    scores = rows_under_test(V)
    v0, v1 = rank * V // world, (rank + 1) * V // world
    word = shard_word(scores[:, v0:v1], v0)
    t = torch.from_numpy((word ^ TOP).view(np.int64).copy())  # unsigned order in signed ints
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    merged = t.numpy().view(np.uint64) ^ TOP
    out[rank] = unpack(merged).tolist()
    dist.destroy_process_group()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("V", [10, 1001])
def test_two_rank_merge_equals_whole_row_argmax(V):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, V, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    want = torch.argmax(torch.from_numpy(rows_under_test(V)), dim=1).numpy()
    for r in range(2):
        np.testing.assert_array_equal(np.array(out[r]), want)


def test_packing_matches_argmax_without_sharding():
    """One shard holding everything: the packed maximum is torch.argmax."""
    s = rows_under_test(64)
    np.testing.assert_array_equal(unpack(shard_word(s, 0)), torch.argmax(torch.from_numpy(s), dim=1).numpy())
