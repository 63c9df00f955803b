"""Pins of the accepted-path KV compaction oracle (``oracle.kv``), CPU only.

What fixes it (not the oracle itself): a plain token-by-token decoder. Each temporary KV row of a
verified tree is made a deterministic function of the token sequence it was computed for (the
context plus the tokens on the root-to-position path), as a transformer's KV row is a function of
the token and its prefix. After a round, the rows appended to the cache must be exactly the rows a
sequential decoder would have written for the committed tokens (the root, then the accepted tokens),
in order: right rows, right order, nothing from rejected branches, nothing overwritten.
"""
import hashlib

import numpy as np
import pytest

from oracle.kv import commit_kv
from oracle.tree import OracleTree, build_meta, packed_row_offsets
from oracle.verify import verify_greedy

ROW = 16  # bytes of a synthetic KV row


def kv_row(seq):
    """A token sequence's KV row: 16 bytes of its SHA-256 (a stand-in for a forward's K/V)."""
    return np.frombuffer(hashlib.sha256(np.asarray(seq, np.int64).tobytes()).digest()[:ROW], np.uint8)


def random_round(seed, B=3, V=12, K=3, W=2, D=3, m=8):
    rng = np.random.default_rng(seed)
    roots = rng.integers(0, V, B)
    t = OracleTree(B, K, W, D, roots)
    for d in range(1, D + 1):
        t.expand_layer(lambda b, f: rng.normal(0, 2, V))
        if d < D:
            t.select_frontier(W)
    m_cap = int(np.max(m))
    sel = t.rerank(m, m_cap)
    meta = build_meta(t, sel, np.zeros(B, np.int64), P=m_cap + 1, D_path=D + 1)
    rows = rng.normal(0, 2, (B, m_cap + 1, V))  # target rows: argmax decides the accepted path
    acc, path, bonus = verify_greedy(meta, lambda b, i: rows[b, i])
    return t, meta, acc, path, rng


def rng_m(seed):
    """Verify counts: 8 for every request, or per-request counts (ragged requests) for the packed cases."""
    return 8 if seed < 6 else [2 + seed % 3, 8, 1 + seed % 5]


def path_tokens(meta, b, i):
    """Tokens from the root to position i (root first)."""
    out = []
    while i >= 0:
        out.append(int(meta["tokens"][b, i]))
        i = int(meta["parents"][b, i]) if i > 0 else -1
    return out[::-1]


@pytest.mark.parametrize("seed,packed", [(s, False) for s in range(6)] + [(s, True) for s in range(6, 10)])
def test_commit_equals_sequential_decode(seed, packed):
    """Padded temporary rows ([B][P]), or padding-free ones (request b's used positions at
    row_off[b] + i, one request after the other, nothing in between)."""
    t, meta, acc, path, rng = random_round(seed, m=rng_m(seed))
    B, P = meta["tokens"].shape
    ctx = [list(rng.integers(0, 12, rng.integers(0, 5))) for _ in range(B)]  # already committed tokens
    tmp = np.zeros((B, P, ROW), np.uint8)
    for b in range(B):
        for i in range(int(meta["n_pos"][b])):
            tmp[b, i] = kv_row(ctx[b] + path_tokens(meta, b, i))
    row_off = None
    if packed:
        row_off = packed_row_offsets(meta["n_pos"])
        tmp = np.concatenate([tmp[b, :int(meta["n_pos"][b])] for b in range(B)])  # used rows, in order
        assert tmp.shape[0] == row_off[B] and len(set(meta["n_pos"].tolist())) > 1  # ragged
    L = 16
    cache = np.zeros((B, L, ROW), np.uint8)
    cache_len = np.array([len(c) for c in ctx], np.int64)
    for b in range(B):
        for j in range(len(ctx[b])):
            cache[b, j] = kv_row(ctx[b][:j + 1])
    before = cache.copy()
    refused = commit_kv(tmp, cache, cache_len, acc, path, row_off=row_off)
    assert refused == []
    for b in range(B):
        committed = [int(meta["tokens"][b, 0])] + [int(meta["tokens"][b, p]) for p in path[b, 1:acc[b] + 1]]
        seq = ctx[b] + committed
        # a sequential decoder writes row j for the prefix of length j + 1
        assert int(cache_len[b]) == len(seq)
        for j in range(len(seq)):
            assert np.array_equal(cache[b, j], kv_row(seq[:j + 1])), (b, j)
        assert np.array_equal(cache[b, len(seq):], before[b, len(seq):])  # nothing past the new end


def test_no_acceptance_commits_the_root_only():
    tmp = np.arange(2 * 4 * ROW, dtype=np.uint8).reshape(2, 4, ROW)
    cache = np.zeros((2, 5, ROW), np.uint8)
    cache_len = np.array([0, 3])
    path = np.full((2, 3), -1)
    path[:, 0] = 0
    commit_kv(tmp, cache, cache_len, np.array([0, 0]), path)
    assert list(cache_len) == [1, 4]
    assert np.array_equal(cache[0, 0], tmp[0, 0]) and np.array_equal(cache[1, 3], tmp[1, 0])
    assert not cache[0, 1:].any() and not cache[1, 4:].any()


def test_full_cache_is_refused_and_left_alone():
    tmp = np.ones((2, 4, ROW), np.uint8)
    cache = np.zeros((2, 5, ROW), np.uint8)
    cache_len = np.array([3, 1])
    path = np.array([[0, 1, 2], [0, 2, -1]])
    refused = commit_kv(tmp, cache, cache_len, np.array([2, 1]), path)  # 3 rows do not fit after 3
    assert refused == [0]
    assert list(cache_len) == [3, 3] and not cache[0].any()
    assert cache[1, 1:3].all() and not cache[1, 3:].any()
