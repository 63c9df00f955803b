"""Accepted-path KV compaction on the GPU vs the oracle (``oracle.kv``), through the C ABI.

The accepted lengths and paths come from real GPU rounds (which the round parity tests compare with
the oracle); the KV rows are random bytes. Every committed row and every cache length must be equal.
"""
import numpy as np
import pytest

from synth.workloads import with_sizes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t

    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    return t


def _round(torch, name, over, rnd=0, packed=False):
    import harness

    w = with_sizes(name, **over)
    gr = harness.GpuRound(w, packed=packed)
    attempts = np.zeros(w["B"], np.int64)
    roots = harness.root_tokens(w, harness.salts_of(w, rnd, attempts))
    gr.round(rnd, attempts, roots)
    return gr


@pytest.mark.parametrize("name,over,row_bytes", [("cast", dict(V=12007), 131072), ("vicuna", dict(V=4096, T=1), 4096),
                                                 ("stress", dict(V=3001, B=8, D=5), 272)])
def test_commit_kv_matches_oracle(torch, name, over, row_bytes):
    import dynamic_draft_tree_gb300 as dt
    from oracle.kv import commit_kv

    gr = _round(torch, name, over)
    run = gr.run
    B, P = run.meta.tokens.shape
    L = 3 * P
    rng = np.random.default_rng(row_bytes + B)
    tmp = rng.integers(0, 256, (B, P, row_bytes), dtype=np.uint8)
    cache = rng.integers(0, 256, (B, L, row_bytes), dtype=np.uint8)
    cache_len = rng.integers(0, P, B).astype(np.int32)
    d_tmp, d_cache = torch.from_numpy(tmp).cuda(), torch.from_numpy(cache).cuda()
    d_len = torch.from_numpy(cache_len).cuda()
    dt.dt_commit_kv(run.h, d_tmp, d_cache, d_len, run.accept_len, run.accept_path)
    assert dt.dt_get_status(run.h) == 0
    acc = run.accept_len.cpu().numpy()
    path = run.accept_path.cpu().numpy()
    want_len = cache_len.astype(np.int64).copy()
    refused = commit_kv(tmp, cache, want_len, acc, path)
    assert refused == []
    np.testing.assert_array_equal(d_len.cpu().numpy(), want_len)
    np.testing.assert_array_equal(d_cache.cpu().numpy(), cache)
    run.h.close()


def test_commit_kv_full_cache_is_refused(torch):
    import dynamic_draft_tree_gb300 as dt
    from oracle.kv import commit_kv

    gr = _round(torch, "pr1", dict(V=4099, B=1, m=8))
    run = gr.run
    P = run.meta.tokens.shape[1]
    row = 64
    tmp = np.arange(P * row, dtype=np.uint8).reshape(1, P, row)
    cache = np.zeros((1, 4, row), np.uint8)
    acc = run.accept_len.cpu().numpy()
    cache_len = np.array([4 - int(acc[0])], np.int32)  # one row short of room for accept_len + 1 rows
    d_cache, d_len = torch.from_numpy(cache).cuda(), torch.from_numpy(cache_len).cuda()
    dt.dt_commit_kv(run.h, torch.from_numpy(tmp).cuda(), d_cache, d_len, run.accept_len, run.accept_path)
    assert dt.dt_get_status(run.h) & dt.DT_DEV_KV_FULL
    want = cache_len.astype(np.int64).copy()
    assert commit_kv(tmp, cache, want, acc, run.accept_path.cpu().numpy()) == [0]
    assert d_len.cpu().numpy()[0] == want[0] == cache_len[0]
    assert not d_cache.cpu().numpy().any()
    run.h.close()


def test_commit_kv_packed_matches_oracle(torch):
    """Padding-free temporary KV (the layout of DT_VERIFY_PACKED): request b's positions at rows
    row_off[b] + i of one buffer, row_off from the tree metadata; per-request CAST gives ragged trees."""
    import dynamic_draft_tree_gb300 as dt
    from oracle.kv import commit_kv
    from synth.workloads import WORKLOADS

    gr = _round(torch, "cast", dict(V=12007, cast=dict(WORKLOADS["cast"]["cast"], per_request=True)), packed=True)
    run = gr.run
    B, P = run.meta.tokens.shape
    row_off = run.meta.row_off.cpu().numpy()
    rows = int(row_off[B])
    row_bytes = 4096
    rng = np.random.default_rng(7)
    tmp = rng.integers(0, 256, (rows, row_bytes), dtype=np.uint8)
    cache = rng.integers(0, 256, (B, 2 * P, row_bytes), dtype=np.uint8)
    cache_len = rng.integers(0, P, B).astype(np.int32)
    d_cache, d_len = torch.from_numpy(cache).cuda(), torch.from_numpy(cache_len).cuda()
    dt.dt_commit_kv(run.h, torch.from_numpy(tmp).cuda(), d_cache, d_len, run.accept_len, run.accept_path,
                    row_off=run.meta.row_off, P=P)
    assert dt.dt_get_status(run.h) == 0
    want_len = cache_len.astype(np.int64).copy()
    assert commit_kv(tmp, cache, want_len, run.accept_len.cpu().numpy(), run.accept_path.cpu().numpy(),
                     row_off=row_off) == []
    np.testing.assert_array_equal(d_len.cpu().numpy(), want_len)
    np.testing.assert_array_equal(d_cache.cpu().numpy(), cache)
    run.h.close()
