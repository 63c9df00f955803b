"""dt_row_topk_static (row log-softmax top-K on a static device scratch) against dt_expand_layer.

The children of an expanded node are the top-K tokens of softmax(row) with their log
probabilities (EAGLE-2 page, §"扩展阶段"); dt_expand_layer writes them into the tree and
dt_row_topk_static returns them directly. Ids must agree exactly, log probabilities within the
tolerance of the float outputs (2e-6 relative, 2e-6 absolute below magnitude 1). Two calls are
issued back to back on one stream before anything is read, so the second call depends on the
first one having left its arrival counters at zero.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t

    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    return t


def _tol_check(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = 2e-6 * np.maximum(1.0, np.abs(ref))
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{what}: {bad.sum()} mismatches, max err {np.abs(got - ref).max()}"


def _tree_children(dt, h, B, F, K, layer):
    t = dt.dt_get_tree(h)
    base = 1 if layer == 1 else 1 + K + (layer - 2) * t["LW"]
    tok = t["token"][:B, base:base + F * K].cpu().numpy().reshape(B * F, K)
    logc = t["logc"][:B, base:base + F * K].cpu().numpy().reshape(B * F, K)
    return tok, logc


@pytest.mark.parametrize("dtype_name,V,K,B,W", [("bf16", 128256, 10, 8, 10), ("f32", 32000, 8, 4, 4),
                                                ("bf16", 4099, 32, 3, 2)])
def test_static_topk_matches_expand(torch, dtype_name, V, K, B, W):
    import dynamic_draft_tree_gb300 as dt

    tdt = torch.bfloat16 if dtype_name == "bf16" else torch.float32
    dtype = dt.DT_BF16 if dtype_name == "bf16" else dt.DT_F32
    g = torch.Generator(device="cuda")
    g.manual_seed(V * 31 + K)
    rows1 = (torch.randn(B, 1, V, generator=g, device="cuda") * 2.0).to(tdt).contiguous()
    rows2 = (torch.randn(B, W, V, generator=g, device="cuda") * 3.0).to(tdt).contiguous()

    # existing path: two layers of the tree
    h = dt.Handle(B, V, K, W, 2, 8, dtype)
    dt.dt_tree_reset(h, torch.arange(B, dtype=torch.int32, device="cuda"))
    dt.dt_expand_layer(h, rows1, 1)
    tok1, logc1 = _tree_children(dt, h, B, 1, K, 1)
    dt.dt_select_frontier(h)
    t = dt.dt_get_tree(h)
    assert int(t["frontier_count"][:B].min()) == W
    dt.dt_expand_layer(h, rows2, W)
    tok2, logc2 = _tree_children(dt, h, B, W, K, 2)
    assert dt.dt_get_status(h) == 0
    h.close()

    # static-scratch path: two calls in a row, nothing read in between
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp1 = torch.empty(B, K, dtype=torch.float32, device="cuda")
    id1 = torch.empty(B, K, dtype=torch.int32, device="cuda")
    lp2 = torch.empty(B * W, K, dtype=torch.float32, device="cuda")
    id2 = torch.empty(B * W, K, dtype=torch.int32, device="cuda")
    dt.dt_row_topk_static(rows1.reshape(B, V), K, lp1, id1, status=status)
    dt.dt_row_topk_static(rows2.reshape(B * W, V), K, lp2, id2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    np.testing.assert_array_equal(id1.cpu().numpy(), tok1)
    np.testing.assert_array_equal(id2.cpu().numpy(), tok2)
    _tol_check(lp1.cpu().numpy(), logc1, "layer-1 log p")
    _tol_check(lp2.cpu().numpy(), logc2, "layer-2 log p")

    # the same two calls again give the same results bit for bit
    lp1b, id1b = torch.empty_like(lp1), torch.empty_like(id1)
    lp2b, id2b = torch.empty_like(lp2), torch.empty_like(id2)
    dt.dt_row_topk_static(rows1.reshape(B, V), K, lp1b, id1b, status=status)
    dt.dt_row_topk_static(rows2.reshape(B * W, V), K, lp2b, id2b, status=status)
    torch.cuda.synchronize()
    assert torch.equal(id1b, id1) and torch.equal(id2b, id2)
    assert torch.equal(lp1b, lp1) and torch.equal(lp2b, lp2)


def test_static_topk_rejects_too_many_rows(torch):
    import dynamic_draft_tree_gb300 as dt

    V, K = 1000, 4
    x = torch.zeros(1025, V, dtype=torch.bfloat16, device="cuda")
    lp = torch.empty(1025, K, dtype=torch.float32, device="cuda")
    ids = torch.empty(1025, K, dtype=torch.int32, device="cuda")
    with pytest.raises(dt.DtError, match="static scratch"):
        dt.dt_row_topk_static(x, K, lp, ids)
    # the largest allowed call still runs and keeps the all-equal tie rule (lowest ids first)
    dt.dt_row_topk_static(x[:1024], K, lp[:1024], ids[:1024])
    torch.cuda.synchronize()
    assert (ids[:1024].cpu().numpy() == np.arange(K, dtype=np.int32)).all()
    _tol_check(lp[:1024].cpu().numpy(), np.full((1024, K), -np.log(V)), "uniform log p")
