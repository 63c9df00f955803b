"""GPU path vs the fp64 oracle, element by element, through the C ABI (needs a GB300)."""
import numpy as np
import pytest

import synth
from synth.workloads import with_sizes, spec_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t

    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    return t


# ----------------------------------------------------------------- host-row gather ----
def test_host_row_gather_matches_copies(torch):
    """The end-to-end timing's host -> device gather kernel moves exactly the bytes of its spans: aligned
    and unaligned spans, spans shorter and longer than one work item; bytes outside every span stay."""
    host = torch.from_numpy(np.random.default_rng(5).integers(0, 256, 1 << 21, dtype=np.uint8)).pin_memory()
    src = synth.host_device_ptr(host)
    if src is None:
        pytest.skip("pinned host memory is not mapped for the device")
    dev = torch.zeros(1 << 21, dtype=torch.uint8, device="cuda")
    cuts = [(0, 0, 256512 * 3), (1 << 20, 1 << 20, 64 * 1024 + 16), (7, 800000, 1000), (1900001, 1900003, 77),
            (1950000, 1960000, 16)]
    spans = torch.tensor([(src + a, dev.data_ptr() + b, n) for a, b, n in cuts], dtype=torch.int64,
                         device="cuda")
    for blocks in (1, 3, 32):
        dev.zero_()
        synth.gather_spans_gpu(torch, spans, blocks)
        torch.cuda.synchronize()
        want = torch.zeros_like(host)
        for a, b, n in cuts:
            want[b:b + n] = host[a:a + n]
        assert torch.equal(dev.cpu(), want), blocks


# ----------------------------------------------------------------- generator ----
@pytest.mark.parametrize("name,over", [("pr1", dict(V=4099)), ("vicuna", dict(V=32000)),
                                       ("cast", dict(V=128256)), ("stress", dict(V=5003, B=6))])
def test_device_generator_matches_host_bitwise(torch, name, over):
    w = with_sizes(name, **over)
    spec = spec_for(w)
    rng = np.random.default_rng(1)
    B, F = w["B"], 3
    ctx = rng.integers(-1, w["V"], B * F).astype(np.int32)
    depth = rng.integers(0, 9, B * F).astype(np.int32)
    for stream in (synth.DRAFT, synth.TARGET):
        host = np.zeros((B * F, w["V"]), spec.np_dtype)
        for b in range(B):
            host[b * F:(b + 1) * F] = synth.gen_rows_cpu(spec, 7, 3, stream, ctx[b * F:(b + 1) * F],
                                                         depth[b * F:(b + 1) * F], 1, F, b0=b)
        dt = torch.int16 if spec.dtype == synth.BF16 else torch.float32
        dev = torch.zeros((B * F, w["V"]), dtype=dt, device="cuda")
        synth.gen_rows_gpu(torch, spec, 7, 3, stream, torch.from_numpy(ctx).cuda(), dev, w["V"],
                           depth_dev=torch.from_numpy(depth).cuda(), depth_add=1, rows_per_b=F)
        got = dev.cpu().numpy().view(spec.np_dtype)
        assert np.array_equal(got, host)


# ------------------------------------------------------------ single layer ----
def _expand_case(torch, V, K, B, dtype, rows_fn, F=1, W=None):
    import dynamic_draft_tree_gb300 as dt
    from oracle.tree import OracleTree

    W = W or max(F, 1)
    h = dt.Handle(B, V, K, W, 2, 8, dtype)
    roots = np.arange(B, dtype=np.int32) % V
    dt.dt_tree_reset(h, torch.from_numpy(roots).cuda())
    x = rows_fn(B, V)  # float64 [B][V], exactly representable in dtype
    tdt = torch.bfloat16 if dtype == dt.DT_BF16 else torch.float32
    logits = torch.from_numpy(x).to(tdt).cuda().reshape(B, 1, V).contiguous()
    dt.dt_expand_layer(h, logits, 1)
    assert dt.dt_get_status(h) == 0
    ot = OracleTree(B, K, W, 2, roots)
    ot.expand_layer(x.reshape(B, 1, V))
    t = dt.dt_get_tree(h)
    from harness import assert_close

    tok = t["token"][:B].cpu().numpy()
    np.testing.assert_array_equal(tok, ot.token)
    valid = ot.token >= 0
    np.testing.assert_array_equal(t["parent"][:B].cpu().numpy()[valid], ot.parent[valid])
    assert_close(t["logc"][:B].cpu().numpy()[valid], ot.logc[valid], "logc")
    assert_close(t["value"][:B].cpu().numpy()[valid], ot.value[valid], "value")
    order = t["layer_order"][:B, 1, :K].cpu().numpy()
    for b in range(B):
        np.testing.assert_array_equal(order[b], ot.layer_sorted[b][1])
    h.close()


def _bf16_exact(x):
    import torch as t

    return t.from_numpy(x).to(t.bfloat16).to(t.float64).numpy()


@pytest.mark.parametrize("V,K,B", [(1000, 10, 3), (1001, 4, 2), (4096 * 3 + 5, 32, 2), (32000, 1, 4),
                                   (128256, 10, 8), (151936, 8, 3), (17, 17, 1)])
def test_expand_layer_bf16(torch, V, K, B):
    rng = np.random.default_rng(V + K)
    _expand_case(torch, V, K, B, 0, lambda B, V: _bf16_exact(rng.normal(0, 2, (B, V))))


@pytest.mark.parametrize("V,K,B", [(1000, 8, 2), (128256, 8, 4), (3, 2, 1)])
def test_expand_layer_f32(torch, V, K, B):
    rng = np.random.default_rng(V * 7 + K)
    _expand_case(torch, V, K, B, 1, lambda B, V: rng.normal(0, 2, (B, V)).astype(np.float32).astype(np.float64))


def test_expand_layer_all_equal_and_neg_inf(torch):
    _expand_case(torch, 5000, 10, 2, 0, lambda B, V: np.zeros((B, V)))
    def rows(B, V):
        x = np.full((B, V), -np.inf)
        x[:, ::97] = _bf16_exact(np.random.default_rng(3).normal(0, 1, (B, x[:, ::97].shape[1])))
        return x
    _expand_case(torch, 6000, 12, 2, 0, rows)


def test_expand_layer_nan_sets_status(torch):
    import dynamic_draft_tree_gb300 as dt

    h = dt.Handle(1, 3000, 4, 1, 2, 8, dt.DT_F32)
    dt.dt_tree_reset(h, torch.zeros(1, dtype=torch.int32, device="cuda"))
    x = torch.zeros((1, 1, 3000), dtype=torch.float32, device="cuda")
    x[0, 0, 1234] = float("nan")
    dt.dt_expand_layer(h, x, 1)
    assert dt.dt_get_status(h) & dt.DT_DEV_BAD_LOGITS
    h.close()


def test_timeout_path_reports_status(torch):
    import dynamic_draft_tree_gb300 as dt

    h = dt.Handle(1, 70000, 4, 1, 2, 8, dt.DT_BF16, flags=dt.DT_FLAG_TEST_TIMEOUT)
    dt.dt_tree_reset(h, torch.zeros(1, dtype=torch.int32, device="cuda"))
    x = torch.zeros((1, 1, 70000), dtype=torch.bfloat16, device="cuda")
    dt.dt_expand_layer(h, x, 1)
    assert dt.dt_get_status(h) & dt.DT_DEV_TIMEOUT
    dt.dt_clear_status(h)
    assert dt.dt_get_status(h) == 0
    h.close()


def test_host_argument_errors(torch):
    import dynamic_draft_tree_gb300 as dt

    h = dt.Handle(2, 1000, 4, 2, 3, 9, dt.DT_BF16)
    x = torch.zeros((2, 2, 1000), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dt.DtError):
        dt.dt_expand_layer(h, x, 1)                     # no tree yet
    dt.dt_tree_reset(h, torch.zeros(2, dtype=torch.int32, device="cuda"))
    with pytest.raises(dt.DtError):
        dt.dt_expand_layer(h, x, 3)                     # F > W
    # right after the reset the newest layer is layer 0 = {root}: the layer-1 frontier is the root
    ft = torch.full((2, 2), 7, dtype=torch.int32, device="cuda")
    dt.dt_tree_reset(h, torch.tensor([5, 9], dtype=torch.int32, device="cuda"))
    dt.dt_select_frontier(h, frontier_token=ft)
    assert ft.cpu().tolist() == [[5, -1], [9, -1]]
    t = dt.dt_get_tree(h)
    assert t["frontier"][:2].cpu().tolist() == [[0, -1], [0, -1]]
    assert t["frontier_count"][:2].cpu().tolist() == [1, 1]
    with pytest.raises(dt.DtError):
        dt.dt_expand_layer(h, x, 1, ld=999)             # ld < V
    with pytest.raises(dt.DtError):
        dt.dt_tree_reset(h, torch.zeros(3, dtype=torch.int32, device="cuda"))  # B > B_max
    # the entry points of the extensions refuse bad arguments on the host, before any launch
    blk = torch.zeros((2, 4, 1000), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dt.DtError):
        dt.dt_block_expand(h, blk, 4)                   # L > D_max
    dt.dt_expand_layer(h, x, 1)
    with pytest.raises(dt.DtError):
        dt.dt_block_expand(h, blk, 2)                   # not right after a reset
    meta = dt.Meta(2, 9, 4)
    i32 = dict(dtype=torch.int32, device="cuda")
    out = [torch.zeros(2, **i32), torch.zeros((2, 4), **i32), torch.zeros(2, **i32)]
    tgt = torch.zeros((2, 9, 1000), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dt.DtError):                    # sampled verify: mode is 0 or DT_VERIFY_PACKED only
        lib_mode = dt.lib.dt_verify_sampled(h.h, dt.ctypes.byref(meta.c), tgt.data_ptr(), 1000, dt.DT_SAMPLE,
                                            tgt.data_ptr(), 1000, 0, 0, out[0].data_ptr(), out[1].data_ptr(),
                                            out[2].data_ptr(), None)
        dt.check(lib_mode)
    tpl = dt.Template([-1, 0], [0, 0], anchor=dt.DT_ANCHOR_TAIL)
    M = torch.full((2, 1000, 8), -1, **i32)
    with pytest.raises(dt.DtError):                    # a tail anchor needs the kept nodes
        dt.dt_graft_retrieve(h, M, tpl, 4, torch.zeros((2, 4), **i32), torch.zeros((2, 4), **i32), out[0])
    kv = torch.zeros((2, 9, 24), dtype=torch.uint8, device="cuda")   # 24-byte rows: not a multiple of 16
    cache = torch.zeros((2, 16, 24), dtype=torch.uint8, device="cuda")
    with pytest.raises(dt.DtError):
        dt.dt_commit_kv(h, kv, cache, out[0], out[0], out[1])
    h.close()


# --------------------------------------------------------------- full rounds ----
SMALL = [("pr1", dict(V=4099)), ("pr1", dict(V=32000)), ("vicuna", dict(V=32000)),
         ("cast", dict(V=20011)), ("graft", dict(V=9001, B=4)), ("stress", dict(V=7001, B=6, D=5)),
         ("vicuna", dict(V=8192, T=1)), ("pr1", dict(V=3001, K=1, k=1, m=1)), ("pr1", dict(V=3001, m=60))]


def _run_rounds(torch, w, rounds, label=None, compare_from=0, chain_roots=True, packed=False, on_ref=None):
    """GPU rounds against the oracle's, element by element; ``rounds`` is a count or the list of
    round indices. Graft chains its rounds: M comes from the previous round, and so does the next
    root (its bonus token) unless ``chain_roots`` is false (then every round drafts from the same
    root tokens). Rounds before ``compare_from`` run on both sides (warm-up) but are compared only
    through M. ``packed``: padding-free target rows (DT_VERIFY_PACKED). ``on_ref(ref)`` is called with
    every compared oracle round. Logs the seed redraws under ``label``."""
    import harness
    from dynamic_draft_tree_gb300 import dt_get_status

    gr = harness.GpuRound(w, packed=packed)
    M = None
    if w["policy"] == "graft":
        M = np.full((w["B"], w["V"], 8), -1, np.int64)
    roots = None
    redrawn = hit = 0
    idx = list(range(rounds)) if isinstance(rounds, int) else list(rounds)
    for n, rnd in enumerate(idx):
        ref, attempts, rej = harness.oracle_round(w, rnd, roots=roots, M=M)
        redrawn += rej
        hit += rej > 0
        gr.round(rnd, attempts, ref["roots"])
        assert dt_get_status(gr.run.h) == 0
        if n >= compare_from:
            harness.compare_round(gr, ref)
            if on_ref is not None:
                on_ref(ref)
        elif w["policy"] == "graft":  # warm-up: the refreshed M must still agree
            np.testing.assert_array_equal(gr.M.cpu().numpy(), ref["M"], err_msg="M after warm-up round")
        if w["policy"] == "graft":
            M = ref["M"]
            roots = ref["bonus"].astype(np.int32) if chain_roots else ref["roots"]
    gr.run.h.close()
    harness.log_redraws(label or f"{w['policy']} B={w['B']} V={w['V']} T={w['T']}", len(idx) - compare_from,
                        redrawn, hit)
    return redrawn


@pytest.mark.parametrize("name,over", SMALL)
def test_round_parity_small(torch, name, over):
    w = with_sizes(name, **over)
    if w["m"] > 1 and name == "pr1" and over.get("m") == 60:
        w["D"] = 6
    _run_rounds(torch, w, 3, label=f"small {name} {over}")


# Stochastic verify (T = 1): 24 rounds each of a Vicuna-shaped and a stress-shaped batch at reduced
# V, so that a few hundred acceptance tests and residual draws are compared (EAGLE-2 page,
# §无损性为什么没有被动态树破坏).
# The stress shape's low-entropy requests also reject children that hold most of a row's mass, which
# sends the device walk through its exact residual recomputation: that branch must be among the
# compared decisions.
@pytest.mark.parametrize("name,over", [("vicuna", dict(V=4096, T=1)), ("stress", dict(V=3001, B=8, D=5))])
def test_round_parity_sampling_many_rounds(torch, name, over):
    import harness

    w = with_sizes(name, **over)
    events = []
    _run_rounds(torch, w, 24, label=f"T=1 {name} {over}",
                on_ref=lambda ref: events.append(harness.exact_residual_events(w, ref)))
    if name == "stress":
        assert sum(events) > 0, "no exact residual recomputation among the compared rounds"


def test_round_parity_graft_sampling(torch):
    """Graft with the stochastic verify (T = 1): the M refresh reads the top-8 of every verified row
    whatever the acceptance rule (Graft page step (3))."""
    w = with_sizes("graft", V=2003, B=4, T=1)
    _run_rounds(torch, w, 8, label="graft T=1", chain_roots=False)


def test_round_parity_graft_after_warmup(torch):
    """Graft page step (3): every round drafts again from the same root tokens, so the refresh of M
    from the verified positions fills the rows the template reads: after five warm-up rounds
    (about 80 % of the grafted nodes are real tokens by then, all of them two rounds later) eight
    more rounds run with accepted paths through grafted nodes. Every round is compared in full."""
    w = with_sizes("graft", V=2003, B=4)
    _run_rounds(torch, w, 13, label="graft, 5 warm-up + 8 rounds, filled M", chain_roots=False)


def test_round_parity_cast_table_rows(torch):
    """CAST page §关键设计 1: rounds whose prefix lengths n0 = 512 (1 + r mod 16) select eight
    different cost-table rows (r = 0, 2, ..., 14 -> rows 1, 3, ..., 15), plus the rows the growing
    context reaches within each round."""
    w = with_sizes("cast", V=12007)
    _run_rounds(torch, w, range(0, 16, 2), label="cast table rows 1..15")


def _cast_per_request(**over):
    from synth.workloads import WORKLOADS

    return with_sizes("cast", cast=dict(WORKLOADS["cast"]["cast"], per_request=True), **over)


@pytest.mark.parametrize("over,rounds", [(dict(V=12007), range(0, 16, 2)), ({}, 2)])
def test_round_parity_cast_per_request(torch, over, rounds):
    """CAST page §局限与展望: the per-request rule (each request's own widths, stop and verify count)
    against the oracle's, at reduced and at full size."""
    w = _cast_per_request(**over)
    _run_rounds(torch, w, rounds, label=f"cast per request {over}")


@pytest.mark.parametrize("name,over,rounds", [
    ("cast_req", dict(V=12007), range(0, 8, 2)),  # ragged trees: per-request widths, stops and m
    ("cast_req", {}, 1),                           # full size
    ("graft", dict(V=2003, B=4), 6),               # the top-8 refresh reads packed rows
    ("stress", dict(V=3001, B=8, D=5), 8),         # T = 1: sampled walk and bonus draw on packed rows
    ("vicuna", dict(V=4096, T=1), 4)])
def test_round_parity_packed_rows(torch, name, over, rounds):
    """CAST page §局限与展望 (padded batches are a limit): the verify reads request b's rows at
    row_off[b] + i of a padding-free buffer (rows past the used ones hold NaN, so a stray read sets
    a status bit); every output equals the oracle's, and row_off equals its prefix sums."""
    w = _cast_per_request(**over) if name == "cast_req" else with_sizes(name, **over)
    _run_rounds(torch, w, rounds, label=f"packed rows {name} {over}", packed=True,
                chain_roots=name != "graft")


def test_cast_per_request_fused_calls_equal_separate_calls(torch):
    import harness

    w = _cast_per_request(V=32000)
    outs = []
    for fused in (True, False):
        gr = harness.GpuRound(w, fused=fused)
        res = []
        for rnd in range(3):
            attempts = np.zeros(w["B"], np.int64)
            roots = harness.root_tokens(w, harness.salts_of(w, rnd, attempts))
            gr.round(rnd, attempts, roots)
            t = harness.tree_numpy(gr.run.h)
            res.append((t["token"].copy(), t["value"].copy(), gr.run.selected.cpu().numpy().copy(),
                        gr.run.m_dev.cpu().numpy().copy(), gr.run.width.cpu().numpy().copy(),
                        gr.run.accept_len.cpu().numpy().copy(), gr.run.bonus.cpu().numpy().copy()))
        outs.append(res)
        gr.run.h.close()
    for ra, rb in zip(*outs):
        for a, b in zip(ra, rb):
            np.testing.assert_array_equal(a, b)


def test_sampling_first_token_law_on_gpu(torch):
    """Monte Carlo on the GPU alone: the first token a T = 1 round emits (the accepted child, or the
    bonus if every child of the root is rejected) is distributed as the target's root row,
    whatever the tree (EAGLE-2 page, §无损性为什么没有被动态树破坏). V = 8, a draft row unlike the
    target, 1024 requests per round (independent Philox counters per request), 12 rounds; chi-square
    with 7 degrees of freedom against softmax(target root row)."""
    import dynamic_draft_tree_gb300 as dt
    from dynamic_draft_tree_gb300.rounds import RoundRunner

    V, B, K, k, D, m = 8, 1024, 3, 2, 2, 5
    P, D_path = m + 1, D + 1
    draft_row = torch.tensor([2.0, 1.5, 1.0, 0.2, -0.5, -1.0, 0.1, 0.0])
    target_root = torch.tensor([0.3, 1.2, -0.4, 0.8, 0.0, -1.5, 0.5, 0.9])
    other = torch.tensor([0.0, 0.5, 1.0, -0.5, 0.2, 0.1, -0.2, 0.3])
    run = RoundRunner("eagle", B, V, K, k, D, P, D_path, m, dt.DT_F32, T=1)
    draft = draft_row.repeat(B, k, 1).cuda().contiguous()
    target = other.repeat(B, P, 1).clone()
    target[:, 0] = target_root
    target = target.cuda().contiguous()
    roots = torch.zeros(B, dtype=torch.int32, device="cuda")
    counts = np.zeros(V, np.int64)
    for rnd in range(12):
        run.run(roots, lambda d, ft: draft, lambda meta: target, seed=99, rnd=rnd << 8)
        assert dt.dt_get_status(run.h) == 0
        acc = run.accept_len.cpu().numpy()
        path = run.accept_path.cpu().numpy()
        tok = run.meta.tokens.cpu().numpy()
        bonus = run.bonus.cpu().numpy()
        first = np.where(acc >= 1, tok[np.arange(B), np.maximum(path[:, 1], 0)], bonus)
        counts += np.bincount(first, minlength=V)
    run.h.close()
    p = torch.softmax(target_root.double(), 0).numpy()
    n = counts.sum()
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert n == 12 * B
    assert chi2 < 29.9, (chi2, counts, n * p)   # 7 dof: P(chi2 > 29.9) ~ 1e-4


def test_full_size_round_is_deterministic(torch):
    """The same CAST round (B=8, V=128256) run twice gives bit-identical trees and outputs."""
    import harness

    w = with_sizes("cast")
    gr = harness.GpuRound(w)
    attempts = np.zeros(w["B"], np.int64)
    roots = harness.root_tokens(w, harness.salts_of(w, 0, attempts))
    outs = []
    for _ in range(3):
        gr.round(0, attempts, roots)
        t = harness.tree_numpy(gr.run.h)
        outs.append((t["token"].copy(), t["value"].copy(), gr.run.meta.numpy()["tokens"].copy(),
                     gr.run.accept_len.cpu().numpy().copy(), gr.run.bonus.cpu().numpy().copy()))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            np.testing.assert_array_equal(a, b)
    gr.run.h.close()


def test_cast_fused_calls_equal_separate_calls(torch):
    """dt_cast_prune_select and dt_cast_verify_rerank give exactly what the separate calls give."""
    import harness

    w = with_sizes("cast", V=32000)
    outs = []
    for fused in (True, False):
        gr = harness.GpuRound(w, fused=fused)
        res = []
        for rnd in range(3):
            attempts = np.zeros(w["B"], np.int64)
            roots = harness.root_tokens(w, harness.salts_of(w, rnd, attempts))
            gr.round(rnd, attempts, roots)
            t = harness.tree_numpy(gr.run.h)
            res.append((t["token"].copy(), t["value"].copy(), gr.run.selected.cpu().numpy().copy(),
                        gr.run.m_dev.cpu().numpy().copy(), gr.run.accept_len.cpu().numpy().copy(),
                        gr.run.bonus.cpu().numpy().copy(), gr.run.frontier_token.cpu().numpy().copy()))
        outs.append(res)
        gr.run.h.close()
    for ra, rb in zip(*outs):
        for a, b in zip(ra, rb):
            np.testing.assert_array_equal(a, b)


# Full sizes of the five workloads, in the launch configuration the benchmark uses (several rounds
# back to back on one handle, so that stale per-launch state would show up).
FULL = [("pr1", {}, 3), ("vicuna", {}, 2), ("vicuna", dict(T=1), 2), ("cast", {}, 3), ("graft", {}, 3),
        ("stress", {}, 1)]


@pytest.mark.parametrize("name,over,rounds", FULL)
def test_round_parity_full_size(torch, name, over, rounds):
    w = with_sizes(name, **over)
    _run_rounds(torch, w, rounds, label=f"full size {name} {over}")


@pytest.mark.parametrize("V,K", [(128256, 32), (128256, 10), (70001, 8)])
def test_expand_layer_ties_across_stages(torch, V, K):
    """Exact ties everywhere (all-equal rows) and coarse values with many ties at the K-th boundary:
    ties must go to the lower token id across stages, warps and segments (and the overflow path)."""
    _expand_case(torch, V, K, 2, 0, lambda B, V: np.zeros((B, V)))
    rng = np.random.default_rng(V + K)
    _expand_case(torch, V, K, 3, 0, lambda B, V: rng.integers(0, 4, (B, V)).astype(np.float64))
