"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics (CPU only).

Each test ties an oracle function to something other than itself: published
known-answer vectors, a library routine computing the same definition, brute
force over tiny inputs, invariants the pages state, closed forms, and special
cases that reduce to a known answer.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import philox
from oracle import cast as ocast
from oracle import graft as ograft
from oracle.tree import OracleTree, build_meta, row_softmax_topk, Gaps, layer_base, n_nodes
from oracle.verify import verify_greedy, verify_sample, row_top8, argmax_lowest


# ---------------------------------------------------------------- Philox ----
def test_philox_known_answers(golden_dir):
    """Published Random123 vectors for Philox4x32-10 (SC'11 paper's generator)."""
    n = 0
    for line in open(f"{golden_dir}/philox4x32_10_kat.txt"):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        out = philox.philox4x32_10(tuple(w[0:4]), (w[4], w[5]))
        assert [int(x) for x in out] == w[6:10]
        n += 1
    assert n == 3


def test_philox_uniform_ranges():
    us = [philox.accept_uniform(7, r, 3, 5) for r in range(2000)]
    assert min(us) >= 0.0 and max(us) < 1.0
    assert abs(np.mean(us) - 0.5) < 0.03
    g = philox.gumbel_uniforms(7, 1, 0, 2, 4096)
    assert g.min() > 0.0 and g.max() < 1.0
    assert abs(g.mean() - 0.5) < 0.02
    # the uniform of token v uses word v & 3 of counter v >> 2
    w = philox.philox4x32_10((1, 0, 2, 5), (7, 0))
    assert g[21] == ((int(w[1]) >> 9) + 0.5) * 2.0 ** -23


# ---------------------------------------------------- softmax + top-K (a1) ----
def _bf16_round(x):
    t = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64)
    return t.numpy()


@pytest.mark.parametrize("V,K", [(7, 1), (50, 4), (300, 10), (1000, 32)])
def test_softmax_topk_matches_library_and_bruteforce(V, K):
    rng = np.random.default_rng(V * 31 + K)
    x = _bf16_round(rng.normal(0, 2, V))          # bf16 quantisation makes ties common
    toks, logc, m, logS = row_softmax_topk(x, K)
    # softmax: library routine in fp64
    p = torch.softmax(torch.tensor(x, dtype=torch.float64), 0).numpy()
    np.testing.assert_allclose(np.exp(logc), p[toks], rtol=1e-13)
    assert m == x.max()
    # top-K: brute force with the (logit desc, id asc) order
    brute = sorted(range(V), key=lambda v: (-x[v], v))[:K]
    assert list(toks) == brute


def test_softmax_topk_all_equal_and_extremes():
    x = np.zeros(16)
    toks, logc, _, _ = row_softmax_topk(x, 5)
    assert list(toks) == [0, 1, 2, 3, 4]
    np.testing.assert_allclose(logc, np.log(1 / 16), rtol=1e-15)
    x = np.full(8, -np.inf)
    x[3] = 1.5
    toks, logc, _, _ = row_softmax_topk(x, 2)
    assert toks[0] == 3 and logc[0] == 0.0 and logc[1] == -np.inf
    for bad in (np.array([0.0, np.nan]), np.array([0.0, np.inf]), np.full(3, -np.inf)):
        with pytest.raises(ValueError):
            row_softmax_topk(bad, 1)


# -------------------------------------------------- tree construction (a2) ----
def _random_tree(B=2, K=3, W=2, D=4, V=40, seed=0, width=None, quant=False):
    rng = np.random.default_rng(seed)
    rows = {}

    def draft_row(b, d, ctx):
        key = (b, d, ctx)
        if key not in rows:
            r = rng.normal(0, 2, V)
            rows[key] = _bf16_round(r) if quant else r
        return rows[key]

    roots = rng.integers(0, V, B)
    t = OracleTree(B, K, W, D, roots)
    t.expand_layer(lambda b, f: draft_row(b, 1, int(t.token[b, t.frontier[b][f]])))
    for d in range(2, D + 1):
        t.select_frontier(W if width is None else width)
        t.expand_layer(lambda b, f, d=d: draft_row(b, d, int(t.token[b, t.frontier[b][f]])))
    return t, draft_row


def test_value_monotone_and_path_product():
    """V_child <= V_parent, and exp(value) = product of library-softmax confidences on the path."""
    t, draft_row = _random_tree(B=3, K=4, W=3, D=5, V=60, seed=1)
    for b in range(t.B):
        for i in t.nodes(b):
            par = t.parent[b, i]
            assert t.value[b, i] <= t.value[b, par]
            prod = 1.0
            for a, c in zip(t.path(b, i)[:-1], t.path(b, i)[1:]):
                row = draft_row(b, t.depth[b, c], int(t.token[b, a]))
                p = torch.softmax(torch.tensor(row, dtype=torch.float64), 0)[t.token[b, c]].item()
                prod *= p
            assert math.isclose(math.exp(t.value[b, i]), prod, rel_tol=1e-12)


def test_layout_and_frontier_is_topk_of_layer():
    K, W, D = 3, 2, 4
    t, _ = _random_tree(B=2, K=K, W=W, D=D, V=30, seed=2)
    assert t.N == n_nodes(K, W, D) == 1 + K + (D - 1) * W * K
    for b in range(t.B):
        # layer 2's parents are exactly the top-W of layer 1 by value, in id order
        l1 = t.layer_ids(b, 1)
        top = sorted(sorted(l1, key=lambda i: (-t.value[b, i], i))[:W])
        base2 = layer_base(2, K, W)
        for f in range(W):
            for r in range(K):
                assert t.parent[b, base2 + f * K + r] == top[f]
        # children of one frontier slot are that row's top-K in rank order
        for d in range(1, D + 1):
            ids = t.layer_ids(b, d)
            for s in range(0, len(ids), K):
                sib = ids[s:s + K]
                assert len({t.parent[b, i] for i in sib}) == 1
                assert all(t.logc[b, sib[j]] >= t.logc[b, sib[j + 1]] for j in range(len(sib) - 1))


def test_frontier_width_and_stop():
    t, _ = _random_tree(B=3, K=3, W=3, D=2, V=30, seed=3)
    t.cur_depth = 1
    toks = t.select_frontier([1, 3, 2], stop=[False, False, True])
    assert [len(f) for f in t.frontier] == [1, 3, 0]
    assert toks[2].tolist() == [-1, -1, -1]
    assert toks[0, 0] == t.token[0, t.frontier[0][0]]


# ------------------------------------------------------------ rerank (a5) ----
def _parent_closed(t, b, sel):
    s = set(sel)
    return all(t.parent[b, i] == 0 or t.parent[b, i] in s for i in sel)


@pytest.mark.parametrize("seed", range(6))
def test_rerank_bruteforce_connected_max(seed):
    """Top-m in the total order is parent-closed and maximises sum exp(value) (tiny trees)."""
    t, _ = _random_tree(B=1, K=2, W=2, D=3, V=25, seed=10 + seed)
    nodes = t.nodes(0)
    assert len(nodes) <= 13
    for m in range(1, len(nodes) + 1):
        sel = [int(i) for i in t.rerank(m, m)[0] if i >= 0]
        assert sel == sorted(sel) and len(sel) == m
        assert _parent_closed(t, 0, sel)
        best, arg = -1.0, None
        for sub in itertools.combinations(nodes, m):
            if not _parent_closed(t, 0, sub):
                continue
            s = sum(math.exp(t.value[0, i]) for i in sub)
            if s > best:
                best, arg = s, sorted(sub)
        assert sel == arg


def test_rerank_shallow_first_on_ties():
    """Equal values: the shallower (lower id) node wins, so the selection stays connected."""
    t = OracleTree(1, 2, 1, 2, [0])
    x = np.array([0.0, 0.0, -50.0, -50.0])       # root row: tokens 0 and 1 tie
    t.expand_layer(np.array([[x]]))
    t.select_frontier(1)
    t.expand_layer(np.array([[np.array([10.0, -40.0, -40.0, -40.0])]]))  # child c ~= 1
    sel = t.rerank(2, 2)[0]
    # layer-1 nodes both have log(0.5); the depth-2 child is log(0.5)+~0: ties broken by id
    assert list(sel) == [1, 2]
    assert _parent_closed(t, 0, list(sel))


# -------------------------------------------------------------- meta (a7) ----
def test_meta_mask_is_transitive_closure():
    t, _ = _random_tree(B=2, K=3, W=2, D=4, V=30, seed=4)
    sel = t.rerank(9, 12)
    meta = build_meta(t, sel, np.array([100, 7]), P=13, D_path=5)
    for b in range(2):
        n = int(meta["n_pos"][b])
        assert n == 10
        A = np.zeros((n, n), np.int64)
        for i in range(1, n):
            A[i, meta["parents"][b, i]] = 1
        R = np.eye(n, dtype=np.int64)
        for _ in range(n):
            R = np.minimum(1, R + R @ A)
        np.testing.assert_array_equal(meta["mask"][b, :n, :n], R)
        assert not meta["mask"][b, n:].any()
        np.testing.assert_array_equal(meta["position_ids"][b, :n], [100, 7][b] + meta["depth"][b, :n])
        # leaves and retrieve rows
        has_child = set(int(meta["parents"][b, i]) for i in range(1, n))
        leaves = [i for i in range(n) if i not in has_child]
        assert meta["n_leaves"][b] == len(leaves)
        for r, leaf in enumerate(leaves):
            row = [int(p) for p in meta["retrieve"][b, r] if p >= 0]
            assert row[0] == 0 and row[-1] == leaf
            assert all(meta["parents"][b, row[j + 1]] == row[j] for j in range(len(row) - 1))
        # positions 1.. are the selected ids in ascending order
        assert list(meta["node_id"][b, 1:n]) == sorted(int(i) for i in sel[b] if i >= 0)


# ----------------------------------------------------------- verify (a8-a9) ----
def test_greedy_target_equals_draft_gives_greedy_chain():
    B, K, W, D, V = 3, 3, 3, 5, 40
    t, draft_row = _random_tree(B=B, K=K, W=W, D=D, V=V, seed=5)
    sel = t.rerank(12, 12)
    meta = build_meta(t, sel, np.zeros(B, np.int64), P=13, D_path=D + 1)

    def trow(b, i):
        return draft_row(b, int(meta["depth"][b, i]) + 1, int(meta["tokens"][b, i]))

    acc, path, bonus = verify_greedy(meta, trow)
    for b in range(B):
        pos_of = {int(meta["node_id"][b, i]): i for i in range(int(meta["n_pos"][b]))}
        cur, depth, node = 0, 0, 0
        while True:
            row = draft_row(b, depth + 1, int(t.token[b, node]))
            tok = argmax_lowest(row)
            nxt = [i for i in t.nodes(b) if t.parent[b, i] == node and t.token[b, i] == tok]
            if not nxt or nxt[0] not in pos_of:
                break
            node, depth = nxt[0], depth + 1
        assert acc[b] == depth
        assert bonus[b] == argmax_lowest(draft_row(b, depth + 1, int(t.token[b, node])))
        assert path[b, depth] == pos_of[node]


def test_greedy_no_match_gives_root_bonus():
    B, K, W, D, V = 2, 3, 2, 3, 30
    t, draft_row = _random_tree(B=B, K=K, W=W, D=D, V=V, seed=6)
    sel = t.rerank(6, 6)
    meta = build_meta(t, sel, np.zeros(B, np.int64), P=7, D_path=D + 1)
    used = set(int(x) for x in meta["tokens"].ravel() if x >= 0)
    free = [v for v in range(V) if v not in used][0]

    def trow(b, i):
        r = np.zeros(V)
        r[free] = 5.0
        return r

    acc, path, bonus = verify_greedy(meta, trow)
    assert list(acc) == [0, 0] and list(bonus) == [free, free]
    assert list(path[:, 0]) == [0, 0] and (path[:, 1:] == -1).all()


def _exact_next_token_dist(P_row, child_tokens, child_pos):
    """Exact distribution of the next emitted token at a node under the rule (point-mass proposals).

    Enumerates accept/reject outcomes analytically: child j is accepted with
    probability resid(x_j)/sum(resid); on rejection x_j is removed from resid.
    """
    resid = P_row.copy()
    out = np.zeros_like(P_row)
    reach = 1.0
    for x in child_tokens:
        if x < 0:
            continue
        a = resid[x] / resid.sum()
        out[x] += reach * a
        reach *= 1 - a
        resid[x] = 0.0
    out += reach * resid / resid.sum()
    return out


@pytest.mark.parametrize("seed", range(4))
def test_sampling_rule_lossless_exact_enumeration(seed):
    """Point-mass reading of min(1,p/q) + residual: the next-token law equals the target's (V=8)."""
    rng = np.random.default_rng(100 + seed)
    V = 8
    for _ in range(20):
        P = rng.dirichlet(np.ones(V) * rng.uniform(0.2, 3))
        n_child = rng.integers(0, 6)
        kids = list(rng.integers(-1, V, n_child))          # duplicates and invalid (-1) allowed
        np.testing.assert_allclose(_exact_next_token_dist(P, kids, None), P, atol=1e-12)


def _chi2_ok(counts, probs, n):
    exp = probs * n
    keep = exp > 5
    stat = float((((counts - exp) ** 2)[keep] / exp[keep]).sum())
    dof = int(keep.sum()) - 1
    from scipy.stats import chi2
    return chi2.sf(stat, dof) > 1e-4, stat, dof


def test_sampling_monte_carlo_first_two_tokens():
    """Oracle's sampled verify: first emitted token ~ P_root; second ~ P_child given acceptance."""
    V, B = 8, 64
    rng = np.random.default_rng(9)
    # hand-built tree: root with children tokens [2, 5, 2(dup)], child pos1 has children [1, 6];
    # the root row puts half its mass on token 2 so that renormalising after a rejection matters
    P_rows = [rng.normal(0, 1.2, V) for _ in range(6)]
    P_rows[0] = np.log(np.array([0.02, 0.03, 0.5, 0.05, 0.05, 0.25, 0.06, 0.04]))
    P_rows[1] = np.log(np.array([0.05, 0.4, 0.05, 0.1, 0.1, 0.05, 0.2, 0.05]))
    tokens = np.array([3, 2, 5, 2, 1, 6])
    parents = np.array([-1, 0, 0, 0, 1, 1])
    P = 6
    meta = dict(tokens=np.tile(tokens, (B, 1)), parents=np.tile(parents, (B, 1)),
                n_pos=np.full(B, P), retrieve=np.full((B, P, 4), -1))
    first = np.zeros(V)
    second = np.zeros(V)
    rounds = 160
    for rnd in range(rounds):
        acc, path, bonus = verify_sample(meta, lambda b, i: P_rows[i], seed=11, rnd=rnd)
        for b in range(B):
            toks = [int(tokens[p]) for p in path[b] if p >= 1] + [int(bonus[b])]
            first[toks[0]] += 1
            if acc[b] >= 1 and path[b, 1] == 1:
                second[toks[1]] += 1
    sm = lambda x: np.exp(x - x.max()) / np.exp(x - x.max()).sum()
    ok, stat, dof = _chi2_ok(first, sm(P_rows[0]), first.sum())
    assert ok, (stat, dof)
    ok, stat, dof = _chi2_ok(second, sm(P_rows[1]), second.sum())
    assert ok, (stat, dof)


def test_sampling_certain_accept_and_leaf_bonus():
    V = 6
    big = np.array([0.0, 0.0, 60.0, 0.0, 0.0, 0.0])      # P(2) = 1 to fp64 precision
    meta = dict(tokens=np.array([[0, 2]]), parents=np.array([[-1, 0]]), n_pos=np.array([2]),
                retrieve=np.full((1, 2, 3), -1))
    for rnd in range(50):
        acc, path, bonus = verify_sample(meta, lambda b, i: big if i == 0 else np.arange(V, dtype=float),
                                         seed=3, rnd=rnd)
        assert acc[0] == 1 and list(path[0, :2]) == [0, 1]
    # a leaf's bonus is a Gumbel-max draw from its row: check its law by Monte Carlo
    row = np.log(np.array([0.05, 0.1, 0.15, 0.2, 0.25, 0.25]))
    meta = dict(tokens=np.zeros((1, 1), np.int64), parents=np.full((1, 1), -1),
                n_pos=np.array([1]), retrieve=np.full((1, 1, 2), -1))
    cnt = np.zeros(V)
    for rnd in range(4000):
        _, _, bonus = verify_sample(meta, lambda b, i: row, seed=5, rnd=rnd)
        cnt[bonus[0]] += 1
    ok, stat, dof = _chi2_ok(cnt, np.exp(row), cnt.sum())
    assert ok, (stat, dof)


def test_row_top8_bruteforce():
    rng = np.random.default_rng(12)
    V = 50
    rows = [_bf16_round(rng.normal(0, 1, V)) for _ in range(3)]
    meta = dict(tokens=np.array([[1, 2, -1]]), n_pos=np.array([3]))
    t8 = row_top8(meta, lambda b, i: rows[i])
    for i in range(2):
        assert list(t8[0, i]) == sorted(range(V), key=lambda v: (-rows[i][v], v))[:8]
    assert (t8[0, 2] == -1).all()


# -------------------------------------------------------------- CAST (a3) ----
def test_cast_select_row():
    assert ocast.select_row(0, 512, 16) == 0
    assert ocast.select_row(511, 512, 16) == 0
    assert ocast.select_row(512, 512, 16) == 1
    assert ocast.select_row(5 * 512 + 3, 512, 16) == 5
    assert ocast.select_row(10 ** 9, 512, 16) == 15


def _theorem_tree(seed):
    t, _ = _random_tree(B=3, K=10, W=1, D=1, V=200, seed=seed)
    return t


@pytest.mark.parametrize("seed", range(3))
def test_cast_theorem_4_1_width_equals_fixed_topk(seed):
    """c_j = lambda*j + delta and C1 = sum_j v^(j)(K)/(B lambda) keep exactly K (Theorem 4.1)."""
    t = _theorem_tree(30 + seed)
    lam, delta, Kfix = 0.37, 0.11, 4
    M_rows, N_cols = 4, 64
    S_T = np.ones((M_rows, N_cols))
    S_D = np.tile(lam * np.arange(1, N_cols + 1) + delta, (M_rows, 1))
    vK = sum(math.exp(t.value[b, sorted(t.layer_ids(b, 1), key=lambda i: (-t.value[b, i], i))[Kfix - 1]])
             for b in range(t.B))
    C1 = vK / (t.B * lam)
    base = dict(S_T=S_T, S_D=S_D, L=512.0, n0=0, C2=0.0, R=3, width_cap=10, D_max=8)
    n, _ = ocast.width_depth(t, 1, ocast.CastState(), dict(base, C1=C1 * (1 - 1e-9)))
    assert n == Kfix
    n, _ = ocast.width_depth(t, 1, ocast.CastState(), dict(base, C1=C1 * (1 + 1e-9)))
    assert n == Kfix - 1


def test_cast_theorem_4_1_exact_equality_keeps_k():
    """Exact binary-fraction instance: C1 equal to v(K)/lambda keeps K (">=" comparator)."""
    items = np.array([0.5, 0.25, 0.25, 0.125, 0.0625])
    cost = np.array([0.0, 1.0, 2.0, 3.0, 4.0, 5.0])         # lambda = 1, delta = 0
    assert ocast.selection_rule(items, cost, 0.25, 5) == 3  # v(K=3) = 0.25
    assert ocast.selection_rule(items, cost, 0.125, 5) == 4
    assert ocast.selection_rule(items, cost, 0.5, 5) == 1
    # non-concave: a dip then a rise; the scan continues after a failed step
    items = np.array([0.5, 0.01, 0.3, 0.01])
    cost = np.array([0.0, 1.0, 2.0, 3.0, 4.0])
    assert ocast.selection_rule(items, cost, 0.1, 4) == 3   # (0.01+0.3)/2 >= 0.1 from k0 = 1


def test_cast_verify_count_linear_cost_gives_fixed_m():
    t, _ = _random_tree(B=2, K=4, W=3, D=3, V=80, seed=40)
    a, lam_T = 1.0, 0.25
    S_T = np.tile(a + lam_T * np.arange(1, 65), (2, 1))
    slope = lam_T / (a + lam_T)
    m_fix = 7
    srt = [sorted(t.nodes(b), key=lambda i: (-t.value[b, i], i)) for b in range(2)]
    vbar = sum(math.exp(t.value[b, srt[b][m_fix - 1]]) for b in range(2)) / 2
    p = dict(S_T=S_T, L=512.0, n0=0, m_cap=60)
    assert ocast.verify_count(t, dict(p, C3=vbar / slope * (1 - 1e-9))) == m_fix
    assert ocast.verify_count(t, dict(p, C3=vbar / slope * (1 + 1e-9))) == m_fix - 1


def test_cast_flat_cost_is_free_and_depth_extremes():
    t = _theorem_tree(50)
    S = np.ones((2, 16))
    p = dict(S_T=S, S_D=S, L=512.0, n0=0, C1=1e30, C2=0.0, R=3, width_cap=10, D_max=8)
    n, grow = ocast.width_depth(t, 1, ocast.CastState(), p)
    assert n == 10 and grow                   # flat cost: every step is free; C2 = 0 always grows
    n, grow = ocast.width_depth(t, 1, ocast.CastState(), dict(p, C2=1e30))
    assert not grow
    n, grow = ocast.width_depth(t, 1, ocast.CastState(), dict(p, D_max=1))
    assert not grow                           # maximum depth reached


def test_cast_depth_fifo_worked_example():
    """Two layers, B=1, hand-computed: phi pushed after layer 2, alpha = mean({1, phi})."""
    t = OracleTree(1, 2, 1, 2, [0])
    t.expand_layer(np.array([[np.log(np.array([0.6, 0.3, 0.1]))]]))
    S_T = np.ones((1, 8))
    S_D = np.tile(np.arange(1, 9, dtype=float), (1, 1))   # c_k = k
    st = ocast.CastState()
    p = dict(S_T=S_T, S_D=S_D, L=512.0, n0=0, C1=0.25, C2=0.1, R=3, width_cap=2, D_max=8)
    n1, g1 = ocast.width_depth(t, 1, st, p)
    # items 0.6, 0.3: marginal 0.3 >= 0.25 -> n1 = 2; key = 1 * 0.9 / 2 = 0.45 >= 0.1
    assert n1 == 2 and g1 and st.fifo == [1.0] and math.isclose(st.u_prev, 0.9)
    t.select_frontier(1)
    t.expand_layer(np.array([[np.log(np.array([0.5, 0.5, 1e-300]))]]))
    n2, g2 = ocast.width_depth(t, 2, st, p)
    # layer 2 values 0.6*0.5 twice: marginal 0.3 >= 0.25 -> n2 = 2, u = 0.6, phi = 0.6/0.9
    assert n2 == 2
    assert st.fifo[0] == 1.0 and math.isclose(st.fifo[1], 0.6 / 0.9)
    assert g2 == ((1 + 0.6 / 0.9) / 2 * 0.6 / 2 >= 0.1)


# ------------------------------------------------------------- Graft (a4, a6, a10) ----
def _graft_tree(seed, D=8):
    return _random_tree(B=3, K=8, W=8, D=1, V=300, seed=seed)[0]


def test_graft_checkpoint_thresholds():
    t = _graft_tree(60)
    p = dict(ckpt_layers=[0, 1, 5], tau=[0.0, 0.0, 0.0], k_draft=[8, 24, 40], K_total=60, D_max=8)
    stop, stage, m = [False] * 3, [-1] * 3, [60] * 3
    ograft.checkpoint(t, 1, p, stop, stage, m)
    assert stop == [False] * 3                   # c > 0 always passes
    p["tau"] = [1.5, 1.5, 1.5]                   # c <= 1 always fails at d0
    ograft.checkpoint(t, 1, p, stop, stage, m)
    assert stop == [True] * 3 and stage == [0] * 3 and m == [8] * 3
    assert [60 - x for x in m] == [52] * 3


def test_graft_checkpoint_is_strict():
    """c_d = tau_d exactly must fail (g_d = 1[c_d > tau_d])."""
    t = OracleTree(1, 2, 1, 8, [0])
    row = np.full(5, -np.inf)
    row[1] = 0.0                                 # a single finite logit: c = exp(0) = 1 exactly
    t.expand_layer(np.array([[row]]))
    p = dict(ckpt_layers=[0, 1, 5], tau=[1.0, 0.0, 0.0], k_draft=[8, 24, 40], K_total=60, D_max=8)
    stop, stage, m = [False], [-1], [60]
    ograft.checkpoint(t, 1, p, stop, stage, m)
    assert stop == [True] and stage == [0] and m == [8]
    p["tau"] = [np.nextafter(1.0, 0.0), 0.0, 0.0]
    stop, stage, m = [False], [-1], [60]
    ograft.checkpoint(t, 1, p, stop, stage, m)
    assert stop == [False]


def test_graft_retrieve_and_update():
    V, B = 20, 1
    M = np.full((B, V, 8), -1, np.int64)
    tpl = ograft.default_template()
    assert len(tpl[0]) == 64 and tpl[0][:8] == [-1] * 8 and tpl[0][8] == 0 and tpl[1][8] == 0
    M[0, 3] = [4, 5, 6, 7, 8, 9, 10, 11]
    M[0, 4] = [12, 13, 14, 15, 16, 17, 18, 19]
    M[0, 12] = [3, 0, 0, 0, 0, 0, 0, 0]
    out = ograft.retrieve(M, [3], [18], tpl)
    toks, pars = out[0]
    assert toks[:8] == [4, 5, 6, 7, 8, 9, 10, 11]
    assert toks[8] == 12 and toks[9:16] == [-1] * 7       # only token 4 has a row
    assert toks[16] == 3 and toks[17] == -1
    assert pars[8] == 0 and pars[16] == 8
    # refresh: highest position wins for a repeated token
    meta = dict(tokens=np.array([[3, 5, 3, -1]]), n_pos=np.array([4]))
    top8 = np.arange(4 * 8).reshape(1, 4, 8)
    ograft.adj_update(M, meta, top8)
    assert list(M[0, 3]) == list(range(16, 24)) and list(M[0, 5]) == list(range(8, 16))


def test_graft_hybrid_positions_constant():
    t = _graft_tree(61)
    sel = t.rerank([8, 8, 8], 60)
    M = np.full((3, 300, 8), -1, np.int64)
    ret = ograft.retrieve(M, list(t.token[:, 0]), [52] * 3, ograft.default_template())
    meta = build_meta(t, sel, np.zeros(3, np.int64), P=61, D_path=10, retrieved=ret)
    assert list(meta["n_pos"]) == [61] * 3
    assert (meta["tokens"][:, 9:] == -1).all()        # empty M: all grafted nodes are padding
    assert meta["depth"][0, 60] == 7                  # 52 nodes: six full levels + 4 of the 7th
