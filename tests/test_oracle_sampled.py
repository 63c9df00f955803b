"""Pins of the sampled-draft oracle (``oracle.sampled``), all on the CPU.

What fixes them (not the oracle itself):
* Plackett-Luce: successive draws without replacement from q give the ordered sequence
  (t_1..t_K) with probability prod_j q(t_j) / (1 - sum_{i<j} q(t_i)); these sum to 1, and the
  Gumbel-top-K order drawn with the Philox uniforms must match them in frequency (chi-square).
* Losslessness (EAGLE-2 page, §"无损性为什么没有被动态树破坏"): whatever the draft distribution and
  the number of siblings, the emitted token is distributed exactly as the target's p. Checked by
  exact enumeration of every ordered draw, and by Monte Carlo with the Philox uniforms over a
  two-level tree (first token ~ p_root; second token, after an accepted first one, ~ p(.|t1)).
* The same for a whole round: with the frontier chosen by value and every drawn node verified,
  exact enumeration of every draw at two layers gives the target's first-token distribution.
* Special cases: q = p accepts the first child always; a single child (K = 1) is the page's
  one-token rule. Two plausible mistakes, planted here on the CPU, are not lossless, so the pins
  above would catch them: a proposal that ignores the earlier siblings, and a rerank that drops
  drawn nodes by their own values.
"""
import itertools

import numpy as np
import pytest

from oracle import philox, sampled


def _dist(rng, V, zeros=0):
    x = rng.normal(size=V) * 1.5
    if zeros:
        x[rng.choice(V, zeros, replace=False)] = -np.inf
    return sampled.softmax(x), x


def test_plackett_luce_sums_to_one():
    rng = np.random.default_rng(1)
    for V, K in ((4, 2), (5, 3), (6, 6)):
        q, _ = _dist(rng, V)
        tot = sum(sampled.plackett_luce(q, s) for s in itertools.permutations(range(V), K))
        assert tot == pytest.approx(1.0, abs=1e-12)


def test_draw_order_frequencies_match_plackett_luce():
    """Gumbel-top-3 orders drawn with the Philox draw noise at 24000 (node, round) pairs."""
    V, K, n = 5, 3, 24000
    x = np.array([0.3, -0.4, 1.1, 0.0, -1.2])
    q = sampled.softmax(x)
    counts = {}
    for i in range(n):
        seq = tuple(sampled.sample_children(x, K, seed=11, rnd=i // 4000, b=i % 3, node=i % 4000 // 3 + 7))
        counts[seq] = counts.get(seq, 0) + 1
    cells = list(itertools.permutations(range(V), K))
    exp = np.array([n * sampled.plackett_luce(q, s) for s in cells])
    obs = np.array([counts.get(s, 0) for s in cells])
    chi2 = float(((obs - exp) ** 2 / exp).sum())
    assert obs.sum() == n
    assert chi2 < 110.0, chi2  # 59 degrees of freedom: p ~ 1e-4 at 104


def _draw_counter_word2(b, node):
    return sampled.DRAW_STREAM + 4096 * b + node


def test_draw_uniforms_are_a_separate_stream():
    """The draw noise does not reuse the residual or the acceptance uniforms of any position.

    The three streams share a round (counter words 0-1) and the key; they differ in words 2-3:
      draw noise   word 2 = 0x40000000 + 4096 b + node, word 3 = v >> 2      (node < 4096)
      residual     word 2 = 512 b + pos,                word 3 = v >> 2      (pos < 512)
      acceptance   word 2 = 512 b + pos,                word 3 = 0x80000000
    For every request b < 2^18, node < 4096 and pos < 512 the draw stream's word 2 lies in
    [2^30, 2^31), the others' below 2^27 + 512; the acceptance stream's word 3 is 2^31, every
    token group's below 2^29 (V < 2^31). So no two streams ever use the same counter."""
    seed, rnd, b, node, V = 5, 3, 1, 2, 64
    u = sampled.draw_uniforms(seed, rnd, b, node, V)
    # the layout itself: each uniform is the published Philox block at the stated counter
    for v in (0, 1, 5, 63):
        w = philox.philox4x32_10((rnd, 0, _draw_counter_word2(b, node), v >> 2), (seed, 0))
        assert u[v] == ((int(w[v & 3]) >> 9) + 0.5) * 2.0 ** -23
    # range arithmetic at the extremes of every index
    b_max, node_max, pos_max = (1 << 18) - 1, 4095, 511
    lo_draw, hi_draw = _draw_counter_word2(0, 0), _draw_counter_word2(b_max, node_max)
    assert lo_draw == 1 << 30 and hi_draw == (1 << 31) - 1
    hi_other = 512 * b_max + pos_max
    assert hi_other < lo_draw
    assert ((1 << 31) - 1) >> 2 < 0x80000000
    # and the values differ from the other two streams at the same (round, request, index)
    g = philox.gumbel_uniforms(seed, rnd, b, node, V)
    assert (u > 0).all() and (u < 1).all()
    assert not np.allclose(u, g)
    a = philox.accept_uniform(seed, rnd, b, node)
    assert not np.any(np.abs(u - a) < 2.0 ** -22)
    with pytest.raises(ValueError):
        sampled.draw_uniforms(5, 3, 1, 4096, 8)


def test_draw_order_ties_and_infinities():
    u = np.full(6, 0.5)  # equal noise: the order is the logit order, ties to the lower id
    x = np.array([1.0, 2.0, 2.0, -np.inf, 0.5, 2.0])
    assert sampled.draw_order(x, 6, u) == [1, 2, 5, 0, 4]  # -inf is never drawn
    assert sampled.draw_order(x, 2, u) == [1, 2]


@pytest.mark.parametrize("seed", range(6))
def test_emitted_token_is_exactly_the_target_distribution(seed):
    rng = np.random.default_rng(100 + seed)
    V = 5
    p, _ = _dist(rng, V, zeros=seed % 2)
    q, _ = _dist(rng, V, zeros=(seed // 2) % 2)
    for K in (1, 2, 3, V):
        out = sampled.emit_distribution(p, q, K)
        np.testing.assert_allclose(out, p, atol=1e-12, rtol=0)


def test_single_child_is_the_one_token_rule():
    rng = np.random.default_rng(7)
    p, _ = _dist(rng, 4)
    q, _ = _dist(rng, 4)
    for t in range(4):  # accept min(1, p/q), else the residual norm(max(0, p - q))
        j, r = sampled.try_children(p, q, [t], [0.999999])
        a = min(1.0, p[t] / q[t])
        if a > 0.999999:
            assert j == 0
        else:
            assert j is None
            np.testing.assert_allclose(r, np.maximum(0, p - q) / np.maximum(0, p - q).sum(), atol=1e-15)


def test_equal_distributions_accept_the_first_child():
    rng = np.random.default_rng(3)
    p, x = _dist(rng, 6)
    for i in range(50):
        kids = sampled.sample_children(x, 3, seed=2, rnd=i, b=0, node=1)
        j, _ = sampled.try_children(p, p, kids, [philox.accept_uniform(2, i, 0, 1 + k) for k in range(3)])
        assert j == 0


def test_ignoring_earlier_siblings_is_not_lossless(monkeypatch):
    """Planted mistake: test every sibling against q itself instead of q without the earlier ones."""
    rng = np.random.default_rng(5)
    p, _ = _dist(rng, 5)
    q, _ = _dist(rng, 5)
    monkeypatch.setattr(sampled, "without", lambda qq, t: np.asarray(qq, dtype=np.float64))
    out = sampled.emit_distribution(p, q, 3)
    assert np.abs(out - p).max() > 1e-3


def test_two_level_walk_monte_carlo():
    """First emitted token ~ p_root; after an accepted first token t1 the next one ~ p(.|t1)."""
    V, K = 4, 2
    rng = np.random.default_rng(9)
    p_root, _ = _dist(rng, V)
    x_root = rng.normal(size=V)
    p_next = {t: _dist(rng, V)[0] for t in range(V)}
    x_next = {t: rng.normal(size=V) for t in range(V)}
    n = 12000
    first = np.zeros(V)
    second = np.zeros((V, V))
    for rnd in range(n):
        kids = sampled.sample_children(x_root, K, seed=4, rnd=rnd, b=0, node=0)
        children = {0: [(1 + j, t) for j, t in enumerate(kids)]}
        tok = {0: -1}
        pos = 1 + K
        for j, t in enumerate(kids):
            tok[1 + j] = t
            g = sampled.sample_children(x_next[t], K, seed=4, rnd=rnd, b=0, node=1 + j)
            children[1 + j] = [(pos + i, tt) for i, tt in enumerate(g)]
            for i, tt in enumerate(g):
                tok[pos + i] = tt
            pos += K

        def target(i):
            return p_root if i == 0 else p_next[tok[i]]

        def draft(i):
            return sampled.softmax(x_root if i == 0 else x_next[tok[i]])

        chain, bonus = sampled.walk(children, target, draft, seed=4, rnd=rnd, b=0, V=V)
        emitted = [tok[i] for i in chain[1:]] + [bonus]
        first[emitted[0]] += 1
        if len(chain) >= 2:
            second[emitted[0], emitted[1]] += 1
    chi2 = float(((first - n * p_root) ** 2 / (n * p_root)).sum())
    assert chi2 < 25.0, chi2  # 3 degrees of freedom
    for t in range(V):
        m = second[t].sum()
        if m < 400:
            continue
        exp = m * p_next[t]
        c2 = float(((second[t] - exp) ** 2 / exp).sum())
        assert c2 < 25.0, (t, c2)


# ------------------------------------------------------------------ the tree side ----
from oracle import tree as otree  # noqa: E402


def _exact_first_token(V, K, xs_draft, x_target_root, keep=None):
    """Exact first-token distribution of a round with one frontier node at layer 2 (W = 1, D = 2):
    every ordered draw at both layers enumerated with its Plackett-Luce probability. ``keep``
    (optional) maps (tree, root draw, layer-2 draw) to the root children actually verified."""
    p = sampled.softmax(x_target_root)
    q0 = sampled.softmax(xs_draft[0])
    out = np.zeros(V)
    for s1 in itertools.permutations(range(V), K):
        w1 = sampled.plackett_luce(q0, s1)
        t = otree.OracleTree(1, K, 1, 2, root_tokens=[0])
        t.expand_layer(lambda b, f: xs_draft[0], sampler=lambda b, node, x: list(s1))
        t.select_frontier(1)
        fnode = int(t.frontier[0][0])
        q1 = sampled.softmax(xs_draft[int(t.token[0, fnode])])
        for s2 in itertools.permutations(range(V), K):
            w = w1 * sampled.plackett_luce(q1, s2)
            t2 = otree.OracleTree(1, K, 1, 2, root_tokens=[0])
            t2.expand_layer(lambda b, f: xs_draft[0], sampler=lambda b, node, x: list(s1))
            t2.select_frontier(1)
            t2.expand_layer(lambda b, f: xs_draft[int(t2.token[0, fnode])], sampler=lambda b, node, x: list(s2))
            kids = list(s1) if keep is None else keep(t2)
            r, qj, stay = p.copy(), q0.copy(), 1.0
            for tok in kids:
                a = sampled.accept_probability(r, qj, tok)
                out[tok] += w * stay * a
                stay *= 1.0 - a
                r = sampled.residual(r, qj)
                qj = sampled.without(qj, tok)
            out += w * stay * r
    return out, p


@pytest.mark.parametrize("trial", range(4))
def test_whole_drawn_tree_is_exactly_lossless(trial):
    """Frontier by value, every drawn node verified: the first token is exactly the target's."""
    rng = np.random.default_rng(40 + trial)
    V, K = 3, 2
    xs = {tok: rng.normal(size=V) * 1.5 for tok in range(V)}
    out, p = _exact_first_token(V, K, xs, rng.normal(size=V) * 1.5)
    np.testing.assert_allclose(out, p, atol=1e-12, rtol=0)


def test_pruning_drawn_nodes_by_value_is_not_lossless():
    """Planted mistake: keep only the best m drawn nodes by value (a rerank after the draws); the
    root children that survive then depend on their own draws, and the first token is biased."""
    rng = np.random.default_rng(43)
    V, K, m = 3, 2, 3
    xs = {tok: rng.normal(size=V) * 1.5 for tok in range(V)}

    def keep(t):
        ids = t.sorted_nodes(0, t.nodes(0))[:m]
        kept = sorted(i for i in ids if t.parent[0, i] == 0)
        # a later-drawn root child without the earlier one is not a prefix: keep the prefix only
        pref = []
        for r, i in enumerate(range(1, 1 + K)):
            if i not in kept:
                break
            pref.append(int(t.token[0, i]))
        return pref

    out, p = _exact_first_token(V, K, xs, rng.normal(size=V) * 1.5, keep=keep)
    assert np.abs(out - p).max() > 1e-3


def test_sampled_round_first_token_is_the_target_distribution():
    """Whole round with sampled drafts and the Philox draws (expand 2 layers, frontier, every drawn
    node verified, flatten, verify): the first emitted token is distributed as the target row at
    the root."""
    V, K, W, D = 4, 2, 2, 2
    rng = np.random.default_rng(23)
    x_draft = {tok: rng.normal(size=V) for tok in range(-1, V)}
    x_target = {tok: rng.normal(size=V) * 1.3 for tok in range(-1, V)}
    p_root = sampled.softmax(x_target[0])
    n = 6000
    first = np.zeros(V)
    for rnd in range(n):
        t = otree.OracleTree(1, K, W, D, root_tokens=[0])
        drawn = lambda b, node, x, rnd=rnd: sampled.sample_children(x, K, seed=8, rnd=rnd, b=b, node=node)
        t.expand_layer(lambda b, f: x_draft[int(t.token[b, t.frontier[b][f]])], sampler=drawn)
        t.select_frontier(W)
        t.expand_layer(lambda b, f: x_draft[int(t.token[b, t.frontier[b][f]])], sampler=drawn)
        n_all = len(t.nodes(0))
        sel = t.rerank(n_all, n_all)  # every drawn node
        meta = otree.build_meta(t, sel, np.zeros(1, np.int64), n_all + 1, D + 1)
        acc, path, bonus = sampled.verify_tree(
            t, meta, lambda b, i: x_target[int(meta["tokens"][b, i]) if i > 0 else 0], seed=8, rnd=rnd)
        tok0 = int(meta["tokens"][0, path[0, 1]]) if acc[0] >= 1 else int(bonus[0])
        first[tok0] += 1
    chi2 = float(((first - n * p_root) ** 2 / (n * p_root)).sum())
    assert chi2 < 25.0, (chi2, first / n, p_root)


def test_run_round_with_sampled_drafts_is_the_pinned_composition():
    """``run_round`` with ``draft_sampling`` takes exactly the steps of the round whose first token is
    pinned to the target distribution above (expand with the Philox draws, frontier by value, every
    drawn node selected, flatten, the sampled walk): same tree, metadata and outputs, round by round."""
    import oracle.round as oround

    V, K, W, D = 5, 2, 2, 3
    rng = np.random.default_rng(5)
    x_draft = {(d, tok): rng.normal(size=V) for d in range(1, D + 1) for tok in range(V)}
    x_target = {(d, tok): rng.normal(size=V) * 1.3 for d in range(1, D + 2) for tok in range(V)}
    N = otree.n_nodes(K, W, D)
    cfg = dict(policy="eagle", draft_sampling=True, B=2, K=K, W=W, D=D, k=W, m=N - 1, m_cap=N - 1, P=N,
               D_path=D + 1, T=1, seed=11)
    for rnd in range(12):
        roots = np.array([rnd % V, (rnd + 2) % V])
        ref = oround.run_round(cfg, roots, lambda b, d, ctx: x_draft[(d, ctx)],
                               lambda b, d, ctx: x_target[(d, ctx)], rnd=rnd)
        t = otree.OracleTree(2, K, W, D, root_tokens=roots)
        drawn = lambda b, node, x: sampled.sample_children(x, K, seed=11, rnd=rnd, b=b, node=node)  # noqa: E731
        for d in range(1, D + 1):
            t.expand_layer(lambda b, f: x_draft[(d, int(t.token[b, t.frontier[b][f]]))], sampler=drawn)
            if d < D:
                t.select_frontier(W)
        sel = t.rerank([len(t.nodes(b)) for b in range(2)], N - 1)
        meta = otree.build_meta(t, sel, np.zeros(2, np.int64), N, D + 1)
        acc, path, bonus = sampled.verify_tree(
            t, meta, lambda b, i: x_target[(int(meta["depth"][b, i]) + 1, int(meta["tokens"][b, i]))], seed=11,
            rnd=rnd)
        np.testing.assert_array_equal(ref["tree"].token, t.token)
        np.testing.assert_array_equal(ref["meta"]["tokens"], meta["tokens"])
        np.testing.assert_array_equal(ref["accept_len"], acc)
        np.testing.assert_array_equal(ref["accept_path"], path)
        np.testing.assert_array_equal(ref["bonus"], bonus)
