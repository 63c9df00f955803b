"""Pins of the oracle's round composition (``oracle.round.run_round``), CPU only.

Every expected value below is worked out by hand from the pages' rules, in the comments next to
it, on rounds whose draft and target rows are written out as probabilities (logits = log p, so a
child's confidence is exactly the probability written down). These tests fix how the steps
compose, which the per-step pins cannot:

* CAST page §关键设计 2-4: the width test of layer i reads the cost-table row of the context
  n0 + sum of the widths chosen so far; the depth test pushes the gain ratio after every pruned
  layer and keeps the last R ratios; the batch stops when the test fails; the verify count runs
  on the whole tree after the last layer;
* Graft page, steps (1)-(2): a failed checkpoint stops the request with stage s and budget
  K_draft[s]; the retrieval fills K_max minus the draft nodes actually selected (not minus the
  budget), with padding where M has no entry;
* EAGLE-2 page §扩展阶段 / §重排阶段: the tree stops at depth D; the frontier is the top-k of the
  newest layer; the rerank keeps the top-m; greedy verify walks the argmax chain.

Each test also plants a mistake in a copy of the oracle (a source edit, compiled on the spot) and
checks that the hand-derived expectation then fails.
"""
import copy
import inspect
import math
import textwrap

import numpy as np

import oracle.cast as ocast
import oracle.round as oround
from oracle.graft import default_template

V = 10


def prow(probs):
    """Logits (log p) of a row over V tokens: the listed tokens get the listed probabilities, the
    others share the remaining mass equally (each below every listed one in these tests)."""
    p = np.full(V, (1.0 - sum(probs.values())) / (V - len(probs)))
    for t, q in probs.items():
        p[t] = q
    return np.log(p)


def rows_from(table, default=None):
    """(b, d, ctx) -> row, from a dict keyed by (d, ctx); every request gets the same rows."""
    default = default if default is not None else {0: 0.34, 1: 0.33}

    def f(b, d, ctx):
        return prow(table.get((d, ctx), default))
    return f


def mutated(func, old, new=None, extra_globals=None):
    """A copy of ``func`` compiled from its source with ``old`` replaced by ``new`` (a planted
    mistake); ``old`` may instead be a list of (old, new) pairs. Fails if an ``old`` is not in the
    source, so a stale mutation cannot pass silently."""
    src = textwrap.dedent(inspect.getsource(func))
    for a, b in (old if new is None else [(old, new)]):
        assert a in src, f"mutation anchor not found: {a!r}"
        src = src.replace(a, b)
    g = dict(func.__globals__)
    g.update(extra_globals or {})
    exec(compile(src, inspect.getsourcefile(func), "exec"), g)
    return g[func.__name__]


# ------------------------------------------------------------------------------ CAST ----
# Draft rows (d = layer the children land in, ctx = token of the expanded node):
#   layer 1 from the root (token 2):  p = .6 (tok 0), .3 (tok 1)      -> ids 1 (v .6), 2 (v .3)
#   layer 2, ctx 0:                   p = .45 (tok 0), .35 (tok 1)     -> ids 3 (.27), 4 (.21)
#   layer 2, ctx 1:                   p = .75 (tok 1), .2 (tok 0)      -> ids 5 (.225), 6 (.06)
#   layer 3, ctx 0:                   p = .85 (tok 0), .1 (tok 1)      -> ids 7 (.2295), 8 (.027)
#   layer 4, ctx 0:                   p = .6 (tok 0), .3 (tok 1)       -> ids 11 (.1377), 12 (.06885)
# (v = linear path value = product of confidences; with K = W = 2 layer d >= 2 owns ids
# base(d) = 3, 7, 11, ..., slot f's child of rank r is base + 2 f + r.)
CAST_DRAFT = {(1, 2): {0: .6, 1: .3}, (2, 0): {0: .45, 1: .35}, (2, 1): {1: .75, 0: .2},
              (3, 0): {0: .85, 1: .1}, (4, 0): {0: .6, 1: .3}}
# Target rows: the draft rows, and after the layer-4 node (depth 4, token 0) a row whose argmax is 2.
CAST_TARGET = {**CAST_DRAFT, (5, 0): {2: .5}}


def cast_cfg():
    # Cost tables on L = 2 (select row = min(floor(c / 2), 2)), N_cols = 8, S_T[r][0] = 1 so that
    # the width cost of k nodes is c_k = S_D[row][k - 1]:
    #   row 0 and row 2: S_D flat (c_2 = c_1: a second node is free);
    #   row 1: S_D = 1 + 9 (n - 1) (c_2 - c_1 = 9: a second node needs utility >= 9 C1 = 2.7,
    #   more than any probability, so the width is 1).
    # S_T row 0 = 1 + 0.1 (n - 1): the verify count keeps adding nodes while their mean linear
    # value is >= 0.1 C3 = 0.1.
    n = np.arange(1, 9, dtype=float)
    S_T = np.ones((3, 8))
    S_T[0] = 1.0 + 0.1 * (n - 1)
    S_D = np.ones((3, 8))
    S_D[1] = 1.0 + 9.0 * (n - 1)
    cast = dict(S_T=S_T, S_D=S_D, L=2.0, n0=0, C1=0.3, C2=0.15, C3=1.0, R=3, width_cap=2, m_cap=8, D_max=6)
    return dict(policy="cast", B=1, K=2, W=2, D=6, k=2, m=8, m_cap=8, P=9, D_path=7, T=0, seed=0, cast=cast)


def run_cast(run_round=oround.run_round):
    draft, target = rows_from(CAST_DRAFT), rows_from(CAST_TARGET)
    return run_round(cast_cfg(), np.array([2]), draft, target)


def test_cast_round_composition_by_hand():
    """Layer by layer (C1 = 0.3, C2 = 0.15, R = 3, n0 = 0):

    d=1: context 0 -> row 0 (flat): n1 = 2. FIFO {1}; key = 1 * u_2 / c_2 = .9 / 1 >= .15: grow.
    d=2: context 0 + 2 = 2 -> row 1 (steep): n2 = 1 (marginal .225 / 9 < .3). u_1 = .27; push
         .27 / .9 = .3 -> FIFO {1, .3}, mean .65; key = .65 * .27 / 1 = .1755: grow.
    d=3: context 3 -> row 1: n3 = 1. u_1 = .2295; push .2295 / .27 = .85 -> {1, .3, .85}, mean
         .71667; key = .164475: grow.
    d=4: context 4 -> row 2 (flat): n4 = 2. u_2 = .1377 + .06885 = .20655; push .20655 / .2295 = .9
         -> {1, .3, .85, .9}, the oldest dropped (R = 3) -> {.3, .85, .9}, mean .68333;
         key = .68333 * .20655 / 1 = .14114 < .15: stop at depth 4 (< D_max = 6).
    Verify count on all 10 nodes, sorted linear values .6 .3 .27 .2295 .225 .21 .1377 | .06885 .06
    .027, cap m_cap = 8, cost row 0: every node down to .1377 is worth >= .1, the 8th (.06885) is
    not: m = 7 -> selected ids 1 2 3 4 5 7 11.
    Greedy verify: root -> tok 0 (pos 1) -> tok 0 (pos 3, id 3) -> tok 0 (pos 6, id 7) -> tok 0
    (pos 7, id 11), whose target argmax is 2: accept 4, bonus 2.
    """
    ref = run_cast()
    t = ref["tree"]
    assert ref["widths"] == [2, 1, 1, 2]
    assert ref["depth"] == 4 and t.cur_depth == 4
    assert ref["m"] == 7
    assert list(ref["selected"][0][:7]) == [1, 2, 3, 4, 5, 7, 11] and ref["selected"][0][7] == -1
    lin = {i: math.exp(t.value[0, i]) for i in t.nodes(0)}
    want = {1: .6, 2: .3, 3: .27, 4: .21, 5: .225, 6: .06, 7: .2295, 8: .027, 11: .1377, 12: .06885}
    assert set(lin) == set(want)
    for i, v in want.items():
        assert math.isclose(lin[i], v, rel_tol=1e-12), (i, lin[i], v)
    meta = ref["meta"]
    assert int(meta["n_pos"][0]) == 8
    assert list(meta["tokens"][0]) == [2, 0, 1, 0, 1, 1, 0, 0, -1]
    assert list(meta["parents"][0]) == [-1, 0, 0, 1, 1, 2, 3, 6, -1]
    assert int(ref["accept_len"][0]) == 4 and int(ref["bonus"][0]) == 2
    assert list(ref["accept_path"][0]) == [0, 1, 3, 6, 7, -1, -1]


def test_cast_round_fifo_contents_by_hand(monkeypatch):
    """The FIFO after every pruned layer, read through the state object (same derivation)."""
    seen = []
    real = ocast.width_depth

    def spy(tree, d, state, p, gaps=None):
        out = real(tree, d, state, p, gaps)
        seen.append((d, list(state.fifo), state.ctx_sum))
        return out
    monkeypatch.setattr(oround.cast_mod, "width_depth", spy)
    run_cast()
    assert [s[0] for s in seen] == [1, 2, 3, 4]
    assert [s[2] for s in seen] == [2, 3, 4, 6]               # n0 + widths so far
    for (d, fifo, _), want in zip(seen, [[1.0], [1.0, .3], [1.0, .3, .85], [.3, .85, .9]]):
        assert len(fifo) == len(want) and all(math.isclose(a, b, rel_tol=1e-12) for a, b in zip(fifo, want)), d


def test_cast_round_planted_mistakes_fail():
    # (1) the context is not accumulated: every layer reads cost row 0 (flat) -> width 2 at layer 2
    wd = mutated(ocast.width_depth, 'p["n0"] + state.ctx_sum', 'p["n0"]')
    rr = mutated(oround.run_round, "cast_mod.width_depth(", "_wd(", {"_wd": wd})
    assert run_cast(rr)["widths"] != [2, 1, 1, 2]
    # (2) the verify count taken on the tree as it was before the last layer: m = 6
    rr = mutated(oround.run_round, [("        d = expand()\n\n    if policy",
                                     "        _snap = copy.deepcopy(tree)\n        d = expand()\n\n    if policy"),
                                    ("cast_mod.verify_count(tree,", "cast_mod.verify_count(_snap,")],
                 extra_globals={"copy": copy})
    assert run_cast(rr)["m"] == 6
    # (3) the FIFO keeps every ratio (R ignored): mean(1, .3, .85, .9) * .20655 = .1523 >= .15, so
    # layer 5 is built
    wd = mutated(ocast.width_depth, 'while len(state.fifo) > p["R"]', "while False")
    rr = mutated(oround.run_round, "cast_mod.width_depth(", "_wd(", {"_wd": wd})
    assert run_cast(rr)["depth"] == 5


# ----------------------------------------------------------------------------- Graft ----
# Draft rows as in the CAST round (layers 1-2). Target rows depend on the context token only:
#   ctx 2 -> argmax 1, ctx 1 -> argmax 2, ctx 0 -> argmax 0 (each p = .5 on that token).
GRAFT_TARGET = {2: {1: .5}, 1: {2: .5}, 0: {0: .5}}


def graft_cfg():
    graft = dict(ckpt_layers=[0, 1, 5], tau=[0.5, 0.5, 0.2], k_draft=[1, 8, 9], K_total=10,
                 template=default_template(2, 3))
    return dict(policy="graft", B=1, K=2, W=2, D=8, k=2, m=10, m_cap=10, P=11, D_path=10, T=0, seed=0,
                graft=graft)


def graft_M():
    M = np.full((1, V, 8), -1, np.int64)
    M[0, 2] = [1, 0, 5, 5, 5, 5, 5, 5]      # successors of the root token 2
    M[0, 1] = [2, 3, 3, 3, 3, 3, 3, 3]      # successors of token 1; token 0 has none
    return M


def run_graft(run_round=oround.run_round):
    draft = rows_from(CAST_DRAFT)

    def target(b, d, ctx):
        return prow(GRAFT_TARGET[ctx])
    M = graft_M()
    ref = run_round(graft_cfg(), np.array([2]), draft, target, M=M)
    ref["M_after"] = M
    return ref


def test_graft_round_composition_by_hand():
    """Checkpoint d0 (layer 1): c = exp(max value) = .6 > .5 passes. Checkpoint d1 (layer 2): .27 is
    not > .5: stop with stage 1 and budget K_draft[1] = 8. The tree has only 6 nodes, so all 6 are
    selected and K_ret = K_max - 6 = 4 template nodes are grafted, breadth first over 2 chains of
    depth 3: M[2][0] = 1, M[2][1] = 0, then M[1][0] = 2 below the first and M[0][0] = unset below
    the second (padding, token -1). Positions: root, ids 1..6, then the 4 grafted nodes: 11.
    Greedy: root argmax 1 matches pos 2 (id 2) and pos 7 (grafted); below pos 7 the argmax of
    token 1's row is 2, which is pos 9: accept 2 along [0, 7, 9], bonus = argmax after token 2 = 1.
    M refresh: every position's top-8 target ids into M[its token], the highest position last:
    M[2] <- row of ctx 2 = [1, 0, 2, 3, 4, 5, 6, 7], M[0] <- [0, 1, ..., 7], M[1] <- [2, 0, 1, 3, ...].
    """
    ref = run_graft()
    assert ref["stage"] == [1] and ref["m_sel"] == [8] and ref["depth"] == 2
    assert int(np.sum(ref["selected"][0] >= 0)) == 6
    toks, pars, anchor = ref["retrieved"][0]
    assert toks == [1, 0, 2, -1] and pars == [-1, -1, 0, 1] and anchor == 0
    meta = ref["meta"]
    assert int(meta["n_pos"][0]) == 11
    assert list(meta["tokens"][0]) == [2, 0, 1, 0, 1, 1, 0, 1, 0, 2, -1]
    assert list(meta["parents"][0]) == [-1, 0, 0, 1, 1, 2, 2, 0, 0, 7, 8]
    assert list(meta["depth"][0]) == [0, 1, 1, 2, 2, 2, 2, 1, 1, 2, 2]
    assert int(ref["accept_len"][0]) == 2 and int(ref["bonus"][0]) == 1
    assert list(ref["accept_path"][0][:4]) == [0, 7, 9, -1]
    M = ref["M_after"]
    assert list(M[0, 2]) == [1, 0, 2, 3, 4, 5, 6, 7]
    assert list(M[0, 0]) == [0, 1, 2, 3, 4, 5, 6, 7]
    assert list(M[0, 1]) == [2, 0, 1, 3, 4, 5, 6, 7]
    assert (M[0, 3:] == -1).all()


def test_graft_round_planted_mistakes_fail():
    # K_ret from the budget (K_max - 8 = 2 grafted nodes) instead of the selected count
    rr = mutated(oround.run_round, "K_total - int(np.sum(selected[b] >= 0))", "K_total - m_sel[b]")
    assert int(run_graft(rr)["meta"]["n_pos"][0]) == 9
    # the checkpoint applied one layer late (d1 tested on layer 3): the round grows past layer 2
    rr = mutated(oround.run_round, "graft_mod.checkpoint(tree, d, ", "graft_mod.checkpoint(tree, d - 1, ")
    assert run_graft(rr)["depth"] != 2


# ----------------------------------------------------------------------------- EAGLE ----
EAGLE_DRAFT = {**CAST_DRAFT, (3, 1): {2: .5, 0: .3}, (4, 0): {1: .6}}


def eagle_cfg():
    return dict(policy="eagle", B=1, K=2, W=2, D=3, k=2, m=5, m_cap=5, P=6, D_path=4, T=0, seed=0)


def run_eagle(run_round=oround.run_round):
    return run_round(eagle_cfg(), np.array([2]), rows_from(EAGLE_DRAFT), rows_from(EAGLE_DRAFT))


def test_eagle_round_stops_at_depth_by_hand():
    """k = 2, D = 3, m = 5. Layer 2 values .27 (id 3) .225 (id 5) .21 (id 4) .06 (id 6): the
    frontier of layer 3 is ids 3 and 5 (slots in id order). Layer 3: slot 0 (ctx 0) gives ids 7
    (.2295) and 8 (.027); slot 1 (ctx 1, p = .5 on 2, .3 on 0) gives ids 9 (.1125) and 10 (.0675).
    Depth 3 = D: stop. Top-5: .6 (1) .3 (2) .27 (3) .2295 (7) .225 (5) -> ids 1 2 3 5 7.
    Greedy (target = draft rows): 0 -> pos 1 (tok 0) -> pos 3 (id 3) -> pos 5 (id 7); after it the
    layer-4 row's argmax is 1: accept 3, bonus 1."""
    ref = run_eagle()
    t = ref["tree"]
    assert ref["depth"] == 3
    assert list(t.frontier[0]) == [3, 5]
    assert [int(t.token[0, i]) for i in (7, 8, 9, 10)] == [0, 1, 2, 0]
    assert math.isclose(math.exp(t.value[0, 9]), .1125, rel_tol=1e-12)
    assert list(ref["selected"][0]) == [1, 2, 3, 5, 7]
    assert list(ref["meta"]["tokens"][0]) == [2, 0, 1, 0, 1, 0]
    assert int(ref["accept_len"][0]) == 3 and int(ref["bonus"][0]) == 1
    assert list(ref["accept_path"][0]) == [0, 1, 3, 5]


def test_eagle_round_planted_mistakes_fail():
    # the depth stop one layer early
    rr = mutated(oround.run_round, "if d >= D:\n                stop = [True] * B",
                 "if d >= D - 1:\n                stop = [True] * B")
    assert run_eagle(rr)["depth"] == 2
    # the frontier by lowest id instead of by value: layer 3 expands ids 3 and 4
    rr = mutated(oround.run_round, "frontiers.append(tree.select_frontier(width, stop, gaps))",
                 "frontiers.append(tree.select_frontier(width, stop, gaps)); "
                 "tree.frontier = [sorted(tree.layer_ids(b, d))[:width] for b in range(B)]")
    ref = run_eagle(rr)
    assert list(ref["tree"].frontier[0]) == [3, 4]
    assert not math.isclose(math.exp(ref["tree"].value[0, 9]), .1125, rel_tol=1e-12)   # .21 * .5 instead
