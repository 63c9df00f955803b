"""Pins of the block-drafter Graft round in the oracle (``run_round`` with ``block``, tail-anchored
templates), CPU only.

Graft page, extension direction 1 (grafting for block drafters) and weakness 4 (token-level
confidence inside the block, templates fitted to the block): the block drafter's rows give a chain
(K = 1) or a chain with its top-K alternatives (K > 1); every block position can be a checkpoint;
the retrieval template may hang from the end of the kept block instead of the root. What fixes the
oracle here: (1) a round worked out by hand (comments); (2) brute force on random rows: the block
tree equals the chain of per-row argmaxes with cumulative log-softmax scores, and the stage equals
the first position whose exp(S_j) is not above tau_j; (3) planted mistakes that must fail.
"""
import math

import numpy as np
import pytest

import oracle.graft as ograft
import oracle.round as oround
import oracle.tree as otree
from oracle.graft import default_template
from test_oracle_round import V, mutated, prow

# Block rows (the same whatever the context: keyed on the root token 2):
#   row 1: tok 4 .8, tok 3 .1   -> layer 1: ids 1 (tok 4, .8), 2 (tok 3, .1)
#   row 2: tok 5 .7, tok 6 .2   -> layer 2 (children of id 1): ids 3 (tok 5, .56), 4 (tok 6, .16)
#   row 3: tok 7 .5, tok 8 .3   -> layer 3 (children of id 3): ids 5 (tok 7, .28), 6 (tok 8, .168)
#   row 4: tok 9 .9, tok 1 .05  -> never built
BLOCK = {1: {4: .8, 3: .1}, 2: {5: .7, 6: .2}, 3: {7: .5, 8: .3}, 4: {9: .9, 1: .05}}
# target rows by context token: the argmax successor of each (p = .5)
TARGET = {2: {4: .5}, 4: {5: .5}, 5: {7: .5}, 7: {3: .5}, 3: {1: .5}, 1: {0: .5}}


def block_cfg(anchor="tail", tau=(.5, .5, .3, .2), K=2, L=4, k_draft=(2, 4, 5, 8), K_total=9):
    graft = dict(ckpt_layers=list(range(L)), tau=list(tau), k_draft=list(k_draft), K_total=K_total,
                 template=default_template(2, 3), anchor=anchor)
    return dict(policy="graft", block=True, B=1, K=K, W=1, D=L, k=1, m=K_total, m_cap=K_total, P=K_total + 1,
                D_path=8, T=0, seed=0, graft=graft)


def block_M():
    M = np.full((1, V, 8), -1, np.int64)
    M[0, 7] = [3, 0, 6, 6, 6, 6, 6, 6]   # successors of the tail token 7
    M[0, 3] = [1, 6, 6, 6, 6, 6, 6, 6]   # of token 3; token 0 has none
    M[0, 2] = [9, 9, 9, 9, 9, 9, 9, 9]   # of the root token 2
    return M


def run_block(cfg=None, run_round=oround.run_round):
    cfg = cfg or block_cfg()

    def draft(b, d, ctx):
        assert ctx == 2, "block rows are keyed on the root token"
        return prow(BLOCK[d])

    def target(b, d, ctx):
        return prow(TARGET.get(ctx, {0: .34, 1: .33}))
    return run_round(cfg, np.array([2]), draft, target, M=block_M())


def test_block_round_by_hand_tail_anchor():
    """Gates: .8 > .5, .56 > .5, then .28 is not > .3: stop at position 3 (stage 2), K_draft = 5; the
    top-5 of the 6 nodes by value are ids 1 3 4 5 6 (id 2, .1, is dropped). Tail: the deepest kept
    nodes are ids 5 (.28) and 6 (.168): id 5, token 7. K_ret = 9 - 5 = 4 template nodes: M[7][0] = 3,
    M[7][1] = 0, M[3][0] = 1 below the first, M[0][0] unset below the second. Positions: root, ids
    1 3 4 5 6, then the four grafted nodes hanging from position 4 (id 5). Greedy: 4, 5, 7, then the
    grafted 3 and 1: accept 5 along [0, 1, 2, 4, 6, 8], bonus = argmax after token 1 = 0."""
    ref = run_block()
    assert ref["stage"] == [2] and ref["m_sel"] == [5] and ref["depth"] == 3
    assert [int(x) for x in ref["selected"][0] if x >= 0] == [1, 3, 4, 5, 6]
    toks, pars, anchor = ref["retrieved"][0]
    assert anchor == 5 and toks == [3, 0, 1, -1] and pars == [-1, -1, 0, 1]
    meta = ref["meta"]
    assert int(meta["n_pos"][0]) == 10
    assert list(meta["tokens"][0]) == [2, 4, 5, 6, 7, 8, 3, 0, 1, -1]
    assert list(meta["parents"][0]) == [-1, 0, 1, 1, 2, 2, 4, 4, 6, 7]
    assert list(meta["depth"][0]) == [0, 1, 2, 2, 3, 3, 4, 4, 5, 5]
    assert int(ref["accept_len"][0]) == 5 and int(ref["bonus"][0]) == 0
    assert list(ref["accept_path"][0][:7]) == [0, 1, 2, 4, 6, 8, -1]
    t = ref["tree"]
    for i, want in [(1, .8), (3, .56), (5, .28), (6, .168), (4, .16), (2, .1)]:
        assert math.isclose(math.exp(t.value[0, i]), want, rel_tol=1e-12)


def test_block_round_by_hand_root_anchor():
    """The same round with the template at the root: M[2] gives token 9 twice, the graft hangs from
    position 0, and acceptance stops after token 7 (no children): accept 3, bonus 3."""
    ref = run_block(block_cfg(anchor="root"))
    toks, pars, anchor = ref["retrieved"][0]
    assert anchor == 0 and toks == [9, 9, -1, -1]
    assert list(ref["meta"]["parents"][0]) == [-1, 0, 1, 1, 2, 2, 0, 0, 6, 7]
    assert int(ref["accept_len"][0]) == 3 and int(ref["bonus"][0]) == 3


def test_block_round_without_a_failing_gate_keeps_k_total():
    """All gates pass (tau 0): all four layers are built, stage = n_ckpt, K_draft = K_total = 9 of
    the 8 nodes (all of them), K_ret = 1; the tail is layer 4's top node (token 9)."""
    ref = run_block(block_cfg(tau=(0, 0, 0, 0)))
    assert ref["stage"] == [4] and ref["m_sel"] == [9] and ref["depth"] == 4
    toks, pars, anchor = ref["retrieved"][0]
    assert anchor == 7 and len(toks) == 1  # layer 4 = ids 7, 8; id 7 holds token 9


def test_block_planted_mistakes_fail():
    # (1) tail tie-break reversed (value ascending): id 6 (token 8) becomes the anchor
    ta = mutated(ograft.tail_anchor, "tree.value[b, i], -i) > (tree.depth[b, best], tree.value[b, best], -best)",
                 "-tree.value[b, i], -i) > (tree.depth[b, best], -tree.value[b, best], -best)")
    rr = mutated(oround.run_round, "graft_mod.tail_anchor(", "_ta(", {"_ta": ta})
    assert run_block(run_round=rr)["retrieved"][0][2] == 6
    # (2) grafted nodes attached to the root whatever the anchor
    bm = mutated(otree.build_meta, "par = pos_of[anchor] if rp[u] < 0", "par = 0 if rp[u] < 0")
    rr = mutated(oround.run_round, "meta = build_meta(", "meta = _bm(", {"_bm": bm})
    assert list(run_block(run_round=rr)["meta"]["parents"][0][6:8]) == [0, 0]
    # (3) block rows keyed on the picked token (a per-layer drafter): the draft callback refuses
    rr = mutated(oround.run_round, "draft_row(b, d, int(roots[b]))",
                 "draft_row(b, d, int(tree.token[b, tree.frontier[b][f]]))")
    with pytest.raises(AssertionError):
        run_block(run_round=rr)


@pytest.mark.parametrize("seed", range(8))
def test_block_tree_is_the_argmax_chain_brute_force(seed):
    """Random block rows: layer j's top node is argmax(row j) (first on ties), its score is the sum of
    log softmax(row i)[argmax] over i <= j, and the alternatives of layer j hang from it; the stage
    is the first position whose exp(S_j) is not above tau_j (tau drawn around the chain's scores)."""
    rng = np.random.default_rng(seed)
    L, K, Vb = 6, 3, 12
    rows = rng.normal(0, 1.5, (L + 1, Vb))
    rows[2, :3] = rows[2].max() + 0.5  # a three-way tie at the top of row 2
    lsm = rows - np.log(np.sum(np.exp(rows - rows.max(1, keepdims=True)), 1, keepdims=True)) - rows.max(1, keepdims=True)
    chain = [int(np.argmax(rows[j])) for j in range(1, L + 1)]
    S = np.cumsum([lsm[j, chain[j - 1]] for j in range(1, L + 1)])
    tau = np.exp(S) * rng.choice([0.5, 1.5], L, p=[0.8, 0.2])
    fail = [j for j in range(L) if not (math.exp(S[j]) > tau[j])]
    want_stage = fail[0] if fail else L
    K_total = K * L
    cfg = dict(policy="graft", block=True, B=1, K=K, W=1, D=L, k=1, m=K_total, m_cap=K_total, P=K_total + 1,
               D_path=L + 2, T=0, seed=0,
               graft=dict(ckpt_layers=list(range(L)), tau=list(tau), k_draft=[K * (j + 1) for j in range(L)],
                          K_total=K_total, template=default_template(2, 2), anchor="tail"))
    M = np.full((1, Vb, 8), -1, np.int64)
    ref = oround.run_round(cfg, np.array([0]), lambda b, d, ctx: rows[d],
                           lambda b, d, ctx: rows[0], M=M)
    t = ref["tree"]
    assert ref["stage"] == [want_stage]
    built = want_stage + 1 if want_stage < L else L
    assert ref["depth"] == built
    for j in range(1, built + 1):
        ids = t.layer_ids(0, j)
        top = min(ids, key=lambda i: (-t.value[0, i], i))
        assert int(t.token[0, top]) == chain[j - 1]
        assert math.isclose(t.value[0, top], S[j - 1], rel_tol=1e-12, abs_tol=1e-12)
        parent_want = 0 if j == 1 else min(t.layer_ids(0, j - 1), key=lambda i: (-t.value[0, i], i))
        assert all(int(t.parent[0, i]) == parent_want for i in ids)
        alt = sorted(range(Vb), key=lambda v: (-rows[j, v], v))[:K]
        assert sorted(int(t.token[0, i]) for i in ids) == sorted(alt)
    # the tail anchor is the deepest kept chain node
    anchor = ref["retrieved"][0][2]
    assert int(t.depth[0, anchor]) == max(int(t.depth[0, i]) for i in ref["selected"][0] if i >= 0)
