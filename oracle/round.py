"""One draft-tree round end to end in the oracle (test infrastructure only).

Order of steps (EAGLE-2 page, §"一段更贴近实现的流程"; CAST page, §关键设计 2-4;
Graft page, steps (1)-(3)):

  layer 1 from the root row; for each further layer: prune decision (CAST
  width/depth or Graft checkpoint), frontier top-w, expand; then the verify
  budget (CAST), rerank, retrieval graft (Graft), flatten + metadata, verify,
  and the M refresh (Graft).

The logits come from callables supplied by the caller:
``draft_row(b, depth, ctx_token)`` is the draft model's row for a node whose
children land in layer ``depth``; ``target_row(b, depth, ctx_token)`` is the
target's next-token row after a tree position at depth ``depth - 1``.
"""

import numpy as np

from . import cast as cast_mod
from . import graft as graft_mod
from . import sampled as sampled_mod
from .tree import OracleTree, Gaps, build_meta
from .verify import verify_greedy, verify_sample, row_top8


def run_round(cfg, roots, draft_row, target_row, rnd=0, M=None, pos_offset=None, gaps=None):
    """Run one round. ``cfg`` keys: policy ('eagle'|'cast'|'graft'), B, K, W, D, m_cap,
    P, D_path, T (0|1), seed, plus the policy's parameters. Returns a dict of outputs."""
    B, K, W, D = cfg["B"], cfg["K"], cfg["W"], cfg["D"]
    gaps = gaps if gaps is not None else Gaps()
    tree = OracleTree(B, K, W, D, roots)
    policy = cfg["policy"]
    stop = [False] * B
    stage = [-1] * B
    m_req = [cfg["m_cap"]] * B
    widths, cast_state = [], cast_mod.CastState()
    per_request = policy == "cast" and bool(cfg["cast"].get("per_request", False))
    cast_states = [cast_mod.CastState() for _ in range(B)]
    frontiers = []
    p_graft = None
    if policy == "graft":
        p_graft = dict(cfg["graft"], gaps=gaps, D_max=D)
    # block drafter (Graft page, extension direction 1): the row of layer d is the block's row for
    # position d, the same whatever tokens were picked above it; frontier width 1 (the block token)
    block = bool(cfg.get("block", False))
    # sampled drafts (EAGLE-2 page, the ledger of speculative sampling with drafted tokens drawn from
    # q): children drawn from the draft row without replacement, every drawn node verified
    draw = bool(cfg.get("draft_sampling", False))
    sampler = None
    if draw:
        if policy != "eagle" or cfg["T"] != 1:
            raise ValueError("sampled drafts: EAGLE-2 trees with T = 1 only")

        def sampler(b, node, x):
            return sampled_mod.sample_children(x, K, cfg["seed"], rnd, b, node, gaps)

    def expand():
        d = tree.cur_depth + 1
        if block:
            tree.expand_layer(lambda b, f: draft_row(b, d, int(roots[b])))
        else:
            tree.expand_layer(lambda b, f: draft_row(b, d, int(tree.token[b, tree.frontier[b][f]])), sampler)
        return d

    d = expand()
    while True:
        if policy == "cast" and per_request:  # every running request decides for itself
            width = [0] * B
            for b in range(B):
                if stop[b]:
                    continue
                n, grow = cast_mod.width_depth(tree, d, cast_states[b], cfg["cast"], gaps, reqs=[b])
                width[b] = n
                if not grow:
                    stop[b] = True
            widths.append(list(width))
        elif policy == "cast":
            n, grow = cast_mod.width_depth(tree, d, cast_state, cfg["cast"], gaps)
            widths.append(n)
            width = n
            if not grow:
                stop = [True] * B
        elif policy == "graft":
            graft_mod.checkpoint(tree, d, p_graft, stop, stage, m_req)
            width = 1 if block else cfg["k"]
        else:
            width = cfg["k"]
            if d >= D:
                stop = [True] * B
        if all(stop) or d >= D:
            break
        frontiers.append(tree.select_frontier(width, stop, gaps))
        d = expand()

    if policy == "cast" and per_request:
        m_sel = [cast_mod.verify_count(tree, cfg["cast"], gaps, reqs=[b]) for b in range(B)]
        m = list(m_sel)
    elif policy == "cast":
        m = cast_mod.verify_count(tree, cfg["cast"], gaps)
        m_sel = [m] * B
    elif policy == "graft":
        m_sel = m_req
        m = None
    elif draw:  # every drawn node (dropping drawn nodes by value is not lossless)
        m_sel = [len(tree.nodes(b)) for b in range(B)]
        m = None
    else:
        m = cfg["m"]
        m_sel = [m] * B
    selected = tree.rerank(m_sel, cfg["m_cap"], None if draw else gaps)

    retrieved = None
    if policy == "graft":
        K_total = cfg["graft"]["K_total"]
        k_ret = [K_total - int(np.sum(selected[b] >= 0)) for b in range(B)]
        if cfg["graft"].get("anchor", "root") == "tail":
            anchors = [graft_mod.tail_anchor(tree, selected[b], b) for b in range(B)]
        else:
            anchors = [0] * B
        retrieved = graft_mod.retrieve(M, [int(tree.token[b, a]) for b, a in enumerate(anchors)], k_ret,
                                       cfg["graft"]["template"])
        retrieved = [(t, p, a) for (t, p), a in zip(retrieved, anchors)]
    if pos_offset is None:
        pos_offset = np.zeros(B, np.int64)
    meta = build_meta(tree, selected, pos_offset, cfg["P"], cfg["D_path"], retrieved)

    def trow(b, i):
        return target_row(b, int(meta["depth"][b, i]) + 1, int(meta["tokens"][b, i]))

    if cfg["T"] == 0:
        acc, path, bonus = verify_greedy(meta, trow)
    elif draw:
        acc, path, bonus = sampled_mod.verify_tree(tree, meta, lambda b, i: trow(b, i), cfg["seed"], rnd, gaps)
    else:
        acc, path, bonus = verify_sample(meta, trow, cfg["seed"], rnd, gaps)
    top8 = None
    if policy == "graft":
        top8 = row_top8(meta, trow)
        graft_mod.adj_update(M, meta, top8)
    return dict(tree=tree, selected=selected, meta=meta, accept_len=acc, accept_path=path,
                bonus=bonus, widths=widths, m=m, m_sel=m_sel, stage=stage, retrieved=retrieved,
                top8=top8, frontiers=frontiers, gaps=gaps, depth=tree.cur_depth)
