"""Graft prune-then-graft: confidence checkpoints, retrieval from M, M refresh (test infrastructure only).

Source: "Draft Less, Retrieve More: Hybrid Tree Construction for Speculative
Decoding", the three-step method description:

(1) prune: S_{d,j} = S_{d-1,F(j)} + log q(...), c_d = exp(max_j S_{d,j}),
    g_d = 1[c_d > tau_d]; the first failing checkpoint truncates the tree; the
    stage s fixes K_draft^s (8/24/40 at checkpoints d0/d1/d5) and
    K_ret^s = K_max - K_draft^s slots go to retrieval;
(2) graft: starting from the root token x_t, x_u = M[x_{F(u)}, r_u] over a
    stage-adaptive template G_ret^s, cut to K_ret^s nodes;
(3) verify the K_max-token hybrid tree with the standard rule, then for every
    verified token refresh its row of M with the top-k successors of the
    target's next-token distribution at that position.

Readings taken where the page is silent or garbled:

* Checkpoints d0/d1/d5 are layer indices 0, 1, 5, i.e. draft layers 1, 2, 6
  of the D_E = 8 layer base tree; the test is strict ">" as printed; it is
  per request. Without a failing checkpoint K_draft = K_max = 60.
* The kept draft nodes are the top-K_draft of the truncated tree in the total
  order (``OracleTree.rerank``).
* Template (parity unpinned: its shape came from a grid search the page does
  not print): 8 chains; level 1 is M[x_t][0..7]; every chain continues with
  rank 0 down to depth 8 (64 nodes); the first K_ret nodes in breadth-first
  (level, chain) order are used.
* A node whose parent token is invalid, or whose M entry is unset (-1), is an
  invalid node (token -1) that still occupies its slot, so |T| = K_max.
* M is one matrix per request, starts all -1, and is refreshed for every
  used position with a valid token (root included), in increasing position,
  so the highest position wins when a token repeats.

Block drafters (the page's extension direction 1, Grafting for block drafters,
and weakness 4, whose remedy is token-level confidence inside the block and
templates fitted to the block's topology). Readings:

* A block drafter gives in one pass one row per block position j = 1..L
  (L = 16 for DFlash), its distribution for the token at j; the rows do not
  depend on the tokens picked at earlier positions of the block.
* Block tree: layer j holds the top-K tokens of row j, children of the block's
  token at position j - 1 (the root for j = 1); the block's token at j is the
  top-1 of row j. K = 1 is the plain block (a chain); K > 1 adds the top-K
  alternatives at every position (the "tree-shaped expansion inside the
  block"). This is the EAGLE-2 expansion with frontier width 1 fed with the
  block's rows, since the highest-value node of a layer is the top-1 child of
  the block token above it.
* Token-level pruning: every block position can be a checkpoint, with the
  rule of step (1): S_j is the block path's score at j, the first position
  whose exp(S_j) is not above tau_j truncates the block after layer j.
* Templates: root-anchored (step (2), template root = x_t) or tail-anchored
  (the page contrasts G_ret^root and G_ret^tail): the template root is the
  deepest kept draft node, ties broken by the total order (value desc, id
  asc), i.e. the end of the kept block prefix; level-1 template nodes become
  its children.
"""

import numpy as np


def checkpoint(tree, d, p, stop, stage, m):
    """Apply the checkpoint test after layer d was built; updates stop/stage/m in place.

    ``p`` holds ckpt_layers (layer indices), tau, k_draft, K_total, D_max.
    """
    for b in range(tree.B):
        if stop[b]:
            continue
        li = d - 1
        if li in p["ckpt_layers"]:
            s = p["ckpt_layers"].index(li)
            ids = tree.layer_ids(b, d)
            c = float(np.exp(max(tree.value[b, i] for i in ids))) if ids else 0.0
            if p.get("gaps") is not None:
                p["gaps"].add("tau", c - p["tau"][s], c, b)
            if not (c > p["tau"][s]):
                stop[b], stage[b], m[b] = True, s, p["k_draft"][s]
                continue
        if d >= p["D_max"]:
            stop[b], stage[b], m[b] = True, len(p["ckpt_layers"]), p["K_total"]


def default_template(width=8, depth=8):
    """Chain template: level 1 = ranks 0..width-1 of the root's row, then rank 0 downwards.

    Returned in breadth-first (level, chain) order as (parent, rank) lists;
    parent -1 is the root. Parity unpinned (shape not printed on the page).
    """
    parent, rank = [], []
    for lvl in range(1, depth + 1):
        for ch in range(width):
            if lvl == 1:
                parent.append(-1)
                rank.append(ch)
            else:
                parent.append((lvl - 2) * width + ch)
                rank.append(0)
    return parent, rank


def tail_anchor(tree, selected_b, b):
    """The deepest kept draft node of request b (ties: value desc, then id asc); 0 (the root) when
    no draft node is kept."""
    best = 0
    for i in (int(x) for x in selected_b if x >= 0):
        if (tree.depth[b, i], tree.value[b, i], -i) > (tree.depth[b, best], tree.value[b, best], -best):
            best = i
    return best


def retrieve(M, root_tokens, k_ret, template):
    """Gather the first k_ret[b] template nodes from M[b], the template root's token being
    root_tokens[b] (the root's, or the anchor node's); returns per-request (tokens, parents)."""
    parent, rank = template
    out = []
    for b in range(len(root_tokens)):
        n = max(0, min(int(k_ret[b]), len(parent)))
        toks, pars = [], []
        for u in range(n):
            pt = root_tokens[b] if parent[u] < 0 else toks[parent[u]]
            t = -1 if pt < 0 else int(M[b][pt][rank[u]])
            toks.append(t)
            pars.append(parent[u])
        out.append((toks, pars))
    return out


def adj_update(M, meta, top8):
    """Refresh M rows from the verified positions' top-8 target successors (in place)."""
    B = meta["tokens"].shape[0]
    for b in range(B):
        for i in range(int(meta["n_pos"][b])):
            t = int(meta["tokens"][b, i])
            if t >= 0:
                M[b][t][:] = top8[b, i]
    return M
