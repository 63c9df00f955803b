"""EAGLE-2 dynamic draft tree, restated step by step in fp64 (test infrastructure only).

Source: "EAGLE-2 完全拆解：动态草稿树如何让投机解码上下文感知",
§"置信度为什么可以近似接受率" (confidence = draft probability of the token),
§"value 公式" (V_i = product of confidences along the root path),
§"扩展阶段" (expand the top-k newest-layer nodes by value; value(child) =
value(parent) * confidence(child)), §"重排阶段" (top-m over all nodes, shallow
first on ties, connected subtree, flatten + ancestor-only mask), and the
implementation flow in §"一段更贴近实现的流程".

Readings taken where the page is silent:

* Values are kept in log form, root value 0, value = sum of log c on the path
  (Graft's page writes the same score as S_d = S_{d-1} + log q).
* Confidence c is the softmax probability of the token in its draft row
  (temperature 1). Per-node top-K is taken on the raw logits (softmax is
  monotone, so the set is the same); equal logits go to the lower token id.
* Total order on nodes: value descending, then depth ascending, then node id
  ascending. Node ids grow with depth (layout below), so depth-then-id is
  simply id ascending.
* Layer 1 expands the root; layer d >= 2 expands the frontier, i.e. the
  top-w nodes of layer d-1 in the total order (w = k for EAGLE-2, n_{d-1}
  for CAST). Frontier slots are numbered in ascending node id, so only the
  frontier *set* matters, not the order inside it.
* Flattening: position 0 is the root, then the selected nodes in ascending
  node id (a topological order), then retrieved nodes (Graft) in template
  order.
* Padding-free target rows (CAST page §局限与展望 names padded batches as a
  limit): request b's used positions take consecutive rows after those of
  requests 0..b-1, in position order (``packed_row_offsets``).

Node-id layout (an interface format: the GPU path writes the same layout from
its own code): with K = per-node top-K, W = maximum frontier width and D =
maximum number of draft layers, layer 1 owns ids 1..K and layer d >= 2 owns
ids base(d) .. base(d)+W*K-1 with base(d) = 1 + K + (d-2)*W*K. The child of
rank r of frontier slot f in layer d has id base(d) + f*K + r.
"""

import numpy as np

NEG_INF = float("-inf")


class Gaps:
    """Distances of the oracle's values from every decision boundary of a round.

    The harness redraws a round whose smallest gap falls below the tolerance,
    so that fp32 rounding on the GPU cannot flip a decision the oracle takes
    with a visible margin.
    """

    def __init__(self):
        self.items = []

    def add(self, kind, gap, key, b=None):
        """Record a decision's distance from its boundary; ``b`` is the request (None: batch-wide)."""
        self.items.append((kind, float(gap), float(key), b))

    def near_tie(self, tol=1e-5):
        return [it for it in self.items if abs(it[1]) < tol * max(1.0, abs(it[2]))]


def layer_base(d, K, W):
    return 1 if d == 1 else 1 + K + (d - 2) * W * K


def layer_width(d, K, W):
    return K if d == 1 else W * K


def n_nodes(K, W, D):
    return 1 + K + (D - 1) * W * K


def row_softmax_topk(x, K):
    """Softmax statistics and the top-K tokens of one draft (or target) row.

    c_v = exp(x_v - m) / sum_u exp(x_u - m), m = max_u x_u.  Returns the K
    token ids ordered by (logit descending, id ascending), their log c, m and
    log S.  A row with NaN or +inf, or without any finite entry, is rejected.
    """
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any() or np.isposinf(x).any():
        raise ValueError("row holds NaN or +inf")
    m = x.max()
    if not np.isfinite(m):
        raise ValueError("row has no finite logit")
    S = np.exp(x - m).sum()
    order = np.lexsort((np.arange(x.size), -x))[:K]
    logS = np.log(S)
    logc = (x[order] - m) - logS
    return order.astype(np.int64), logc, m, logS


def total_order_key(value, node_id):
    """Sort key for the total order: value descending, then id ascending."""
    return (-value, node_id)


class OracleTree:
    """Per-request draft trees in the shared node-id layout, fp64 scores."""

    def __init__(self, B, K, W, D, root_tokens):
        self.B, self.K, self.W, self.D = B, K, W, D
        self.N = n_nodes(K, W, D)
        self.token = np.full((B, self.N), -1, np.int64)
        self.parent = np.full((B, self.N), -1, np.int64)
        self.depth = np.zeros((B, self.N), np.int64)
        self.logc = np.full((B, self.N), NEG_INF)
        self.value = np.full((B, self.N), NEG_INF)
        for d in range(1, D + 1):
            base = layer_base(d, K, W)
            self.depth[:, base:base + layer_width(d, K, W)] = d
        self.token[:, 0] = np.asarray(root_tokens, dtype=np.int64)
        self.logc[:, 0] = 0.0
        self.value[:, 0] = 0.0
        self.cur_depth = 0
        self.frontier = [[0] for _ in range(B)]      # layer 1 expands the root
        self.layer_sorted = [dict() for _ in range(B)]
        self.draft_row = [dict() for _ in range(B)]  # sampled drafts: node -> the row its children came from

    # -- helpers ---------------------------------------------------------------
    def valid(self, b, i):
        return self.token[b, i] >= 0

    def layer_ids(self, b, d):
        base = layer_base(d, self.K, self.W)
        ids = range(base, base + layer_width(d, self.K, self.W))
        return [i for i in ids if self.valid(b, i)]

    def nodes(self, b):
        """All valid non-root node ids of request b."""
        return [i for i in range(1, self.N) if self.valid(b, i)]

    def sorted_nodes(self, b, ids):
        return sorted(ids, key=lambda i: total_order_key(self.value[b, i], i))

    def path(self, b, i):
        out = []
        while i >= 0:
            out.append(i)
            i = self.parent[b, i] if i != 0 else -1
        return out[::-1]

    # -- expansion (a1 + a2) ---------------------------------------------------
    def expand_layer(self, rows, sampler=None):
        """Expand the current frontier into layer d = cur_depth + 1.

        ``rows`` is an array [B][F][V] of logits, or a callable (b, f) -> row;
        row f of request b is the draft row of frontier slot f. With ``sampler``
        (sampled drafts, ``oracle.sampled``), sampler(b, node, row) gives the
        node's children in draw order (at most K; missing ones stay invalid)
        instead of the top-K, and each expanded node keeps its row.
        """
        d = self.cur_depth + 1
        if d > self.D:
            raise ValueError("tree is already at maximum depth")
        K = self.K
        base = layer_base(d, K, self.W)
        for b in range(self.B):
            for f, pid in enumerate(self.frontier[b]):
                row = rows(b, f) if callable(rows) else rows[b][f]
                toks, logc, m, logS = row_softmax_topk(row, K)
                if sampler is not None:
                    x = np.asarray(row, dtype=np.float64)
                    toks = np.asarray(sampler(b, pid, x), dtype=np.int64)[:K]
                    logc = (x[toks] - m) - logS
                    self.draft_row[b][pid] = x
                for r in range(len(toks)):
                    i = base + f * K + r
                    self.token[b, i] = toks[r]
                    self.parent[b, i] = pid
                    self.logc[b, i] = logc[r]
                    self.value[b, i] = self.value[b, pid] + logc[r]
            self.layer_sorted[b][d] = self.sorted_nodes(b, self.layer_ids(b, d))
        self.cur_depth = d
        return d

    def select_frontier(self, width, stop=None, gaps=None):
        """Frontier of the next layer: top-w nodes of the newest layer, slots in id order.

        ``width`` is an int or a per-request list; ``stop[b]`` true gives b an
        empty frontier. Returns the frontier tokens [B][W] padded with -1.
        """
        d = self.cur_depth
        out = np.full((self.B, self.W), -1, np.int64)
        for b in range(self.B):
            w = width if np.isscalar(width) else width[b]
            srt = self.layer_sorted[b].get(d, [])
            if stop is not None and stop[b]:
                w = 0
            w = max(0, min(int(w), self.W, len(srt)))
            if gaps is not None and 0 < w < len(srt):
                self._cut_gap(gaps, "frontier", b, srt[w - 1], srt[w])
            self.frontier[b] = sorted(srt[:w])
            for f, i in enumerate(self.frontier[b]):
                out[b, f] = self.token[b, i]
        return out

    def _cut_gap(self, gaps, kind, b, i_in, i_out):
        v_in, v_out = self.value[b, i_in], self.value[b, i_out]
        if v_in == v_out and self.parent[b, i_in] == self.parent[b, i_out]:
            return  # siblings with bitwise-equal logits: the id tie-break is exact
        gaps.add(kind, v_in - v_out, v_in, b)

    # -- rerank (a5) -------------------------------------------------------------
    def rerank(self, m, m_cap, gaps=None):
        """Top-m nodes of the whole tree in the total order, returned in ascending id.

        ``m`` is an int or a per-request list. Output [B][m_cap] padded with -1.
        """
        out = np.full((self.B, m_cap), -1, np.int64)
        for b in range(self.B):
            mb = m if np.isscalar(m) else m[b]
            mb = max(0, min(int(mb), m_cap))
            srt = self.sorted_nodes(b, self.nodes(b))
            take = srt[:mb]
            if gaps is not None and 0 < mb < len(srt):
                self._cut_gap(gaps, "rerank", b, srt[mb - 1], srt[mb])
            sel = sorted(take)
            out[b, :len(sel)] = sel
        return out


def build_meta(tree, selected, pos_offset, P, D_path, retrieved=None):
    """Flatten each request's verify tree and build its attention metadata (a7).

    Positions: 0 = root, then the selected draft nodes in ascending id, then the
    retrieved nodes (``retrieved[b] = (tokens, parents)`` or ``(tokens, parents,
    anchor)``: parents index the retrieved list, -1 = the template root, which
    is the root or the draft node ``anchor``) in template order. Positions past the request's
    count are unused: token, parent, depth and position id -1, empty mask row.

    mask[i][j] = 1 iff position j is an ancestor of position i or i itself.
    position_ids = pos_offset + depth. A leaf is a used position without
    children; its retrieve row lists the positions from the root to the leaf,
    padded with -1, and rows are ordered by leaf position.
    """
    B = tree.B
    tokens = np.full((B, P), -1, np.int64)
    parents = np.full((B, P), -1, np.int64)
    depth = np.full((B, P), -1, np.int64)
    node_id = np.full((B, P), -1, np.int64)
    mask = np.zeros((B, P, P), np.uint8)
    posid = np.full((B, P), -1, np.int64)
    retrieve = np.full((B, P, D_path), -1, np.int64)
    n_leaves = np.zeros(B, np.int64)
    n_pos = np.zeros(B, np.int64)
    for b in range(B):
        sel = [int(i) for i in selected[b] if i >= 0]
        pos_of = {0: 0}
        tokens[b, 0], depth[b, 0], node_id[b, 0] = tree.token[b, 0], 0, 0
        p = 1
        for i in sorted(sel):
            pid = tree.parent[b, i]
            if pid not in pos_of:
                raise AssertionError("selection is not parent-closed")
            pos_of[i] = p
            tokens[b, p] = tree.token[b, i]
            parents[b, p] = pos_of[pid]
            depth[b, p] = tree.depth[b, i]
            node_id[b, p] = i
            p += 1
        if retrieved is not None:
            rt, rp = retrieved[b][0], retrieved[b][1]
            anchor = retrieved[b][2] if len(retrieved[b]) > 2 else 0
            first = p
            for u in range(len(rt)):
                par = pos_of[anchor] if rp[u] < 0 else first + rp[u]
                tokens[b, p] = rt[u]
                parents[b, p] = par
                depth[b, p] = depth[b, par] + 1
                p += 1
        if p > P:
            raise ValueError("more positions than P")
        n_pos[b] = p
        has_child = np.zeros(P, bool)
        for i in range(1, p):
            has_child[parents[b, i]] = True
        row = 0
        for i in range(p):
            chain = [i]
            while chain[-1] != 0:
                chain.append(parents[b, chain[-1]])
            chain = chain[::-1]
            for j in chain:
                mask[b, i, j] = 1
            posid[b, i] = pos_offset[b] + depth[b, i]
            if not has_child[i]:
                if len(chain) > D_path:
                    raise ValueError("tree deeper than D_path - 1")
                retrieve[b, row, :len(chain)] = chain
                row += 1
        n_leaves[b] = row
    return dict(tokens=tokens, parents=parents, depth=depth, node_id=node_id, mask=mask,
                position_ids=posid, retrieve=retrieve, n_leaves=n_leaves, n_pos=n_pos,
                row_off=packed_row_offsets(n_pos))


def packed_row_offsets(n_pos):
    """Padding-free layout of a ragged batch's target rows.

    CAST page §局限与展望 names padded equal-length batches as a limit of the method; without padding,
    request b's n_pos[b] used positions take consecutive rows after those of requests 0..b-1, so the
    row of (b, i) is row_off[b] + i. Returns row_off[0..B], row_off[B] = the rows in all.
    """
    off = [0]
    for n in n_pos:
        off.append(off[-1] + int(n))
    return np.array(off, np.int64)
