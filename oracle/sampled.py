"""Sampled-draft speculative sampling on a tree (test infrastructure only: see the package docstring).

Source: EAGLE-2 page, §"先把投机解码的账本摆清楚": a drafted token t, drawn from the draft
distribution q, is accepted with probability min(1, p(t) / q(t)); on rejection the next token is
drawn from the residual norm(max(0, p - q)); and §"无损性为什么没有被动态树破坏": this rule, not the
shape of the tree, keeps the output distribution equal to the target's.

Readings (the page states the rule for one drafted token; the several children of a node are
repeated applications of it, each against the distribution the child was actually drawn from):

* The K children of a node are the first K tokens of an order drawn without replacement from the
  node's draft distribution q = softmax(x): the tokens by decreasing x_v + G_v (ties to the lower
  id), with G_v = -log(-log u_v) standard Gumbel noise. The first j tokens of this order are
  distributed as j successive draws without replacement (Plackett-Luce probabilities).
* Child j (in draw order) was drawn from q_j = q with the earlier children removed and
  renormalised. It is tested against the current residual r_j (r_1 = p, the target distribution
  at the node): accept with probability min(1, r_j(t_j) / q_j(t_j)); on rejection
  r_{j+1} = norm(max(0, r_j - q_j)).
* An accepted child becomes the current node (its own target and draft distributions and
  children next). When every child of the current node is rejected, or it has none, the bonus
  token is drawn from the last residual and the round ends.
* The verified tree is every drawn node: the frontier still chooses by value which nodes get
  children (a node's children are drawn after that choice, so it cannot bias them), but no node
  is dropped after its draw. Dropping drawn nodes by their own values (a rerank) makes whether a
  child is tested depend on the child itself, and the first emitted token is then no longer
  distributed as the target's (exact enumeration on a three-token vocabulary shows errors up to
  0.09). The size of the verified tree is set by the frontier widths and the depth.

Uniforms (Philox4x32-10, key = seed, round r; see ``philox``):

* draw noise of token v at node n of request b: counter (r_lo, r_hi, 0x40000000 + 4096 b + n,
  v >> 2), word v & 3, top 23 bits, u = (k + 0.5) 2^-23 in (0, 1);
* test of the child at tree position j: the acceptance uniform of position j;
* bonus at position i: Gumbel-max over log r with the residual uniforms of position i (the
  largest log r_v + G_v over the tokens with r_v > 0, ties to the lower id).
"""

import itertools

import numpy as np

from . import philox

DRAW_STREAM = 0x40000000


def softmax(x):
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def draw_uniforms(seed, rnd, b, node, V):
    """23-bit uniforms in (0, 1) for every token 0..V-1: the draw noise of node ``node``."""
    if not (0 <= node < 4096):
        raise ValueError("node id must be in [0, 4096)")
    v = np.arange(V, dtype=np.uint64)
    n = v.size
    ctr = (np.full(n, rnd & 0xFFFFFFFF, np.uint64), np.full(n, (rnd >> 32) & 0xFFFFFFFF, np.uint64),
           np.full(n, DRAW_STREAM + 4096 * b + node, np.uint64), v >> np.uint64(2))
    w = philox.philox4x32_10(ctr, philox._key(seed))
    words = np.stack(w, axis=0)
    sel = words[(v & np.uint64(3)).astype(np.int64), np.arange(n)]
    k = (sel >> np.uint32(9)).astype(np.float64)
    return (k + 0.5) * 2.0 ** -23


def draw_order(x, K, u, gaps=None, b=None):
    """The first K tokens by decreasing x_v - log(-log u_v), ties to the lower id (-inf never drawn).
    With ``gaps``, the distance between consecutive keys of the first K + 1 is recorded (the draw
    order and the set of K drawn tokens depend on those comparisons)."""
    x = np.asarray(x, dtype=np.float64)
    key = x + (-np.log(-np.log(np.asarray(u, dtype=np.float64))))
    key[~np.isfinite(x)] = -np.inf
    order = np.lexsort((np.arange(x.size), -key))
    order = [int(t) for t in order if np.isfinite(key[t])]
    if gaps is not None:
        for a, c in zip(order[:K], order[1:K + 1]):
            gaps.add("draw", key[a] - key[c], key[a], b)
    return order[:K]


def sample_children(x, K, seed, rnd, b, node, gaps=None):
    """The K children of node ``node`` (draw order), drawn from softmax(x) without replacement."""
    return draw_order(x, K, draw_uniforms(seed, rnd, b, node, np.asarray(x).size), gaps, b)


def plackett_luce(q, seq):
    """Probability that successive draws without replacement from q give the sequence seq."""
    prob, rest = 1.0, 1.0
    for t in seq:
        if rest <= 0.0:
            return 0.0
        prob *= q[t] / rest
        rest -= q[t]
    return prob


def without(q, t):
    """q with token t removed, renormalised (the distribution of the next draw)."""
    q = np.array(q, dtype=np.float64)
    q[t] = 0.0
    s = q.sum()
    return q / s if s > 0.0 else q


def residual(r, q):
    """norm(max(0, r - q)): the distribution to continue from after a rejection."""
    d = np.maximum(0.0, np.asarray(r, dtype=np.float64) - np.asarray(q, dtype=np.float64))
    s = d.sum()
    return d / s if s > 0.0 else d


def accept_probability(r, q, t):
    """min(1, r(t) / q(t)) for a token drawn from q (q(t) > 0)."""
    return min(1.0, r[t] / q[t])


def try_children(p, q, children, uniforms, gaps=None):
    """Tests the children (draw order) of a node against target p and draft q with the given
    uniforms. Returns (index of the accepted child or None, residual after the last rejection)."""
    r = np.array(p, dtype=np.float64)
    qj = np.array(q, dtype=np.float64)
    for j, t in enumerate(children):
        a = accept_probability(r, qj, t)
        if gaps is not None:
            gaps.add("accept", uniforms[j] - a, a)
        if uniforms[j] < a:
            return j, r
        r = residual(r, qj)
        qj = without(qj, t)
    return None, r


def bonus_from_residual(r, u, gaps=None):
    """Gumbel-max draw from r: the largest log r_v - log(-log u_v) over r_v > 0, lowest id on ties."""
    r = np.asarray(r, dtype=np.float64)
    y = np.full(r.size, -np.inf)
    pos = r > 0.0
    y[pos] = np.log(r[pos]) + (-np.log(-np.log(np.asarray(u, dtype=np.float64)[pos])))
    t = int(np.flatnonzero(y == y.max())[0])
    if gaps is not None:
        y2 = y.copy()
        y2[t] = -np.inf
        gaps.add("gumbel", y[t] - y2.max(), y[t])
    return t


def emit_distribution(p, q, K):
    """Exact distribution of the token a node emits (its accepted child, else the bonus) when its
    K children are drawn from q without replacement: a sum over every ordered draw of its
    Plackett-Luce probability times the acceptance walk's outcome probabilities."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    support = [t for t in range(q.size) if q[t] > 0.0]
    K = min(K, len(support))
    out = np.zeros(q.size)
    for seq in itertools.permutations(support, K):
        w = plackett_luce(q, seq)
        if w == 0.0:
            continue
        r, qj, stay = p.copy(), q.copy(), 1.0
        for t in seq:
            a = accept_probability(r, qj, t)
            out[t] += w * stay * a
            stay *= 1.0 - a
            r = residual(r, qj)
            qj = without(qj, t)
        out += w * stay * r
    return out


def walk(children, target, draft, seed, rnd, b, V, gaps=None):
    """The acceptance walk over one request's tree.

    ``children[i]``: list of (position, token) of the children of tree position i, in draw order
    (the root is position 0); ``target(i)`` / ``draft(i)``: the target distribution and the draft
    distribution the children of position i were drawn from. Returns the accepted positions (root
    first) and the bonus token.
    """
    cur, chain = 0, [0]
    while True:
        kids = children.get(cur, [])
        u = [philox.accept_uniform(seed, rnd, b, j) for j, _ in kids]
        j, r = try_children(target(cur), draft(cur), [t for _, t in kids], u, gaps)
        if j is None:
            return chain, bonus_from_residual(r, philox.gumbel_uniforms(seed, rnd, b, cur, V), gaps)
        cur = kids[j][0]
        chain.append(cur)


def verify_tree(tree, meta, target_row, seed, rnd, gaps=None):
    """Sampled-draft verify of every request of a flattened tree (``tree.build_meta`` layout).

    ``tree`` is the ``OracleTree`` whose expansion drew the children (it keeps, for every expanded
    node, the draft row its children were drawn from) and ``meta`` its flattening with every drawn
    node selected; ``target_row(b, i)`` is the target row at position i. A position's children are tested in position order, which is their draw order
    (ids grow with the draw rank and positions with the id). Returns accepted lengths, accepted
    positions (root first, -1 padded) and bonus tokens.
    """
    B, P, D_path = meta["retrieve"].shape
    acc = np.zeros(B, np.int64)
    path = np.full((B, D_path), -1, np.int64)
    bonus = np.zeros(B, np.int64)
    for b in range(B):
        n_pos = int(meta["n_pos"][b])
        tok, par, node = meta["tokens"][b], meta["parents"][b], meta["node_id"][b]
        children = {}
        for j in range(1, n_pos):
            children.setdefault(int(par[j]), []).append((j, int(tok[j])))
        V = np.asarray(target_row(b, 0)).size

        def target(i):
            return softmax(target_row(b, i))

        def draft(i):
            row = tree.draft_row[b].get(int(node[i]))
            return softmax(row) if row is not None else np.full(V, 1.0 / V)  # unused: no children

        chain, bt = walk(children, target, draft, seed, rnd, b, V, gaps)
        acc[b] = len(chain) - 1
        path[b, :len(chain)] = chain
        bonus[b] = bt
    return acc, path, bonus
