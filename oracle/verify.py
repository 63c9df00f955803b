"""Tree verification against target rows: greedy and speculative sampling (test infrastructure only).

Source: EAGLE-2 page, §"先把投机解码的账本摆清楚" (accept t with
probability a = min(1, p(t)/q(t)), on rejection resample from
norm(max(0, p - q))), §"无损性为什么没有被动态树破坏" (the rule, not the tree
shape, makes the output distribution equal the target's; greedy is
deterministic) and step 3 of §"一段更贴近实现的流程" (apply the rule along
the candidate paths, commit the accepted tokens).

Readings taken where the page is silent or garbled:

* Greedy: for every root-to-leaf retrieve row, count the leading positions
  whose token equals the argmax (ties to the lower id) of the target row of
  their parent; the longest count wins, ties to the earlier row. The bonus
  token is the argmax of the target row of the last accepted position.
* Sampling: the candidates are deterministic (top-K / top-m), so the proposal
  of each candidate is a point mass q = delta_x. Then a = P_res(x) and the
  residual norm(max(0, P_res - delta_x)) is P_res with x zeroed and
  renormalised. Children are tried in position order; an accepted child
  becomes the new node; when every child is rejected, or at a leaf, the bonus
  token is drawn from the current residual.
* The residual draw is a Gumbel-max draw: argmax, over the tokens not
  rejected at this node, of x_v + G_v with G_v = -log(-log(u_v)); this draws
  exactly from softmax(x) restricted to those tokens, i.e. from the residual. Uniforms come from Philox (see
  ``philox``).
"""

import numpy as np

from . import philox


def _row(rows, b, i):
    return np.asarray(rows(b, i) if callable(rows) else rows[b][i], dtype=np.float64)


def argmax_lowest(x):
    """Index of the largest entry, the lowest index among equal maxima."""
    x = np.asarray(x)
    return int(np.flatnonzero(x == x.max())[0])


def topk_ids(x, k):
    """Ids of the k largest entries, ordered by (value desc, id asc)."""
    x = np.asarray(x, dtype=np.float64)
    return np.lexsort((np.arange(x.size), -x))[:k].astype(np.int64)


def verify_greedy(meta, rows):
    B, P, D_path = meta["retrieve"].shape
    acc = np.zeros(B, np.int64)
    path = np.full((B, D_path), -1, np.int64)
    bonus = np.zeros(B, np.int64)
    for b in range(B):
        tok = meta["tokens"][b]
        amax = {}

        def am(i):
            if i not in amax:
                amax[i] = argmax_lowest(_row(rows, b, i))
            return amax[i]

        best, best_row = -1, 0
        for r in range(meta["n_leaves"][b]):
            chain = [int(p) for p in meta["retrieve"][b, r] if p >= 0]
            cnt = 0
            for j in range(1, len(chain)):
                if tok[chain[j]] >= 0 and tok[chain[j]] == am(chain[j - 1]):
                    cnt += 1
                else:
                    break
            if cnt > best:
                best, best_row = cnt, r
        chain = [int(p) for p in meta["retrieve"][b, best_row] if p >= 0][:best + 1]
        acc[b] = best
        path[b, :len(chain)] = chain
        bonus[b] = am(chain[-1])
    return acc, path, bonus


def _softmax(x):
    e = np.exp(x - x.max())
    return e / e.sum()


def verify_sample(meta, rows, seed, rnd, gaps=None):
    """Speculative sampling along the tree with point-mass proposals (see module docstring)."""
    B, P, D_path = meta["retrieve"].shape
    acc = np.zeros(B, np.int64)
    path = np.full((B, D_path), -1, np.int64)
    bonus = np.zeros(B, np.int64)
    for b in range(B):
        tok = meta["tokens"][b]
        par = meta["parents"][b]
        n_pos = int(meta["n_pos"][b])
        cur, chain = 0, [0]
        while True:
            x = _row(rows, b, cur)
            resid = _softmax(x)
            children = [j for j in range(1, n_pos) if par[j] == cur]
            rejected = []
            moved = False
            for j in children:
                t = int(tok[j])
                p_acc = 0.0
                if t >= 0:
                    p_acc = resid[t] / resid.sum()
                u = philox.accept_uniform(seed, rnd, b, j)
                if gaps is not None and t >= 0 and resid[t] > 0:
                    gaps.add("accept", u - p_acc, p_acc, b)
                if u < p_acc:
                    cur = j
                    chain.append(j)
                    moved = True
                    break
                if t >= 0:
                    resid[t] = 0.0
                    rejected.append(t)
            if not moved:
                uu = philox.gumbel_uniforms(seed, rnd, b, cur, x.size)
                y = x + (-np.log(-np.log(uu)))
                y[rejected] = -np.inf
                t = argmax_lowest(y)
                if gaps is not None:
                    y2 = y.copy()
                    y2[t] = -np.inf
                    gaps.add("gumbel", y[t] - y2.max(), y[t], b)
                bonus[b] = t
                break
        acc[b] = len(chain) - 1
        path[b, :len(chain)] = chain
    return acc, path, bonus


def row_top8(meta, rows, k=8):
    """Top-k ids of every used position's target row (Graft's M refresh input)."""
    B, P = meta["tokens"].shape
    out = np.full((B, P, k), -1, np.int64)
    for b in range(B):
        for i in range(int(meta["n_pos"][b])):
            if meta["tokens"][b, i] >= 0:
                out[b, i] = topk_ids(_row(rows, b, i), k)
    return out
