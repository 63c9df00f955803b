"""CAST cost-aware width, depth and verify-count pruning, fp64 (test infrastructure only).

Source: "Inference-Cost-Aware Dynamic Tree Construction for Efficient Inference
in Large Language Models", §关键设计:

1. cost lookup tables S_T(B), S_D(B) over context c on the grid c = kL and
   input length n = 1..N, with a quantiser select(c);
2. width pruning: u_k = (1/B) sum_j sum_{s<=k} v_i^(j)(s) over the layer's
   candidates sorted by confidence, c_k = S_D[select(ctx)][k] / S_T[select(ctx)][1],
   keep n_i nodes by the marginal-utility test against C1 ("Algorithm 1");
   Theorem 4.1: with c_j = lambda*j + delta and C1 = sum_j v^(j)(K)/(B lambda)
   the rule keeps exactly K;
3. depth pruning: FIFO buffer A of the last R gain ratios
   phi_i = u^(i+1)_{n_{i+1}} / u^(i)_{n_i}, initial content {1};
   grow layer i+1 iff Avg(A) * u^(i)_{n_i} / c^(i)_{n_i} >= C2;
4. verify count: u_k = sum_{j<=k} v_(j), c_k = S_T[select(n_0)][k] / S_T[select(n_0)][1],
   threshold C3, same selection rule.

Readings taken where the page is silent or garbled (the body of Algorithm 1 is not on the page):

* select(): the printed form max(floor(c/L), M-1) maps every c past the table;
  read as row = min(floor(c/L), M_rows - 1).
* Table column n-1 holds input length n (1-based n in the formulas).
* v = exp(value), the linear path value (product of confidences).
* ctx for layer i = n_0 + sum_{j<i} n_j (n_0 = prefix length, n_j the widths
  already chosen); the verify count uses ctx = n_0.
* Selection rule: k0 = 1; for k = 2..cap, move k0 to k when the cost does not
  grow (c_k <= c_{k0}) or (u_k - u_{k0}) / (c_k - c_{k0}) >= threshold; the
  scan continues after a failed step. ">=" (not ">") is the comparator for
  which Theorem 4.1 yields exactly K. u_k - u_{k0} is summed over the added
  items directly.
* Width cap = the per-node K (10 for the CAST workload); n_i is batch-wide.
  Verify cap m_cap = 60, minimum 1, batch-wide m.
* Per-request rule (the page's stated limitation, §局限与展望: padded equal-length batches, no
  continuous batching): every request applies the same rules to its own utilities alone (a
  "batch" of one: u_k = sum_{s<=k} v^(b)(s)), with its own context sum, its own FIFO and its own
  stop, and its own verify count m_b; the cost tables are the running batch's, as in the batch-wide
  rule.
* Depth: layer 1 always exists; after layer i (i >= 2) is pruned the ratio
  phi_{i-1} is pushed (oldest dropped beyond R), then the C2 test decides
  whether layer i+1 is built; layer D_max is the last.
"""

import math

import numpy as np


def select_row(c, L, M_rows):
    """Grid row of context length c (the page's select(), clamped to the table)."""
    return min(int(math.floor(c / L)), M_rows - 1)


def selection_rule(item_sums, cost, threshold, cap, gaps=None, kind="C", b=None):
    """Marginal-utility selection over k = 1..cap.

    ``item_sums[s]`` is the batch-averaged utility of the s-th item (0-based),
    ``cost[k]`` the normalised cost of taking k items (1-based, k = 1..cap).
    Returns k0 >= 1.
    """
    k0 = 1
    for k in range(2, cap + 1):
        if cost[k] <= cost[k0]:
            k0 = k
            continue
        du = float(np.sum(item_sums[k0:k]))
        marg = du / (cost[k] - cost[k0])
        if gaps is not None:
            gaps.add(kind, marg - threshold, marg, b)
        if marg >= threshold:
            k0 = k
    return k0


def sorted_linear_values(tree, b, ids):
    srt = tree.sorted_nodes(b, ids)
    return np.exp(np.array([tree.value[b, i] for i in srt], dtype=np.float64))


def batch_item_sums(per_req, B, cap):
    """(1/B) * sum over requests of the s-th sorted linear value, s < cap (missing = 0)."""
    acc = np.zeros(cap)
    for v in per_req:
        n = min(cap, v.size)
        acc[:n] += v[:n]
    return acc / B


class CastState:
    """Per-round CAST state: FIFO ratio buffer, context sum and last utility."""

    def __init__(self):
        self.fifo = [1.0]
        self.ctx_sum = 0
        self.u_prev = None


def width_depth(tree, d, state, p, gaps=None, reqs=None):
    """Width n_d and the grow decision after layer d (CAST key designs 2 and 3).

    ``p`` holds S_T, S_D (arrays [M_rows][N_cols]), L, n0, C1, C2, R,
    width_cap, D_max. ``reqs``: the requests whose utilities are averaged (all of the batch by
    default; one request for the per-request rule, with that request's own state). Returns
    (n_d, grow).
    """
    reqs = list(range(tree.B)) if reqs is None else list(reqs)
    B = len(reqs)
    per_req = [sorted_linear_values(tree, b, tree.layer_ids(b, d)) for b in reqs]
    maxcand = max(v.size for v in per_req)
    if maxcand == 0:
        return 0, False
    cap = min(p["width_cap"], maxcand)
    items = batch_item_sums(per_req, B, cap)
    gb = reqs[0] if len(reqs) == 1 and reqs != list(range(tree.B)) else None
    u = np.concatenate([[0.0], np.cumsum(items)])          # u[k], k = 0..cap
    row = select_row(p["n0"] + state.ctx_sum, p["L"], p["S_T"].shape[0])
    cost = np.zeros(cap + 1)
    for k in range(1, cap + 1):
        cost[k] = p["S_D"][row][k - 1] / p["S_T"][row][0]
    n = selection_rule(items, cost, p["C1"], cap, gaps, "C1", gb)
    if state.u_prev is not None:
        state.fifo.append(u[n] / state.u_prev)
        while len(state.fifo) > p["R"]:
            state.fifo.pop(0)
    alpha = float(np.mean(state.fifo))
    key = alpha * u[n] / cost[n]
    grow = False
    if d < p["D_max"]:
        if gaps is not None:
            gaps.add("C2", key - p["C2"], key, gb)
        grow = key >= p["C2"]
    state.u_prev = u[n]
    state.ctx_sum += n
    return n, grow


def verify_count(tree, p, gaps=None, reqs=None):
    """Verify budget m (CAST key design 4): batch-wide, or for the requests ``reqs`` alone (the
    per-request rule passes one request)."""
    reqs = list(range(tree.B)) if reqs is None else list(reqs)
    B = len(reqs)
    per_req = [sorted_linear_values(tree, b, tree.nodes(b)) for b in reqs]
    gb = reqs[0] if len(reqs) == 1 and reqs != list(range(tree.B)) else None
    maxn = max(v.size for v in per_req)
    if maxn == 0:
        return 0
    cap = min(p["m_cap"], maxn)
    items = batch_item_sums(per_req, B, cap)
    row = select_row(p["n0"], p["L"], p["S_T"].shape[0])
    cost = np.zeros(cap + 1)
    for k in range(1, cap + 1):
        cost[k] = p["S_T"][row][k - 1] / p["S_T"][row][0]
    return selection_rule(items, cost, p["C3"], cap, gaps, "C3", gb)


def linear_table(M_rows, N_cols, L, a, b_coef, e):
    """Synthetic cost table f(c, n) = a + b*n + e*c on the grid c = (row+1)*L."""
    c = (np.arange(M_rows, dtype=np.float64)[:, None] + 1.0) * L
    n = np.arange(1, N_cols + 1, dtype=np.float64)[None, :]
    return a + b_coef * n + e * c
