"""Pins of the per-request CAST rule in the oracle (``oracle.cast`` with ``reqs``, ``run_round`` with
``cast.per_request``), CPU only.

CAST page §局限与展望 names padded equal-length batches as a limit of the method; the per-request
rule applies the same width, depth and verify-count rules to each request's own utilities, context,
FIFO and stop. What fixes it: (1) on a batch of identical requests it must decide exactly what the
batch-wide rule decides (a batch average of equal values is that value), and on one request the two
rules are the same; (2) a hand-worked batch of two requests whose trees differ, where each request
must follow its own trajectory (worked out in the comments) while the batch-wide rule averages them.
"""
import math

import numpy as np

import oracle.round as oround
from test_oracle_round import CAST_DRAFT, CAST_TARGET, cast_cfg, prow


def rows_by_request(tables, default=None):
    default = default if default is not None else {0: 0.34, 1: 0.33}

    def f(b, d, ctx):
        return prow(tables[b].get((d, ctx), default))
    return f


def run(B, tables_draft, tables_target, per_request):
    cfg = cast_cfg()
    cfg["B"] = B
    cfg["cast"] = dict(cfg["cast"], per_request=per_request)
    return oround.run_round(cfg, np.array([2] * B), rows_by_request(tables_draft), rows_by_request(tables_target))


def test_identical_requests_decide_like_the_batch_rule():
    B = 3
    a = run(B, [CAST_DRAFT] * B, [CAST_TARGET] * B, per_request=True)
    c = run(B, [CAST_DRAFT] * B, [CAST_TARGET] * B, per_request=False)
    assert [w[0] for w in a["widths"]] == c["widths"] == [2, 1, 1, 2]
    assert all(len(set(w)) == 1 for w in a["widths"])
    assert a["m"] == [c["m"]] * B == [7] * B
    np.testing.assert_array_equal(a["selected"], c["selected"])
    np.testing.assert_array_equal(a["accept_len"], c["accept_len"])
    np.testing.assert_array_equal(a["tree"].token, c["tree"].token)


def test_one_request_is_the_batch_rule():
    a = run(1, [CAST_DRAFT], [CAST_TARGET], per_request=True)
    c = run(1, [CAST_DRAFT], [CAST_TARGET], per_request=False)
    assert [w[0] for w in a["widths"]] == c["widths"] and a["m"] == [c["m"]]
    np.testing.assert_array_equal(a["meta"]["tokens"], c["meta"]["tokens"])


# Request 1 drafts like request 0 at layer 1, then much less confidently:
#   layer 2, ctx 0: p = .2 (tok 0), .15 (tok 1) -> values .12, .09;  ctx 1: .2 (tok 1), .1 (tok 0) -> .06, .03
REQ1_DRAFT = {(1, 2): {0: .6, 1: .3}, (2, 0): {0: .2, 1: .15}, (2, 1): {1: .2, 0: .1}}


def test_two_requests_follow_their_own_trajectories():
    """Request 0: the single-request round of test_oracle_round (widths 2, 1, 1, 2; stops after
    layer 4; m = 7). Request 1, by its own rule: d=1 as request 0 (n = 2, key .9: grow); d=2 context
    2 -> steep row: n = 1 (.09 / 9 < .3), u_1 = .12, FIFO {1, .12/.9}, mean .56667, key .56667 * .12
    = .068 < .15: stop after layer 2, so its widths are 2, 1 and then 0. Its verify count: values
    .6 .3 .12 | .09 .06 .03 against .1 per node: m = 3."""
    a = run(2, [CAST_DRAFT, REQ1_DRAFT], [CAST_TARGET, CAST_TARGET], per_request=True)
    assert [w[0] for w in a["widths"]] == [2, 1, 1, 2]
    assert [w[1] for w in a["widths"]] == [2, 1, 0, 0]
    assert a["m"] == [7, 3]
    t = a["tree"]
    lin1 = sorted((math.exp(t.value[1, i]) for i in t.nodes(1)), reverse=True)
    want1 = [.6, .3, .12, .09, .06, .03]
    assert len(lin1) == 6 and all(math.isclose(x, y, rel_tol=1e-12) for x, y in zip(lin1, want1))
    assert int(a["meta"]["n_pos"][0]) == 8 and int(a["meta"]["n_pos"][1]) == 4
    # the batch-wide rule averages the two requests and decides otherwise
    c = run(2, [CAST_DRAFT, REQ1_DRAFT], [CAST_TARGET, CAST_TARGET], per_request=False)
    assert c["widths"] != [w[0] for w in a["widths"]] or c["m"] != 7


# ---- padding-free target rows (the verify layout of ragged batches) ----
def test_packed_row_offsets_of_the_two_request_round():
    """Request 0 uses 8 positions and request 1 uses 4: without padding their target rows are rows
    0..7 and 8..11 of one buffer."""
    a = run(2, [CAST_DRAFT, REQ1_DRAFT], [CAST_TARGET, CAST_TARGET], per_request=True)
    assert list(a["meta"]["row_off"]) == [0, 8, 12]


def test_packed_rows_cover_the_used_positions_once_and_verify_alike():
    """Every used position (b, i) gets its own row row_off[b] + i, the rows of all requests cover
    0..row_off[B]-1 exactly once, and the greedy verify reading packed rows decides exactly what it
    decides on the padded rows (same rows, other addresses)."""
    from oracle.tree import OracleTree, build_meta, packed_row_offsets
    from oracle.verify import verify_greedy

    for seed in range(5):
        rng = np.random.default_rng(100 + seed)
        B, V, K, W, D = 4, 10, 3, 2, 3
        t = OracleTree(B, K, W, D, rng.integers(0, V, B))
        for d in range(1, D + 1):
            t.expand_layer(lambda b, f: rng.normal(0, 2, V))
            if d < D:
                t.select_frontier(W)
        m = [int(x) for x in rng.integers(0, 9, B)]
        sel = t.rerank(m, 8)
        meta = build_meta(t, sel, np.zeros(B, np.int64), P=9, D_path=D + 1)
        n_pos = meta["n_pos"]
        off = packed_row_offsets(n_pos)
        assert list(n_pos) == [1 + x for x in m]
        seen = sorted(int(off[b]) + i for b in range(B) for i in range(int(n_pos[b])))
        assert seen == list(range(int(off[B])))
        padded = rng.normal(0, 2, (B, 9, V))
        packed = np.concatenate([padded[b, :int(n_pos[b])] for b in range(B)])
        g1 = verify_greedy(meta, lambda b, i: padded[b, i])
        g2 = verify_greedy(meta, lambda b, i: packed[int(off[b]) + i])
        for x, y in zip(g1, g2):
            np.testing.assert_array_equal(x, y)
