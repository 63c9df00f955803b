"""Pins of the sampled-draft oracle (``oracle.sampled``), all on the CPU.

What fixes them (not the oracle itself):
* Plackett-Luce: successive draws without replacement from q give the ordered sequence
  (t_1..t_K) with probability prod_j q(t_j) / (1 - sum_{i<j} q(t_i)); these sum to 1, and the
  Gumbel-top-K order drawn with the Philox uniforms must match them in frequency (chi-square).
* Losslessness (EAGLE-2 page, §"无损性为什么没有被动态树破坏"): whatever the draft distribution and
  the number of siblings, the emitted token is distributed exactly as the target's p. Checked by
  exact enumeration of every ordered draw, and by Monte Carlo with the Philox uniforms over a
  two-level tree (first token ~ p_root; second token, after an accepted first one, ~ p(.|t1)).
* Special cases: q = p accepts the first child always; a single child (K = 1) is the page's
  one-token rule; a proposal that ignores the earlier siblings (a plausible mistake, planted here
  on the CPU) is not lossless, so the pins above would catch it.
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


def test_draw_uniforms_are_a_separate_stream():
    """The draw noise does not reuse the residual or the acceptance uniforms of any position."""
    u = sampled.draw_uniforms(5, 3, 1, 2, 64)
    g = philox.gumbel_uniforms(5, 3, 1, 2, 64)
    assert (u > 0).all() and (u < 1).all()
    assert not np.allclose(u, g)
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
