"""Graft with a block drafter, and tail-anchored templates, on the GPU vs the oracle (C ABI).

Graft page, extension direction 1 and weakness 4: dt_block_expand builds every draft layer of a
16-position block in one launch, with the checkpoint rule at every position; the retrieval template
hangs from the end of the kept block (or from the root). Every output of every round (tree, gates,
selection, retrieval, metadata, verify, M refresh) must equal the oracle's, which runs the layers one
by one.
"""
import pytest

from synth.workloads import WORKLOADS, with_sizes
from test_gpu_parity import _run_rounds, torch  # noqa: F401  (the module's CUDA fixture)

pytestmark = pytest.mark.gpu


def _graft(name, **over):
    g = dict(WORKLOADS[name]["graft"])
    g.update(over.pop("graft", {}))
    return with_sizes(name, graft=g, **over)


@pytest.mark.parametrize("over,rounds", [
    (dict(V=4099, B=4), 8),                                                    # tail anchor, M learns
    (dict(V=4099, B=4, graft=dict(anchor="root")), 6),                         # root anchor (side stream)
    (dict(V=3001, B=3, K=1, graft=dict(k_draft=[j + 1 for j in range(16)])), 6),  # the plain block chain
    (dict(V=3001, B=2, graft=dict(tau=[0.0] * 16)), 3),                        # no gate fails: all layers
    (dict(V=3001, B=5, D=6, graft=dict(ckpt_layers=[0, 2, 5], tau=[0.05, 0.1, 0.1],
                                       k_draft=[4, 12, 24])), 5),              # L = 6, three gates
    ({}, 3)])                                                                  # full size
def test_block_rounds_match_oracle(torch, over, rounds):  # noqa: F811
    w = _graft("graft_block", **over)
    _run_rounds(torch, w, rounds, label=f"graft block {over}", chain_roots=False)


@pytest.mark.parametrize("over,rounds", [(dict(V=9001, B=4, graft=dict(anchor="tail")), 6),
                                         (dict(graft=dict(anchor="tail")), 2)])
def test_tail_anchored_graft_matches_oracle(torch, over, rounds):  # noqa: F811
    """The per-layer Graft tree with its template at the deepest kept draft node."""
    w = _graft("graft", **over)
    _run_rounds(torch, w, rounds, label=f"graft tail {over}", chain_roots=False)
