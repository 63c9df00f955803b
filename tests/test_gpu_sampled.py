"""Sampled drafts on the GPU vs the oracle (C ABI): children drawn from the draft rows by Philox
Gumbel-top-K (dt_expand_layer_sampled), every drawn node verified by the recursive-residual walk
(dt_verify_sampled). EAGLE-2 page, §先把投机解码的账本摆清楚 and §无损性为什么没有被动态树破坏.

Every output of every round (drawn tree, values, metadata, accepted paths, bonus tokens) must equal
the oracle's; rounds whose oracle decisions (draw order, acceptance tests, bonus draw) fall within
1e-5 relative of a boundary are redrawn and counted.
"""
import pytest

from synth.workloads import with_sizes
from test_gpu_parity import _run_rounds, torch  # noqa: F401  (the module's CUDA fixture)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("over,rounds", [
    (dict(V=4099, B=3), 12),                         # bf16 Zipf rows
    (dict(V=3001, B=2, K=3, k=2, D=4, m=21), 12),    # a narrower tree, more rejections per node
    (dict(V=2053, B=2, dtype=1), 8),                 # fp32 rows
    ({}, 3)])                                        # full size (B = 4, V = 32000, 84 drawn nodes)
def test_sampled_draft_rounds_match_oracle(torch, over, rounds):  # noqa: F811
    w = with_sizes("sampled", **over)
    _run_rounds(torch, w, rounds, label=f"sampled drafts {over}")


def test_sampled_draft_packed_rows(torch):  # noqa: F811
    w = with_sizes("sampled", V=4099, B=3)
    _run_rounds(torch, w, 6, label="sampled drafts, packed target rows", packed=True)
