"""The synthetic workloads (shapes, recipes and method parameters), as plain data.

Stand-ins for the pages' benchmark runs (MT-bench, HumanEval, GSM8K, Alpaca,
CNN/DM, NQ, ShareGPT warm-up, LongBench): no dataset or trained model is used;
rows come from ``synth`` with the shapes and value distributions below.

Each entry: policy, batch B, vocab V, logits dtype, per-node top-K, frontier
width k (W = the handle's maximum), draft layers D, verify budget m (or caps),
temperature T, seed, rounds, and the row recipe.
"""
import numpy as np

from . import BF16, F32, Spec


def cast_tables(B, M_rows=16, N_cols=1024, L=512.0):
    """Synthetic cost tables f(B, c, n) = a_B + b_B*n + e*c on the grid c = (row+1)*L.

    Target: one forward ~1 unit, +0.1% * B per extra input token, +2e-5 per context token.
    Draft: 0.3 units per layer, +0.1% * B per input token, +2e-6 per context token.
    (Chosen so that, with the CAST rows below, widths shrink with depth from 10 towards 1 and the
    verify count lands between ~25 and 60; steeper per-token costs prune every tree to a chain.)
    """
    c = (np.arange(M_rows, dtype=np.float64)[:, None] + 1.0) * L
    n = np.arange(1, N_cols + 1, dtype=np.float64)[None, :]
    S_T = 1.0 + 0.001 * B * n + 2e-5 * c
    S_D = 0.3 + 0.001 * B * n + 2e-6 * c
    return S_T, S_D


def chain_template(width=8, depth=8):
    """Retrieval template: level 1 = ranks 0..width-1 of the root's row, then rank 0 downwards,
    breadth-first (level, chain) order. Returns (parent, rank) lists; parent -1 = root."""
    parent, rank = [], []
    for lvl in range(1, depth + 1):
        for ch in range(width):
            parent.append(-1 if lvl == 1 else (lvl - 2) * width + ch)
            rank.append(ch if lvl == 1 else 0)
    return parent, rank


WORKLOADS = {
    # EAGLE-2 tree, PR1 reference shape
    "pr1": dict(policy="eagle", B=1, V=32000, dtype=BF16, K=4, k=4, D=6, m=16, T=0, seed=1, rounds=200,
                recipe=dict(kind=0, sigma=2 ** 0.5, peak=(2.0, 8.0), per_request_height=False, depthkey=True)),
    # EAGLE-2 Vicuna-7B shape: Zipf(1.1) over a seeded permutation + N(0, 0.5^2)
    "vicuna": dict(policy="eagle", B=1, V=32000, dtype=BF16, K=10, k=10, D=6, m=60, T=0, seed=2, rounds=1000,
                   recipe=dict(kind=1, sigma=0.5, zipf_s=1.1, depthkey=True)),
    # CAST batch shape: width/depth/verify pruning; Zipf(1.1) base + N(0, 0.5^2) + a peak of height
    # U[0, 10] per (request, round)
    "cast": dict(policy="cast", B=8, V=128256, dtype=BF16, K=10, k=10, D=8, m=60, T=0, seed=3, rounds=200,
                 recipe=dict(kind=2, sigma=0.5, zipf_s=1.1, peak=(0.0, 10.0), per_request_height=True,
                             depthkey=True),
                 cast=dict(L=512.0, M_rows=16, N_cols=1024, C1=0.3, C2=0.5, C3=0.2, R=3, width_cap=10,
                           m_cap=60)),
    # Graft hybrid: EAGLE-3-style base tree K = k = 8, D_E = 8, K_max = 60, checkpoints d0/d1/d5
    "graft": dict(policy="graft", B=16, V=151936, dtype=BF16, K=8, k=8, D=8, m=60, T=0, seed=4, rounds=200,
                  warmup_rounds=5,
                  recipe=dict(kind=0, sigma=2 ** 0.5, peak=(2.0, 8.0), per_request_height=False, depthkey=False),
                  graft=dict(ckpt_layers=[0, 1, 5], tau=[0.6, 0.4, 0.2], k_draft=[8, 24, 40], K_total=60)),
    # Graft with a block drafter (DFlash-like, 16 positions per pass): Qwen3 vocabulary, the top-4
    # alternatives at every block position, a gate at every position, K_max = 60, an 8 x 8 chain
    # template hanging from the end of the kept block; block rows: Zipf(1.1) + N(0, 0.5^2) + a peak
    # of height U[0, 10] per (request, position), so that confidence varies along the block
    "graft_block": dict(policy="graft", block=True, B=16, V=151936, dtype=BF16, K=4, k=1, D=16, m=60, T=0, seed=6,
                        rounds=200, warmup_rounds=5,
                        recipe=dict(kind=2, sigma=0.5, zipf_s=1.1, peak=(0.0, 10.0), per_request_height=False,
                                    depthkey=True),
                        graft=dict(ckpt_layers=list(range(16)), tau=[0.05] * 4 + [0.1] * 12,
                                   k_draft=[min(60, 4 * (j + 1)) for j in range(16)], K_total=60, anchor="tail",
                                   template_shape=(8, 8))),
    # sampled drafts (T = 1): EAGLE-2 tree of the PR1 shape whose children are drawn from the draft
    # rows (Gumbel-top-K); every drawn node is verified (84 nodes); Vicuna-like Zipf rows
    "sampled": dict(policy="eagle", draft_sampling=True, B=4, V=32000, dtype=BF16, K=4, k=4, D=6, m=84, T=1,
                    seed=7, rounds=200, recipe=dict(kind=1, sigma=0.5, zipf_s=1.1, depthkey=True)),
    # large-batch stress: fp32, half low-entropy (peak +U[6,12]) and half high-entropy (+U[0,2]), T = 1
    "stress": dict(policy="eagle", B=64, V=128256, dtype=F32, K=8, k=8, D=10, m=64, T=1, seed=5, rounds=500,
                   recipe=dict(kind=0, sigma=2 ** 0.5, peak=None, per_request_height=False, depthkey=True)),
}


def spec_for(w):
    """synth.Spec of a workload (per-request peak ranges for the stress mix)."""
    r = w["recipe"]
    B, V = w["B"], w["V"]
    if r["kind"] == 1:
        return Spec(V, w["dtype"], kind=1, sigma=r["sigma"], zipf_s=r["zipf_s"], B=B)
    if r["kind"] == 2:
        return Spec(V, w["dtype"], kind=2, sigma=r["sigma"], zipf_s=r["zipf_s"], peak_lo=[r["peak"][0]] * B,
                    peak_hi=[r["peak"][1]] * B, height_per_request=r["per_request_height"], B=B)
    if r["peak"] is None:  # stress: requests b < B/2 low entropy, the rest high entropy
        lo = np.array([6.0 if b < B // 2 else 0.0 for b in range(B)], np.float32)
        hi = np.array([12.0 if b < B // 2 else 2.0 for b in range(B)], np.float32)
    else:
        lo = np.full(B, r["peak"][0], np.float32)
        hi = np.full(B, r["peak"][1], np.float32)
    return Spec(V, w["dtype"], kind=0, sigma=r["sigma"], peak_lo=lo, peak_hi=hi,
                height_per_request=r["per_request_height"], B=B)


def graft_template(w):
    """(parent, rank) of a Graft workload's retrieval template: chains of template_shape = (width,
    depth), by default (k, D)."""
    width, depth = w["graft"].get("template_shape", (w["k"], w["D"]))
    return chain_template(width, depth)


def geometry(w):
    """Handle/meta sizes of a workload: W, D_max, P (positions), D_path, m_cap, R_cap."""
    pol = w["policy"]
    if pol == "graft":
        K_total = w["graft"]["K_total"]
        depth = w["graft"].get("template_shape", (w["k"], w["D"]))[1]
        if w["graft"].get("anchor", "root") == "tail":  # the template may hang from the deepest layer
            depth += w["D"]
        nodes = w["K"] + (w["D"] - 1) * w["k"] * w["K"]  # draft nodes the tree can hold
        return dict(W=w["k"], D_max=w["D"], P=K_total + 1, D_path=max(w["D"], depth) + 2, m_cap=min(K_total, nodes),
                    R_cap=K_total)
    m_cap = w["cast"]["m_cap"] if pol == "cast" else w["m"]
    if w.get("draft_sampling"):  # every drawn node is verified
        m_cap = w["K"] + (w["D"] - 1) * w["k"] * w["K"]
    return dict(W=w["k"], D_max=w["D"], P=m_cap + 1, D_path=w["D"] + 1, m_cap=m_cap, R_cap=0)


def with_sizes(name, **over):
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    w = dict(WORKLOADS[name])
    w.update(over)
    return w
