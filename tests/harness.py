"""Test harness: the same seeded rows fed to the oracle (host generator) and the GPU path
(device generator), round drivers for both, and the comparison rules.

Comparison rules:
  * index outputs (tokens, parents, frontier sets, selections, masks, position ids, retrieve rows,
    accepted lengths and paths, bonus tokens, M rows) must be equal;
  * log confidences and log values: |gpu - oracle| <= 2e-6 * max(1, |oracle|);
  * a request whose oracle decision gaps fall below 1e-5 relative is redrawn (its attempt + 1, a new
    generator salt) and counted; batch-coupled CAST decisions redraw the whole batch.
"""
import numpy as np

import synth
from synth.workloads import spec_for, geometry, cast_tables, graft_template
from oracle.round import run_round
from oracle.tree import Gaps

TOL = 2e-6
GAP = 1e-5


def salts_of(w, rnd, attempts):
    """Per-request generator salts. Graft rows are stationary across rounds (the salt is the
    attempt only) so that M can learn successors; other workloads key rows by round."""
    a = np.asarray(attempts, np.uint64)
    if w["policy"] == "graft":
        return a.copy()
    return (np.uint64(rnd) << np.uint64(8)) | a


def round_id(rnd):
    """Philox round of a round (the same for every redraw of its requests)."""
    return rnd << 8


_ROWS = {"owner": None, "rows": {}}

# Seed redraws of the parity runs of this process: (label, rounds compared, requests redrawn, rounds
# with at least one redraw). Printed at the end of the test session.
REDRAW_LOG = []


def log_redraws(label, rounds, redrawn, rounds_hit):
    REDRAW_LOG.append((label, int(rounds), int(redrawn), int(rounds_hit)))


class HostRows:
    """Row providers for the oracle, keyed like the device generator.

    Generated rows are cached (raw dtype) per (stream, request, depth key, context, salt), so a
    redraw of some requests regenerates only theirs.
    """

    def __init__(self, w, spec, salts):
        self.w, self.spec = w, spec
        self.salts = np.ascontiguousarray(salts, np.uint64)
        self.depthkey = w["recipe"]["depthkey"]
        owner = (w["seed"], w["V"], w["B"], w["dtype"], repr(w["recipe"]))
        if _ROWS["owner"] != owner:
            _ROWS["owner"] = owner
            _ROWS["rows"] = {}
        self._cache = _ROWS["rows"]

    def _row(self, stream, b, dk, ctx):
        key = (stream, b, dk, ctx, int(self.salts[b]))
        raw = self._cache.get(key)
        if raw is None:
            raw = synth.gen_rows_cpu(self.spec, self.w["seed"], 0, stream, [ctx], depth_add=dk, b0=b,
                                     salts=self.salts)[0]
            self._cache[key] = raw
        return synth.to_f64(raw, self.spec.dtype)

    def draft_row(self, b, d, ctx):
        return self._row(synth.DRAFT, b, d if self.depthkey else 0, ctx)

    def target_row(self, b, d, ctx):
        return self._row(synth.TARGET, b, d if self.depthkey else 0, ctx)


def oracle_cfg(w):
    g = geometry(w)
    c = dict(policy=w["policy"], B=w["B"], K=w["K"], W=g["W"], D=g["D_max"], k=w["k"], m=w["m"],
             m_cap=g["m_cap"], P=g["P"], D_path=g["D_path"], T=w["T"], seed=w["seed"])
    if w["policy"] == "cast":
        cc = w["cast"]
        S_T, S_D = cast_tables(w["B"], cc["M_rows"], cc["N_cols"], cc["L"])
        c["cast"] = dict(S_T=S_T, S_D=S_D, L=cc["L"], n0=0, C1=cc["C1"], C2=cc["C2"], C3=cc["C3"], R=cc["R"],
                         width_cap=cc["width_cap"], m_cap=cc["m_cap"], D_max=g["D_max"],
                         per_request=bool(cc.get("per_request", False)))
    if w["policy"] == "graft":
        c["graft"] = dict(w["graft"], template=graft_template(w))
        c["block"] = bool(w.get("block", False))
    c["draft_sampling"] = bool(w.get("draft_sampling", False))
    return c


def cast_n0(rnd):
    return 512 * (1 + rnd % 16)


def root_tokens(w, salts):
    lib = synth._cpu_lib()
    return np.array([lib.synth_root_token(w["seed"], int(salts[b]), b, w["V"]) for b in range(w["B"])], np.int32)


def oracle_round(w, rnd, roots=None, M=None, max_attempts=16):
    """Oracle round with seed rejection; returns (ref, attempts, redraws).

    A request whose decision gaps fall below GAP relative is redrawn with its next attempt salt;
    batch-coupled decisions (CAST) redraw the whole batch. ``redraws`` counts requests redrawn.
    """
    spec = spec_for(w)
    cfg = oracle_cfg(w)
    B = w["B"]
    attempts = np.zeros(B, np.int64)
    redraws = 0
    for _ in range(max_attempts):
        salts = salts_of(w, rnd, attempts)
        rows = HostRows(w, spec, salts)
        r = roots if roots is not None else root_tokens(w, salts)
        if cfg["policy"] == "cast":
            cfg["cast"]["n0"] = cast_n0(rnd)
        gaps = Gaps()
        M_try = None if M is None else M.copy()
        ref = run_round(cfg, np.asarray(r), rows.draft_row, rows.target_row, rnd=round_id(rnd), M=M_try, gaps=gaps)
        near = gaps.near_tie(GAP)
        if not near:
            ref["M"] = M_try
            ref["roots"] = np.asarray(r)
            ref["salts"] = salts
            return ref, attempts, redraws
        bs = {it[3] for it in near}
        batch_coupled = w["policy"] == "cast" and not w["cast"].get("per_request", False)
        if None in bs or batch_coupled:
            attempts += 1
            redraws += B
        else:
            for b in bs:
                attempts[b] += 1
            redraws += len(bs)
    raise AssertionError("no tie-free draw in %d attempts" % max_attempts)


class GpuRound:
    """GPU side of a workload: a RoundRunner plus device row generators."""

    def __init__(self, w, flags=0, fused=True, packed=False):
        import torch
        from dynamic_draft_tree_gb300.rounds import RoundRunner

        self.torch = torch
        self.w = w
        self.g = g = geometry(w)
        self.spec = spec_for(w)
        B, V, k = w["B"], w["V"], w["k"]
        kw = {}
        if w["policy"] == "cast":
            cc = w["cast"]
            kw = dict(cast=dict(cc), cast_tables=cast_tables(B, cc["M_rows"], cc["N_cols"], cc["L"]))
        if w["policy"] == "graft":
            kw = dict(graft=w["graft"], template=graft_template(w), block=bool(w.get("block", False)))
        self.packed = packed
        self.draw = bool(w.get("draft_sampling", False))
        self.run = RoundRunner(w["policy"], B, V, w["K"], k, g["D_max"], g["P"], g["D_path"], g["m_cap"],
                               self.spec.dtype, T=w["T"], flags=flags, fused=fused, packed=packed, draw=self.draw, **kw)
        dt = torch.int16 if self.spec.dtype == synth.BF16 else torch.float32
        self.block = bool(w.get("block", False))
        self.dbuf = torch.zeros((B, w["D"] if self.block else k, V), dtype=dt, device="cuda")
        if self.draw:  # every layer's rows kept for the sampled verify: [D][B][k][V]
            self.dbuf = torch.zeros((w["D"], B, k, V), dtype=dt, device="cuda")
            self.run.draft_rows = self.dbuf
        self.tbuf = torch.zeros((B, g["P"], V), dtype=dt, device="cuda")
        self.M = None
        if w["policy"] == "graft":
            self.M = torch.full((B, V, 8), -1, dtype=torch.int32, device="cuda")

    def round(self, rnd, attempts, roots):
        torch, w, g = self.torch, self.w, self.g
        salts_dev = torch.as_tensor(salts_of(w, rnd, attempts).astype(np.int64)).cuda()
        salt = 0
        dk = w["recipe"]["depthkey"]
        V, k = w["V"], w["k"]

        def draft_rows(d, ftok):
            if d == 0:  # a block drafter's rows: position j + 1 of request b, keyed on the root token
                L = w["D"]
                ctx = roots_dev.repeat_interleave(L)
                pos = torch.arange(1, L + 1, dtype=torch.int32, device="cuda").repeat(w["B"])
                synth.gen_rows_gpu(torch, self.spec, w["seed"], salt, synth.DRAFT, ctx, self.dbuf, V,
                                   depth_dev=pos if dk else None, rows_per_b=L, salts_dev=salts_dev)
                return self.dbuf
            F = 1 if d == 1 else k
            if self.draw:  # layer d's rows at [d - 1], row (b, f) at b * k + f (only the frontier's read)
                ctx = ftok.contiguous().view(-1)
                synth.gen_rows_gpu(torch, self.spec, w["seed"], salt, synth.DRAFT, ctx, self.dbuf[d - 1], V,
                                   depth_add=d if dk else 0, rows_per_b=k, salts_dev=salts_dev)
                return self.dbuf[d - 1]
            ctx = ftok[:, :F].contiguous().view(-1)
            synth.gen_rows_gpu(torch, self.spec, w["seed"], salt, synth.DRAFT, ctx, self.dbuf, V,
                               depth_add=d if dk else 0, rows_per_b=F, salts_dev=salts_dev)
            return self.dbuf

        def target_rows(meta):
            if self.packed:  # padding-free: row j of the buffer belongs to the request whose rows hold it
                # rows past the used ones hold NaN: a read of one would set DT_DEV_BAD_LOGITS
                self.tbuf.fill_(-1 if self.tbuf.dtype == torch.int16 else float("nan"))  # int16 -1 = bf16 NaN
                req, ctx, dep = synth.packed_row_map(torch, meta.row_off, meta.tokens, meta.depth)
                synth.gen_rows_gpu(torch, self.spec, w["seed"], salt, synth.TARGET, ctx, self.tbuf, V,
                                   depth_dev=dep if dk else None, depth_add=1 if dk else 0, salts_dev=salts_dev,
                                   row_req_dev=req)
                return self.tbuf
            synth.gen_rows_gpu(torch, self.spec, w["seed"], salt, synth.TARGET, meta.tokens.view(-1), self.tbuf,
                               V, depth_dev=meta.depth.view(-1) if dk else None, depth_add=1 if dk else 0,
                               rows_per_b=g["P"], salts_dev=salts_dev)
            return self.tbuf

        roots_dev = torch.as_tensor(np.asarray(roots, np.int32)).cuda()
        self.run.run(roots_dev, draft_rows, target_rows, seed=w["seed"], rnd=round_id(rnd), M=self.M,
                     n0=cast_n0(rnd))


def tree_numpy(h):
    from dynamic_draft_tree_gb300 import dt_get_tree

    t = dt_get_tree(h)
    B = t["B"]
    return {k: (v[:B].cpu().numpy() if hasattr(v, "cpu") else v) for k, v in t.items()}


def assert_close(gpu, ref, what):
    ref = np.asarray(ref, np.float64)
    gpu = np.asarray(gpu, np.float64)
    both_inf = np.isinf(ref) & (gpu == ref)
    err = np.abs(gpu - ref)
    bound = TOL * np.maximum(1.0, np.abs(ref))
    bad = ~both_inf & ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} values off; first at {tuple(i)}: gpu {gpu[tuple(i)]!r} "
                             f"oracle {ref[tuple(i)]!r}")


def compare_round(gr, ref, check_tree=True):
    """Element-wise comparison of a GPU round against the oracle's."""
    run = gr.run
    w = gr.w
    B = w["B"]
    ot = ref["tree"]
    if check_tree:
        t = tree_numpy(run.h)
        valid = ot.token >= 0
        np.testing.assert_array_equal(t["token"], ot.token, err_msg="tree tokens")
        np.testing.assert_array_equal(t["parent"][valid], ot.parent[valid], err_msg="tree parents")
        assert_close(t["logc"][valid], ot.logc[valid], "log confidences")
        assert_close(t["value"][valid], ot.value[valid], "log values")
        assert t["depth"] == ot.cur_depth or w["policy"] != "eagle", "depth"
    meta = run.meta.numpy()
    om = ref["meta"]
    for key in ("n_pos", "row_off", "tokens", "parents", "depth", "node_id", "position_ids", "n_leaves", "mask",
                "retrieve"):
        np.testing.assert_array_equal(meta[key], om[key], err_msg=f"meta {key}")
    np.testing.assert_array_equal(run.accept_len.cpu().numpy(), ref["accept_len"], err_msg="accept_len")
    np.testing.assert_array_equal(run.accept_path.cpu().numpy(), ref["accept_path"], err_msg="accept_path")
    np.testing.assert_array_equal(run.bonus.cpu().numpy(), ref["bonus"], err_msg="bonus")
    if w["policy"] == "cast":
        if w["cast"].get("per_request", False):
            np.testing.assert_array_equal(run.m_dev.cpu().numpy(), np.asarray(ref["m"]), err_msg="verify counts")
        else:
            assert int(run.m_dev.cpu()[0]) == ref["m"], "CAST verify count"
    if w["policy"] == "graft":
        np.testing.assert_array_equal(run.stage.cpu().numpy(), np.asarray(ref["stage"]), err_msg="graft stage")
        np.testing.assert_array_equal(gr.M.cpu().numpy(), ref["M"], err_msg="M after refresh")
    del B


def exact_residual_events(w, ref):
    """Children of a T = 1 round's acceptance walk tested after the children rejected before them at
    the same node held more than 7/8 of the row's softmax mass: there the device walk replaces its
    running residual by an exact recomputation over the row. Counted from the oracle round ``ref``."""
    rows = HostRows(w, spec_for(w), ref["salts"])
    meta = ref["meta"]
    V = w["V"]
    n = 0
    for b in range(w["B"]):
        path = [int(p) for p in ref["accept_path"][b] if p >= 0]
        tok, par, dep = meta["tokens"][b], meta["parents"][b], meta["depth"][b]
        npos = int(meta["n_pos"][b])
        for k, cur in enumerate(path):
            nxt = path[k + 1] if k + 1 < len(path) else None
            x = rows.target_row(b, int(dep[cur]) + 1, int(tok[cur]))
            p = np.exp(x - x.max())
            p /= p.sum()
            rejected, share = set(), 0.0
            for j in range(1, npos):
                if int(par[j]) != cur:
                    continue
                t = int(tok[j])
                if t < 0 or t >= V or t in rejected:
                    continue  # not tested (the walk skips it)
                if share > 7.0 / 8.0:
                    n += 1
                if j == nxt:
                    break
                rejected.add(t)
                share += float(p[t])
    return n
