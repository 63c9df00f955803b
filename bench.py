"""Benchmark of the draft-tree hot path; headline on the CAST batch workload (B=8, V=128256, bf16).

One step = one complete round of the path (EAGLE-2 expansion with CAST width/depth pruning for up
to 8 layers, CAST verify count, rerank, flatten + metadata, greedy verify) over one batch of B=8
requests, with its inputs already in HBM. The draft and target model forwards are not part of the
path: their logits are produced by the seeded generator in an untimed recording pass (R rounds, so
that the recorded inputs exceed L2 and every timed step reads a different round), and the timed
steps replay the path on them. A replayed round must reproduce its recording bit for bit.

The same measurement runs for the four other workloads (PR1, Vicuna greedy and sampling, Graft
after its warm-up rounds, the fp32 B=64 stress batch with sampling); they are reported in the
line's "per_config" block.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workloads a,b,...]

Under torchrun each rank runs its own independent batch (requests shard across GPUs with no
exchange: weak scaling). The reference arm times the fp64 CPU oracle on a bounded sample.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft-tree rounds/s (expand+rerank+verify) at B=8,V=128256; logits HBM GB/s"
UNIT = "rounds/s"
HEADLINE = "cast"
OTHERS = ["pr1", "vicuna", "vicuna_t1", "graft", "stress", "cast_req", "graft_block", "sampled"]
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, help="workload of the headline line")
    ap.add_argument("--sizes", default="", help="sizes replaced in the headline workload, e.g. B=8 (profiling a "
                    "smaller case; the line then names the case)")
    ap.add_argument("--workloads", default=",".join(OTHERS),
                    help="comma-separated workloads measured for the per_config block ('' for none)")
    ap.add_argument("--per-config-steps", type=int, default=100)
    ap.add_argument("--min-replay-s", type=float, default=1.0, help="time the K-step graph for at least this long")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--e2e-gather-blocks", type=int, default=32,
                    help="CTAs of the kernel that reads the host rows for e2e (0: one DMA copy per row block)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--record-rounds", type=int, default=0,
                    help="recorded rounds replayed (0: enough for 3x L2 of inputs); small values for profiling runs")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, world):
    """The largest x over all ranks (the slowest rank's time); x itself on one rank. Works on the
    NCCL (device tensor) and gloo (host tensor) process groups."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as tdist

    dev = "cuda" if tdist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_max):
    """Whole-job rate: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


def workload_of(name, sizes=None):
    """(workload dict, label) of a bench workload name; vicuna_t1 is Vicuna with sampling (T = 1);
    cast_req is the CAST batch with the per-request rule and padding-free target rows. `sizes`
    ({field: int}) replaces sizes of the workload (a smaller case of it, for profiling)."""
    from synth.workloads import WORKLOADS

    if name == "vicuna_t1":
        w = dict(WORKLOADS["vicuna"])
        w["T"] = 1
        label = "vicuna_t1"
    elif name == "cast_req":
        w = dict(WORKLOADS["cast"])
        w["cast"] = dict(w["cast"], per_request=True)
        w["packed"] = True
        label = "cast_req"
    else:
        w, label = dict(WORKLOADS[name]), name
    if sizes:
        w.update(sizes)
        label = f"{label} ({', '.join(f'{k_}={v_}' for k_, v_ in sizes.items())})"
    return w, label


def parse_sizes(text):
    """'B=8,V=4099' -> {'B': 8, 'V': 4099}."""
    out = {}
    for part in filter(None, (text or "").split(",")):
        k_, v_ = part.split("=")
        out[k_.strip()] = int(v_)
    return out


def workload_config(w, g, label):
    dt = "bf16" if w["dtype"] == 0 else "fp32"
    verify = "greedy verify" if w["T"] == 0 else "speculative-sampling verify (T=1)"
    if w.get("packed"):
        verify += " of padding-free target rows"
    rule = ", per-request CAST rule" if w.get("cast", {}).get("per_request") else ""
    return {"workload": f"{label}: {w['policy']} tree round{rule}, B={w['B']}, V={w['V']}, {dt} logits, K={w['K']}, "
                        f"k<={w['k']}, depth<={w['D']}, m<={g['m_cap']}, {verify}",
            "B": w["B"], "V": w["V"], "K": w["K"], "k_max": w["k"], "D_max": w["D"], "m_cap": g["m_cap"],
            "global_batch": w["B"]}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) per algorithmic byte of the streaming
# kernels, per workload, from the ncu captures of the current kernels summarised under profiles/ (CAST:
# expand layers 1-2 and the verify passes of two rounds; stress: its shape at B=32, expand layer 2 and
# one verify pass, scaled by the rows a launch reads); a workload or kernel without a capture of its
# current code has no entry (traffic null).
TRAFFIC_PER_ALGO_BYTE = {("cast", "expand"): 1.0117, ("cast", "verify_rows"): 1.0254,
                         ("stress", "expand"): 1.0245, ("stress", "verify_rows"): 1.0032}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


class EventTiming:
    """Events around the halves of the split expansion / verify calls (see RoundRunner.run)."""

    def __init__(self, torch):
        self.torch = torch
        self.ev = {}

    def _new(self):
        try:
            return self.torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return self.torch.cuda.Event(enable_timing=True)

    def start(self, kind):
        e = self._new()
        e.record()
        self.ev.setdefault(kind, []).append([e, None])

    def stop(self, kind):
        e = self._new()
        e.record()
        self.ev[kind][-1][1] = e

    def ms(self, kind):
        return [a.elapsed_time(b) for a, b in self.ev.get(kind, [])]


def measure_workload(name, steps, warmup, args, rank, world, local, with_e2e):
    """Record rounds of workload `name`, replay them as a CUDA graph of `steps` rounds, time it."""
    import torch
    import torch.distributed as tdist

    import synth
    from synth.workloads import spec_for, geometry, cast_tables, graft_template
    from dynamic_draft_tree_gb300 import dt_get_status
    from dynamic_draft_tree_gb300.rounds import RoundRunner

    w, label = workload_of(name, parse_sizes(args.sizes) if name == args.workload else None)
    w["seed"] = w["seed"] + 1000 * rank  # independent batch per rank
    g = geometry(w)
    spec = spec_for(w)
    B, V, k, D, P = w["B"], w["V"], w["k"], g["D_max"], g["P"]
    kw = {}
    if w["policy"] == "cast":
        cc = w["cast"]
        kw = dict(cast=dict(cc), cast_tables=cast_tables(B, cc["M_rows"], cc["N_cols"], cc["L"]))
    graft = w["policy"] == "graft"
    if graft:
        kw = dict(graft=w["graft"], template=graft_template(w), block=bool(w.get("block", False)))
    packed = bool(w.get("packed", False))
    draw = bool(w.get("draft_sampling", False))
    run = RoundRunner(w["policy"], B, V, w["K"], k, D, P, g["D_path"], g["m_cap"], spec.dtype, T=w["T"],
                      packed=packed, draw=draw, **kw)
    dt = torch.int16 if spec.dtype == synth.BF16 else torch.float32
    esz = 2 if spec.dtype == synth.BF16 else 4
    round_bytes = (D * B * k + B * P) * V * esz
    # recorded rounds: at least 16 (a mix of rounds) and at least 3x L2 of inputs, at most 48 GiB
    R = int(max(2, min(max(16, math.ceil(3 * L2_BYTES / round_bytes)), 256, (48 << 30) // round_bytes)))
    if args.record_rounds > 0:
        R = args.record_rounds
    block = bool(w.get("block", False))
    # a block drafter's rows: one [B][L][V] set per round (L = D), at rec_draft[r, 0]
    rec_draft = torch.empty((R, 1, B, D, V) if block else (R, D, B, k, V), dtype=dt, device="cuda")
    rec_target = torch.empty((R, B, P, V), dtype=dt, device="cuda")
    roots = torch.empty((R, B), dtype=torch.int32, device="cuda")
    M = torch.full((B, V, 8), -1, dtype=torch.int32, device="cuda") if graft else None
    dk = w["recipe"]["depthkey"]

    def salt_of(r):
        # Graft: successors are stationary and every round drafts from the same root tokens, so M learns
        # the rows its template reads (as when one position is drafted again); others: a new round each time
        return 0 if graft else (r << 8)

    def record(r, slot, widths=None):
        salt = salt_of(r)
        roots[slot] = torch.from_numpy(synth.root_tokens(w["seed"], salt, B, V)).cuda()

        def draft_rows(d, ftok):
            if d == 0:  # block rows: position j + 1 of request b, keyed on its root token
                ctx = roots[slot].repeat_interleave(D)
                pos = torch.arange(1, D + 1, dtype=torch.int32, device="cuda").repeat(B)
                synth.gen_rows_gpu(torch, spec, w["seed"], salt, synth.DRAFT, ctx, rec_draft[slot, 0], V,
                                   depth_dev=pos if dk else None, rows_per_b=D)
                if widths is not None:
                    widths.append(np.full(B, D))
                return rec_draft[slot, 0]
            F = 1 if d == 1 else k
            if widths is not None:
                widths.append((ftok[:, :F] >= 0).sum(1).cpu().numpy())
            if draw:  # every layer kept for the sampled verify: row (b, f) of layer d at rec_draft[slot, d - 1, b, f]
                synth.gen_rows_gpu(torch, spec, w["seed"], salt, synth.DRAFT, ftok.contiguous().view(-1),
                                   rec_draft[slot, d - 1], V, depth_add=d if dk else 0, rows_per_b=k)
                return rec_draft[slot, d - 1]
            ctx = ftok[:, :F].contiguous().view(-1)
            synth.gen_rows_gpu(torch, spec, w["seed"], salt, synth.DRAFT, ctx, rec_draft[slot, d - 1], V,
                               depth_add=d if dk else 0, rows_per_b=F)
            return rec_draft[slot, d - 1]

        def target_rows(meta):
            if packed:  # padding-free: request b's rows at meta.row_off[b] + i
                req, ctx, dep = synth.packed_row_map(torch, meta.row_off, meta.tokens, meta.depth)
                synth.gen_rows_gpu(torch, spec, w["seed"], salt, synth.TARGET, ctx, rec_target[slot], V,
                                   depth_dev=dep if dk else None, depth_add=1 if dk else 0, row_req_dev=req)
                return rec_target[slot]
            synth.gen_rows_gpu(torch, spec, w["seed"], salt, synth.TARGET, meta.tokens.view(-1), rec_target[slot],
                               V, depth_dev=meta.depth.view(-1) if dk else None, depth_add=1 if dk else 0,
                               rows_per_b=P)
            return rec_target[slot]

        run.draft_rows = rec_draft[slot]
        run.run(roots[slot], draft_rows, target_rows, seed=w["seed"], rnd=r, M=M, n0=512 * (1 + r % 16))

    # Graft: the configured warm-up rounds seed M, then more until it no longer changes (a steady M, so
    # that replayed rounds reproduce their recording); untimed
    warm = 0
    if graft:
        for warm in range(1, 41):
            before = M.clone()
            record(0, 0)
            torch.cuda.synchronize()
            if warm >= w.get("warmup_rounds", 5) and torch.equal(before, M):
                break

    # ---- recording pass (untimed): the model forwards are stood in for by the generator ----
    rec_out, rows_expand, rows_verify, npos_rec, act_rec = [], [], [], [], []
    for r in range(R):
        widths = []
        record(r, r, widths)
        torch.cuda.synchronize()
        rec_out.append((run.accept_len.clone(), run.bonus.clone(), run.m_dev.clone(), run.accept_path.clone()))
        rows_verify.append(int((run.meta.tokens >= 0).sum()))
        rows_expand.append([int(x.sum()) for x in widths])
        npos_rec.append(run.meta.n_pos.cpu().numpy().copy())
        act_rec.append(widths)
    assert dt_get_status(run.h) == 0, "device status set during recording"

    # ---- timed replay: the path only, on recorded inputs, captured as one CUDA graph ----
    def replay(r, timing=None):
        run.draft_rows = rec_draft[r]
        run.run(roots[r], lambda d, ftok: rec_draft[r, d - 1], lambda meta: rec_target[r], seed=w["seed"], rnd=r,
                M=M, n0=512 * (1 + r % 16), timing=timing)

    for i in range(warmup):
        replay(i % R)
    torch.cuda.synchronize()
    # consistency: a replayed round equals its recording
    replay(R - 1)
    torch.cuda.synchronize()
    consistent = bool(torch.equal(run.accept_len, rec_out[R - 1][0]) and torch.equal(run.bonus, rec_out[R - 1][1]))

    timing = EventTiming(torch)

    def capture(tm):
        gph = torch.cuda.CUDAGraph()
        cap_stream = torch.cuda.Stream()
        cap_stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(gph, stream=cap_stream):
                for s in range(steps):
                    replay(s % R, tm)
        torch.cuda.current_stream().wait_stream(cap_stream)
        gph.replay()  # untimed: uploads the graph
        torch.cuda.synchronize()
        return gph

    graph = capture(None)
    graph_ev = capture(timing)

    # K-step replays, each timed with events, for at least min_replay_s and 20 replays
    clocks = Clocks(local)
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    reps, t_begin = [], time.perf_counter()
    while len(reps) < 20 or (time.perf_counter() - t_begin < args.min_replay_s and len(reps) < 2000):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        graph.replay()
        t1.record()
        t1.synchronize()
        reps.append(t0.elapsed_time(t1))
    torch.cuda.synchronize()
    if world > 1:
        tdist.barrier()
    clk = clocks.stop()
    ms = float(np.median(reps))
    ms = max_over_ranks(ms, world)
    value = job_throughput(steps, world, ms)
    spread = {"replays": len(reps), "ms_min": float(np.min(reps)), "ms_p10": float(np.percentile(reps, 10)),
              "ms_median": float(np.median(reps)), "ms_p90": float(np.percentile(reps, 90)),
              "ms_max": float(np.max(reps))}
    graph_ev.replay()  # per-kernel events (not part of the timed region)
    torch.cuda.synchronize()

    peak, peak_kind = measured_peaks()
    kern = {}
    exp_bytes = sum(sum(rows_expand[s % R]) for s in range(steps)) * V * esz
    ver_bytes = sum(rows_verify[s % R] for s in range(steps)) * V * esz
    for kind, nbytes in (("expand", exp_bytes), ("prune_select", None), ("verify_rows", ver_bytes),
                         ("verify_accept", None), ("verify_sampled", ver_bytes)):
        t = timing.ms(kind)
        if not t:
            continue
        d = {"launches": len(t), "avg_us": 1e3 * float(np.mean(t)), "total_us_per_round": 1e3 * sum(t) / steps}
        if nbytes is not None:
            gbs = nbytes / (sum(t) / 1e3) / 1e9
            d.update(gbs=gbs, frac=gbs / peak, bytes_per_launch=nbytes / len(t))
        kern[kind] = d
    # the expansion layer as a whole (expansion kernel + pruning / frontier kernels)
    if "expand" in kern and "prune_select" in kern:
        lay = sum(timing.ms("expand")) + sum(timing.ms("prune_select"))
        kern["expand_layer"] = {"avg_us": 1e3 * lay / len(timing.ms("expand")),
                                "gbs": exp_bytes / (lay / 1e3) / 1e9}
    streaming = [k_ for k_ in ("expand", "verify_rows", "verify_sampled") if k_ in kern]
    top = max(streaming, key=lambda k_: kern[k_]["total_us_per_round"])
    tr = TRAFFIC_PER_ALGO_BYTE.get((label, top))
    names = {"expand": "expand_kernel (vocab softmax + top-K of the frontier rows, children, layer order)",
             "verify_rows": "verify_stream_kernel (argmax / softmax pieces of the used target rows)",
             "verify_sampled": "verify_stream_kernel + verify_sampled_kernel (target-row statistics, then the "
                               "recursive-residual walk; bytes: the used target rows)"}
    roofline = {"bound": "hbm", "achieved": kern[top]["gbs"], "peak": peak, "unit": "GB/s", "frac": kern[top]["frac"],
                "traffic": None if tr is None else tr * kern[top]["bytes_per_launch"], "kernel": names[top],
                "peak_source": peak_kind, "bytes_per_launch": kern[top]["bytes_per_launch"],
                "avg_launch_us": kern[top]["avg_us"]}
    # kernels of the library launched per round: reset + layer-1 frontier; per layer the expansion and
    # the pruning / frontier kernels (CAST: 1 fused; Graft: checkpoint + frontier; EAGLE: frontier; none
    # after the last layer except CAST's and Graft's pruning); verify count + rerank (CAST) or rerank,
    # retrieval (Graft), meta, 2 to 4 for the verify (the top-8 merge with Graft, the bonus draw with sampling),
    # the M refresh (Graft)
    per_layer = {"cast": 1, "graft": 2, "eagle": 1}[w["policy"]]
    last = 1 if w["policy"] in ("cast", "graft") else 0
    verify_launches = (3 if w["T"] == 1 else 2) + (1 if graft else 0)  # pass, (top-8,) walk, (bonus)
    launches = 2 + D + per_layer * (D - 1) + last + (2 if w["policy"] == "cast" else 1) + (1 if graft else 0) + 1 + \
        verify_launches + (1 if graft else 0)
    if block:  # reset, the block expansion, rerank, retrieval, meta, the verify, the M refresh
        launches = 5 + verify_launches + 1
    if draw:  # the sampled verify: the streaming pass and the walk (which draws the bonus itself)
        launches -= 1

    out = {"label": label, "value": value, "unit": UNIT, "ms_per_step": ms / steps, "steps": steps,
           "dtype": "bf16" if spec.dtype == synth.BF16 else "f32",
           "config": dict(workload_config(w, g, label),
                          inputs=f"{R} recorded synthetic rounds ({R * round_bytes / 2**30:.2f} GiB, > L2) replayed "
                                 "from HBM; every step reads a different round's buffers, no flush needed"),
           "roofline": roofline, "kernels": kern, "replay": spread, "replay_consistent": consistent,
           "rows_per_round": {"expand": rows_expand[:min(R, 16)], "verify": rows_verify[:min(R, 16)]},
           "gpu_launches": launches * steps, "clocks": clk}
    if graft:
        out["graft_warmup_rounds"] = warm

    if with_e2e:
        out["kv_commit"] = kv_commit_run(torch, run, rec_out, steps, R)
        out["verify_steady"] = verify_steady_run(torch, run, w, rec_target, R, esz)

    # ---- end to end through the public API with host buffers ----
    if with_e2e and args.e2e_steps > 0:
        out["e2e"] = e2e_run(torch, run, w, rec_draft, rec_target, roots, rec_out, act_rec, npos_rec, esz, M,
                             args.e2e_steps, world, args.e2e_gather_blocks)
    assert dt_get_status(run.h) == 0, "device status set during the timed region"
    del rec_draft, rec_target
    run.h.close()
    torch.cuda.empty_cache()
    return out


def verify_steady_run(torch, run, w, rec_target, R, esz, calls=64):
    """dt_verify (streaming pass + acceptance walk) of the last replayed round's tree against the recorded
    rounds' target rows, `calls` calls back to back in one CUDA graph (programmatic launch overlap
    kept), each reading a different round's rows (> L2 apart): the verify's steady state, as in a
    pipeline that keeps the GPU busy. Bytes = the tree's used rows x V x element size per call."""
    from dynamic_draft_tree_gb300 import dt_verify, dt_get_status, DT_GREEDY, DT_SAMPLE

    mode = DT_SAMPLE if w["T"] == 1 else DT_GREEDY
    nbytes = int((run.meta.tokens >= 0).sum()) * w["V"] * esz
    acc = torch.empty_like(run.accept_len)
    path = torch.empty_like(run.accept_path)
    bon = torch.empty_like(run.bonus)

    def call(i):
        dt_verify(run.h, run.meta, rec_target[i % R], mode, w["seed"], i, acc, path, bon, run.top8)

    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    gph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(gph, stream=cs):
            for i in range(calls):
                call(i)
    torch.cuda.current_stream().wait_stream(cs)
    times = []
    for _ in range(6):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        gph.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert dt_get_status(run.h) == 0
    us = float(np.median(times[1:])) * 1e3 / calls
    peak, _ = measured_peaks()
    return {"us_per_call": us, "bytes_per_call": nbytes, "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak,
            "note": "dt_verify (streaming pass + walk) calls back to back in one CUDA graph, median of 5 replays; "
                    "not part of value"}


KV_ROW_BYTES = 32 * 2 * 8 * 128 * 2  # one token's keys and values: 32 layers, 8 KV heads of 128, bf16


def kv_commit_run(torch, run, rec_out, steps, R):
    """Accepted-path KV compaction (dt_commit_kv) after each recorded round's verify, with KV rows of
    KV_ROW_BYTES (an 8B-parameter model's cache row): the calls of `steps` rounds back to back, timed
    with events; bytes moved = 2 x rows committed x row size."""
    from dynamic_draft_tree_gb300 import dt_commit_kv, dt_get_status

    B, P = run.meta.tokens.shape
    Dp = run.accept_path.shape[1]
    L = max(steps, 3) * Dp  # room for the warm-up calls and for each replay's `steps` calls
    tmp = torch.empty((B, P, KV_ROW_BYTES), dtype=torch.uint8, device="cuda")
    cache = torch.empty((B, L, KV_ROW_BYTES), dtype=torch.uint8, device="cuda")
    cache_len = torch.zeros((B,), dtype=torch.int32, device="cuda")
    rows = sum(int((rec_out[s % R][0] + 1).sum()) for s in range(steps))
    for s in range(3):  # warm-up
        dt_commit_kv(run.h, tmp, cache, cache_len, rec_out[s % R][0], rec_out[s % R][3])
    cache_len.zero_()
    torch.cuda.synchronize()
    # the calls of `steps` rounds captured as one CUDA graph (device time, not the host's call rate),
    # each replay starting again from an empty cache
    gph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(gph, stream=cs):
            for s in range(steps):
                dt_commit_kv(run.h, tmp, cache, cache_len, rec_out[s % R][0], rec_out[s % R][3])
    torch.cuda.current_stream().wait_stream(cs)
    times = []
    for _ in range(6):
        cache_len.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        gph.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert dt_get_status(run.h) == 0
    us = float(np.median(times[1:])) * 1e3 / steps
    nbytes = 2.0 * rows / steps * KV_ROW_BYTES
    peak, _ = measured_peaks()
    del tmp, cache
    return {"row_bytes": KV_ROW_BYTES, "rows_per_call": rows / steps, "avg_us": us,
            "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak,
            "note": "the calls of `steps` rounds (two launches each) as one CUDA graph, median of 5 replays; "
                    "not part of the round's graph"}


def e2e_run(torch, run, w, rec_draft, rec_target, roots, rec_out, act_rec, npos_rec, esz, M, steps, world,
            gather_blocks=0):
    """The recorded round 0 through the public API from pinned host buffers, every step: the rows the
    round reads (each request's active frontier rows per layer, its used target positions) and the roots
    copied host -> device, the round, and the accepted lengths, paths and bonus tokens copied back.
    The inputs are double-buffered: step s + 1's copies run on a copy stream while step s runs. With
    gather_blocks > 0 the copies are one kernel of that many CTAs reading the pinned host memory
    through its device mapping (checked once against plain copies first); else one DMA copy per row
    block."""
    B, k, V = w["B"], w["k"], w["V"]
    h_draft = rec_draft[0].cpu().pin_memory()
    h_target = rec_target[0].cpu().pin_memory()
    h_roots = roots[0].cpu().pin_memory()
    out_len = torch.empty((B,), dtype=torch.int32).pin_memory()
    out_bonus = torch.empty((B,), dtype=torch.int32).pin_memory()
    out_path = torch.empty(tuple(run.accept_path.shape), dtype=torch.int32).pin_memory()
    # contiguous row blocks the round reads: layer d, request b, frontier slots 0..cnt-1 (row (b F + f) of
    # that layer's [B][F][V] buffer); target rows 0..n_pos[b]-1 of request b
    chunks = []
    for d, cnt in enumerate(act_rec[0]):
        F = w["D"] if run.block else (1 if d == 0 else k)  # a block drafter: one [B][L][V] set
        for b in range(B):
            if cnt[b] > 0:
                chunks.append(("d", d, b * F, int(cnt[b])))
    if run.packed:  # padding-free: the used target rows are rows 0 .. sum n_pos - 1
        chunks.append(("t", 0, 0, int(np.sum(npos_rec[0]))))
    else:
        for b in range(B):
            if npos_rec[0][b] > 0:
                chunks.append(("t", 0, b * run.P, int(npos_rec[0][b])))
    bi = sum(c[3] for c in chunks) * V * esz + h_roots.numel() * 4
    bo = (out_len.numel() + out_bonus.numel() + out_path.numel()) * 4
    bufs = [(torch.zeros_like(roots[0]), torch.zeros_like(rec_draft[0]), torch.zeros_like(rec_target[0]))
            for _ in range(2)]
    hd = h_draft.view(h_draft.shape[0], -1, V)
    ht = h_target.view(-1, V)
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]

    # the same row blocks as (source, destination, bytes) spans for the gather kernel
    import synth
    spans = None
    if gather_blocks > 0:
        src0 = [synth.host_device_ptr(t) for t in (h_roots, h_draft, h_target)]
        if all(p is not None for p in src0):
            spans = []
            row_b = V * esz
            per_layer = hd.shape[1]
            for r_, dr_, tg_ in bufs:
                sp = [(src0[0], r_.data_ptr(), h_roots.numel() * 4)]
                for kind, d, r0, n in chunks:
                    off = ((d * per_layer + r0) if kind == "d" else r0) * row_b
                    src_t, dst_t = (h_draft, dr_) if kind == "d" else (h_target, tg_)
                    assert off + n * row_b <= src_t.numel() * esz and off + n * row_b <= dst_t.numel() * esz
                    sp.append((src0[1 if kind == "d" else 2] + off, dst_t.data_ptr() + off, n * row_b))
                spans.append(torch.tensor(sp, dtype=torch.int64, device="cuda"))

    def copy_inputs(i):
        r_, dr_, tg_ = bufs[i % 2]
        dd = dr_.view(dr_.shape[0], -1, V)
        tt = tg_.view(-1, V)
        if spans is not None:
            with torch.cuda.stream(copy_stream):
                synth.gather_spans_gpu(torch, spans[i % 2], gather_blocks, copy_stream)
                copied[i % 2].record(copy_stream)
            return
        with torch.cuda.stream(copy_stream):
            r_.copy_(h_roots, non_blocking=True)
            for kind, d, r0, n in chunks:
                if kind == "d":
                    dd[d, r0:r0 + n].copy_(hd[d, r0:r0 + n], non_blocking=True)
                else:
                    tt[r0:r0 + n].copy_(ht[r0:r0 + n], non_blocking=True)
            copied[i % 2].record(copy_stream)

    if spans is not None:  # the gather's bytes, checked once against plain copies of the same blocks
        for i in range(2):
            copy_inputs(i)
        torch.cuda.synchronize()
        for r_, dr_, tg_ in bufs:
            dd = dr_.view(dr_.shape[0], -1, V)
            tt = tg_.view(-1, V)
            ok = torch.equal(r_.cpu(), h_roots)
            for kind, d, r0, n in chunks:
                ok = ok and (torch.equal(dd[d, r0:r0 + n].cpu(), hd[d, r0:r0 + n]) if kind == "d"
                             else torch.equal(tt[r0:r0 + n].cpu(), ht[r0:r0 + n]))
            if not ok:
                raise RuntimeError("e2e: the host-row gather does not reproduce the copied rows")
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    copy_stream.wait_event(e0)
    copy_inputs(0)
    for s in range(steps):
        cur = torch.cuda.current_stream()
        cur.wait_event(copied[s % 2])
        r_, dr_, tg_ = bufs[s % 2]
        if s + 1 < steps:  # the other buffer set: step s - 1 finished reading it (synchronised below)
            copy_inputs(s + 1)
        run.run(r_, lambda d, ftok, dr_=dr_: dr_[d - 1], lambda meta, tg_=tg_: tg_, seed=w["seed"], rnd=0, M=M,
                n0=512)
        out_len.copy_(run.accept_len, non_blocking=True)
        out_bonus.copy_(run.bonus, non_blocking=True)
        out_path.copy_(run.accept_path, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    copy_stream.synchronize()
    e1.record()
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    consistent = bool(torch.equal(out_len.cuda(), rec_out[0][0]) and torch.equal(out_bonus.cuda(), rec_out[0][1]))
    if not consistent:
        print("e2e mismatch:", out_len.tolist(), rec_out[0][0].tolist(), out_bonus.tolist(), rec_out[0][1].tolist(),
              file=sys.stderr)
    return {"value": job_throughput(steps, world, e_ms), "unit": UNIT, "h2d_bytes_per_step": int(bi),
            "d2h_bytes_per_step": int(bo), "double_buffered": True, "consistent": consistent,
            "copies": "the rows the round reads (active frontier rows per layer and request, used target "
                      "positions), as recorded",
            "h2d_method": (f"one kernel of {gather_blocks} CTAs reading the pinned host rows through their device "
                           f"mapping" if spans is not None else "one DMA copy per row block")}


def run_ours(args):
    import torch
    import torch.distributed as tdist

    import __graft_entry__

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    __graft_entry__.build()  # every rank builds (or finds) the library before importing it

    head = measure_workload(args.workload, args.steps, args.warmup, args, rank, world, local, with_e2e=True)
    per_config = {}
    for name in [x for x in args.workloads.split(",") if x and x != args.workload]:
        r = measure_workload(name, min(args.steps, args.per_config_steps), args.warmup, args, rank, world, local,
                             with_e2e=False)
        per_config[r.pop("label")] = r
    if rank != 0:
        return None
    head.pop("label")
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded counter-hash logits standing in for the draft/target forwards)",
        "config": dict(head["config"], parallelism=f"replicas x{world} (independent batches)"),
        "roofline": head["roofline"], "kernels": head["kernels"], "replay": head["replay"],
        "e2e": head.get("e2e"), "gpu_launches": head["gpu_launches"],
        "replay_consistent": head["replay_consistent"], "rows_per_round": head["rows_per_round"],
        "kv_commit": head.get("kv_commit"), "verify_steady": head.get("verify_steady"),
        "clocks": head["clocks"], "per_config": per_config,
    }
    return line


def run_reference(args):
    """The fp64 CPU oracle as it stands, on a bounded sample of the same workload."""
    rank, world, local = dist_env()
    if rank != 0:
        return None
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import harness
    from synth.workloads import geometry

    w, label = workload_of(args.workload, parse_sizes(args.sizes))
    g = geometry(w)
    # the oracle's rows come from a warm cache so that only the oracle itself is timed; the run is
    # bounded in time (the oracle takes seconds per round), so at most `budget` seconds of rounds are
    # timed out of the requested steps
    budget = 60.0
    seen = set()
    for s in range(min(args.warmup, 2)):
        harness.oracle_round(w, s % 4)
        seen.add(s % 4)
    times = []
    for s in range(args.steps):
        rnd = s % 4
        if rnd not in seen:
            harness.oracle_round(w, rnd)  # warms the row cache of this round
            seen.add(rnd)
        t = time.perf_counter()
        harness.oracle_round(w, rnd)
        times.append(time.perf_counter() - t)
        if sum(times) > budget:
            break
    sec = float(np.sum(times))
    value = len(times) / sec
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(workload_config(w, g, label), parallelism="1 host process"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{len(times)} of {args.steps} requested rounds of the workload, "
                                       f"time-bounded to {budget:.0f} s (rows pre-generated)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def cpu_baseline_sample(name, seconds=12.0, sizes=None):
    """Oracle rounds/s on the host, single process, rows pre-generated: bounded to ~seconds. Also counts
    the rounds whose oracle decision gaps fall below 1e-5 relative (the parity tests redraw those): the
    sampled rounds are the benchmark's own rounds 0, 1, ... (same seeds, salts and prefix lengths)."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import harness

    w, _ = workload_of(name, sizes)
    n, sec, rnd, redrawn, hit = 0, 0.0, 0, 0, 0
    while sec < seconds and n < 50:
        _, _, rej = harness.oracle_round(w, rnd)
        redrawn += rej
        hit += rej > 0
        t = time.perf_counter()
        harness.oracle_round(w, rnd)
        sec += time.perf_counter() - t
        n += 1
        rnd += 1
    base = {"value": n / sec, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} full rounds of the {name} workload, rows pre-generated (only the oracle timed)"}
    seeds = {"rounds_checked": n, "rounds_with_near_tie": hit, "request_redraws": redrawn,
             "rule": "a round is redrawn when an oracle decision gap is below 1e-5 relative"}
    return base, seeds


def main():
    args = parse()
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_ours(args)
        if line is not None and not args.no_cpu_baseline:
            line["cpu_baseline"], line["seed_redraws"] = cpu_baseline_sample(args.workload, sizes=parse_sizes(args.sizes))
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
