"""Benchmark of the draft-tree hot path on the CAST batch workload (B=8, V=128256, bf16).

One step = one complete round of the path (EAGLE-2 expansion with CAST width/depth pruning for up
to 8 layers, CAST verify count, rerank, flatten + metadata, greedy verify) over one batch of B=8
requests, with its inputs already in HBM. The draft and target model forwards are not part of the
path: their logits are produced by the seeded generator in an untimed recording pass (R rounds,
each ~289 MB, so every timed step reads a different round: inputs larger than L2), and the timed
steps replay the path on them. The replay must reproduce the recording pass's outputs bit for bit.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own independent batch (requests shard across GPUs with no
exchange: weak scaling). The reference arm times the fp64 CPU oracle on a bounded sample.
"""
import argparse
import json
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="cast")
    ap.add_argument("--rec-rounds", type=int, default=16)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
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


def workload_config(w, g):
    return {"workload": f"{w['policy']} tree round, B={w['B']}, V={w['V']}, bf16 logits, K={w['K']}, "
                        f"k<={w['k']}, depth<={w['D']}, m<={g['m_cap']}, greedy verify",
            "B": w["B"], "V": w["V"], "K": w["K"], "k_max": w["k"], "D_max": w["D"], "m_cap": g["m_cap"],
            "global_batch": w["B"], "inputs": "recorded synthetic rounds replayed from HBM; every step reads a "
                                              "different round (inputs larger than L2, no flush needed)"}


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
                                          "--format=csv,noheader,nounits", "-lms", "200"],
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


# DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) per algorithmic byte of each row-pass
# kernel, from the captures summarised in profiles/ (None once the kernel has changed since).
TRAFFIC_PER_ALGO_BYTE = {"dt_expand_layer": 20.685056e6 / (80 * 256512),   # layer 2 of a CAST round, 80 rows
                         "dt_verify": (84.258048e6 + 1.573120e6) / (328 * 256512)}  # 328 used rows


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


def run_ours(args):
    import torch
    import torch.distributed as tdist

    import synth
    from synth.workloads import WORKLOADS, spec_for, geometry, cast_tables, chain_template
    import __graft_entry__

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    __graft_entry__.build()  # every rank builds (or finds) the library before importing it
    from dynamic_draft_tree_gb300 import dt_get_status
    from dynamic_draft_tree_gb300.rounds import RoundRunner

    w = dict(WORKLOADS[args.workload])
    w["seed"] = w["seed"] + 1000 * rank  # independent batch per rank
    g = geometry(w)
    spec = spec_for(w)
    B, V, k, D, P = w["B"], w["V"], w["k"], g["D_max"], g["P"]
    kw = {}
    if w["policy"] == "cast":
        cc = w["cast"]
        kw = dict(cast=dict(cc), cast_tables=cast_tables(B, cc["M_rows"], cc["N_cols"], cc["L"]))
    if w["policy"] == "graft":
        kw = dict(graft=w["graft"], template=chain_template(k, w["D"]))
    run = RoundRunner(w["policy"], B, V, w["K"], k, D, P, g["D_path"], g["m_cap"], spec.dtype, T=w["T"], **kw)
    dt = torch.int16 if spec.dtype == synth.BF16 else torch.float32
    esz = 2 if spec.dtype == synth.BF16 else 4
    R = args.rec_rounds
    rec_draft = torch.empty((R, D, B, k, V), dtype=dt, device="cuda")
    rec_target = torch.empty((R, B, P, V), dtype=dt, device="cuda")
    roots = torch.empty((R, B), dtype=torch.int32, device="cuda")
    M = None
    if w["policy"] == "graft":
        M = torch.full((B, V, 8), -1, dtype=torch.int32, device="cuda")
    dk = w["recipe"]["depthkey"]

    # ---- recording pass (untimed): the model forwards are stood in for by the generator ----
    rec_out, rows_expand, rows_verify = [], [], []
    for r in range(R):
        salt = (r << 8)
        roots[r] = torch.from_numpy(synth.root_tokens(w["seed"], salt, B, V)).cuda()
        widths = []

        def draft_rows(d, ftok, r=r, salt=salt):
            F = 1 if d == 1 else k
            ctx = ftok[:, :F].contiguous().view(-1)
            widths.append(int((ctx >= 0).sum()))
            synth.gen_rows_gpu(torch, spec, w["seed"], salt, synth.DRAFT, ctx, rec_draft[r, d - 1], V,
                               depth_add=d if dk else 0, rows_per_b=F)
            return rec_draft[r, d - 1]

        def target_rows(meta, r=r, salt=salt):
            synth.gen_rows_gpu(torch, spec, w["seed"], salt, synth.TARGET, meta.tokens.view(-1), rec_target[r],
                               V, depth_dev=meta.depth.view(-1) if dk else None, depth_add=1 if dk else 0,
                               rows_per_b=P)
            return rec_target[r]

        run.run(roots[r], draft_rows, target_rows, seed=w["seed"], rnd=r, M=M, n0=512 * (1 + r % 16))
        torch.cuda.synchronize()
        rec_out.append((run.accept_len.clone(), run.bonus.clone(), run.m_dev.clone()))
        # rows each kernel actually reads in this round
        rows_verify.append(int((run.meta.tokens >= 0).sum()))
        rows_expand.append(widths)
    assert dt_get_status(run.h) == 0, "device status set during recording"

    # ---- timed replay: the path only, on recorded inputs, captured as one CUDA graph ----
    ev_exp = []   # [start, end] events around each expand launch (graph event-record nodes)
    ev_ver = []

    def new_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return torch.cuda.Event(enable_timing=True)

    def replay(r, timed):
        def draft_rows(d, ftok):
            if timed:
                e0 = new_event()
                e0.record()
                ev_exp.append([e0, None])
            return rec_draft[r, d - 1]

        def target_rows(meta):
            if timed:
                e0 = new_event()
                e0.record()
                ev_ver.append([e0, None])
            return rec_target[r]

        run.run(roots[r], draft_rows, target_rows, seed=w["seed"], rnd=r, M=M, n0=512 * (1 + r % 16),
                after_expand=(lambda: _close(ev_exp)) if timed else None,
                after_verify=(lambda: _close(ev_ver)) if timed else None)

    def _close(lst):
        e1 = new_event()
        e1.record()
        lst[-1][1] = e1

    for i in range(args.warmup):
        replay(i % R, False)
    torch.cuda.synchronize()
    # consistency: a replayed round equals its recording
    replay(0, False)
    torch.cuda.synchronize()
    consistent = bool(torch.equal(run.accept_len, rec_out[0][0]) and torch.equal(run.bonus, rec_out[0][1]))

    # two graphs of the same K steps: the timed one holds the path only; the other adds event records
    # around each expansion and verify launch for the per-kernel figures (events between launches
    # would also split the programmatic launch overlap of the kernels they separate)
    def capture(with_events):
        g = torch.cuda.CUDAGraph()
        cap_stream = torch.cuda.Stream()
        cap_stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(g, stream=cap_stream):
                for s in range(args.steps):
                    replay(s % R, with_events)
        torch.cuda.current_stream().wait_stream(cap_stream)
        g.replay()  # untimed: uploads the graph
        torch.cuda.synchronize()
        return g

    graph = capture(False)
    graph_ev = capture(True)

    clocks = Clocks(local)
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    graph.replay()
    t1.record()
    torch.cuda.synchronize()
    if world > 1:
        tdist.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    graph_ev.replay()  # per-kernel events (not part of the timed region)
    torch.cuda.synchronize()
    ms = max_over_ranks(ms, world)
    value = job_throughput(args.steps, world, ms)

    # per-kernel figures from the live events
    exp_ms = [a.elapsed_time(b) for a, b in ev_exp]
    ver_ms = [a.elapsed_time(b) for a, b in ev_ver]
    exp_bytes = sum(sum(rows_expand[s % R]) for s in range(args.steps)) * V * esz
    ver_bytes = sum(rows_verify[s % R] for s in range(args.steps)) * V * esz
    peak, peak_kind = measured_peaks()
    ver_gbs = ver_bytes / (sum(ver_ms) / 1e3) / 1e9
    exp_gbs = exp_bytes / (sum(exp_ms) / 1e3) / 1e9
    # roofline of the kernel with the most time per round (expansion: D launches; verify: one)
    rl = {"dt_expand_layer": (exp_gbs, exp_bytes / len(exp_ms), 1e3 * sum(exp_ms) / len(exp_ms), sum(exp_ms),
                              "expand_kernel (vocab softmax + top-K per frontier node)"),
          "dt_verify": (ver_gbs, ver_bytes / len(ver_ms), 1e3 * sum(ver_ms) / len(ver_ms), sum(ver_ms),
                        "dt_verify (verify row pass + acceptance walk)")}
    top = max(rl, key=lambda k: rl[k][3])
    gbs, bpl, us, _, kname = rl[top]
    tr = TRAFFIC_PER_ALGO_BYTE.get(top)
    roofline = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                "traffic": None if tr is None else tr * bpl, "kernel": kname, "peak_source": peak_kind,
                "bytes_per_launch": bpl, "avg_launch_us": us}
    launches_per_round = 1 + (D if w["policy"] != "cast" else 1) + D + \
        (D if w["policy"] in ("cast", "graft") else 0) + \
        (2 if w["policy"] == "cast" else 1) + 1 + (3 if w["T"] == 1 else 2) + \
        (2 if w["policy"] == "graft" else 0)

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if args.e2e_steps > 0:
        h_draft = torch.empty_like(rec_draft[0], device="cpu").pin_memory()
        h_target = torch.empty_like(rec_target[0], device="cpu").pin_memory()
        h_draft.copy_(rec_draft[0])
        h_target.copy_(rec_target[0])
        h_roots = roots[0].cpu().pin_memory()
        out_len = torch.empty((B,), dtype=torch.int32).pin_memory()
        out_bonus = torch.empty((B,), dtype=torch.int32).pin_memory()
        out_path = torch.empty(tuple(run.accept_path.shape), dtype=torch.int32).pin_memory()
        d_draft = torch.empty_like(rec_draft[0])
        d_target = torch.empty_like(rec_target[0])
        d_roots = torch.empty_like(roots[0])
        bi = h_draft.numel() * esz + h_target.numel() * esz + h_roots.numel() * 4
        bo = (out_len.numel() + out_bonus.numel() + out_path.numel()) * 4
        # Double-buffered inputs: step s + 1's rows are copied (on a copy stream) while step s runs,
        # into the other buffer set, which step s - 1 has finished reading (every step ends with a
        # synchronisation on its results). Every step's copy is inside the timed region.
        d_draft2, d_target2, d_roots2 = torch.empty_like(d_draft), torch.empty_like(d_target), torch.empty_like(d_roots)
        bufs = [(d_roots, d_draft, d_target), (d_roots2, d_draft2, d_target2)]
        copy_stream = torch.cuda.Stream()
        copied = [torch.cuda.Event(), torch.cuda.Event()]

        def copy_inputs(i):
            r_, dr_, tg_ = bufs[i % 2]
            with torch.cuda.stream(copy_stream):
                r_.copy_(h_roots, non_blocking=True)
                dr_.copy_(h_draft, non_blocking=True)
                tg_.copy_(h_target, non_blocking=True)
                copied[i % 2].record(copy_stream)

        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        copy_stream.wait_event(e0)
        copy_inputs(0)
        for s in range(args.e2e_steps):
            cur = torch.cuda.current_stream()
            cur.wait_event(copied[s % 2])
            r_, dr_, tg_ = bufs[s % 2]
            if s + 1 < args.e2e_steps:
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
        e_ms = e0.elapsed_time(e1)
        e_ms = max_over_ranks(e_ms, world)
        e2e = {"value": job_throughput(args.e2e_steps, world, e_ms), "unit": UNIT, "h2d_bytes_per_step": int(bi),
               "d2h_bytes_per_step": int(bo), "double_buffered": True}
        e2e["consistent"] = bool(torch.equal(out_len.cuda(), rec_out[0][0]) and
                                 torch.equal(out_bonus.cuda(), rec_out[0][1]))
        if not e2e["consistent"]:
            print("e2e mismatch:", out_len.tolist(), rec_out[0][0].tolist(), out_bonus.tolist(),
                  rec_out[0][1].tolist(), file=sys.stderr)

    assert dt_get_status(run.h) == 0, "device status set during the timed region"
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if spec.dtype == synth.BF16 else "f32",
        "data": "synthetic (seeded counter-hash logits standing in for the draft/target forwards)",
        "config": dict(workload_config(w, g), parallelism=f"replicas x{world} (independent batches)"),
        "roofline": roofline,
        "kernels": {"dt_verify": {"gbs": ver_gbs, "avg_us": 1e3 * float(np.mean(ver_ms)),
                                  "avg_bytes": ver_bytes / len(ver_ms), "rows_per_round": rows_verify},
                    "dt_expand_layer": {"gbs": exp_gbs, "avg_us": 1e3 * float(np.mean(exp_ms)),
                                        "avg_bytes": exp_bytes / len(exp_ms), "launches_per_round": D,
                                        "rows_per_round": rows_expand}},
        "e2e": e2e,
        "gpu_launches": launches_per_round * args.steps,
        "replay_consistent": consistent,
        "clocks": clk,
    }
    return line


def run_reference(args):
    """The fp64 CPU oracle as it stands, on a bounded sample of the same workload."""
    rank, world, local = dist_env()
    if rank != 0:
        return None
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import harness
    from synth.workloads import WORKLOADS, geometry

    w = dict(WORKLOADS[args.workload])
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
            "data": "synthetic", "config": dict(workload_config(w, g), parallelism="1 host process"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{len(times)} of {args.steps} requested rounds of the workload, "
                                       f"time-bounded to {budget:.0f} s (rows pre-generated)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def cpu_baseline_sample(seconds=12.0):
    """Oracle rounds/s on the host, single process, rows pre-generated: bounded to ~seconds."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import harness
    from synth.workloads import WORKLOADS

    w = dict(WORKLOADS["cast"])
    n, sec, rnd = 0, 0.0, 0
    while sec < seconds and n < 50:
        harness.oracle_round(w, rnd)
        t = time.perf_counter()
        harness.oracle_round(w, rnd)
        sec += time.perf_counter() - t
        n += 1
        rnd += 1
    return {"value": n / sec, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} full rounds of the CAST workload, rows pre-generated (only the oracle timed)"}


def main():
    args = parse()
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_ours(args)
        if line is not None and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_sample()
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
