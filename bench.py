#!/usr/bin/env python3
"""Benchmark of the speculative-decoding verify-and-commit step on one GB300.

One step is one call of the entry point the workload names: row statistics
over every logits row, acceptance, the correction / bonus draw and the KV
commit for the whole batch, on inputs already resident in HBM.  The default
workload is the DFlash-style block (64 requests x 16 rows, V = 151936, bf16
logits, full p/q rejection with residual sampling and bonus).

Prints one JSON line on rank 0.  `--impl reference` times the fp64 CPU oracle
on the host cores instead (the only reference this path has).
Multi-GPU (torchrun): every rank verifies its own batch (weak scaling, no
collective on the data path); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified rows/s"
UNIT = "rows/s"
# statistics, row merge, then for greedy calls of the benchmark's batch sizes (at most 32 requests) one kernel
# that accepts and commits, else acceptance, the sampler (with the commit) and the draws
KERNELS_PER_STEP = {"greedy_chain": 3, "greedy_tree": 3, "rejection_chain": 5, "rejection_ragged": 5,
                    "target_only_tree": 5, "rejection_chain_sparse": 5, "sample_match_chain": 5}
STATS_SOURCES = ("reject_row_vocab_gb300/csrc/sv_stats.cu", "reject_row_vocab_gb300/csrc/sv_device.cuh")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--tree-mode", default="target_only_tree", choices=["greedy_tree", "target_only_tree"])
    ap.add_argument("--eager", action="store_true", help="launch every step from Python instead of a CUDA graph")
    ap.add_argument("--graph-steps", type=int, default=100, help="steps captured per CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--match", action="store_true",
                    help="rejection-chain workloads verified by independent target sampling and prefix match")
    ap.add_argument("--q-cands", type=int, default=0,
                    help="rejection chains only: q given as K candidates per row (sparse) instead of dense rows")
    ap.add_argument("--kernel", default="step", choices=["step", "dspark", "tree-build"],
                    help="step: the verify step (default); dspark: the verify-length scheduler (256 requests x 15 "
                         "drafts); tree-build: tree-verify inputs from parent arrays (64 trees x 64 nodes)")
    ap.add_argument("--flush-l2", default="auto", choices=["auto", "on", "off"],
                    help="write a buffer larger than L2 before every step (auto: when the logits are smaller "
                         "than twice the L2); the step time then excludes the flushes")
    ap.add_argument("--stats-events-every", type=int, default=10,
                    help="record the row-statistics kernel's events around one launch in this many (1: every "
                         "launch); event nodes between kernels stop the next launch from overlapping the previous")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget-s", type=float, default=150.0)
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# Ranks
# ---------------------------------------------------------------------------


class Ranks:
    """torchrun environment; every data-path step stays local to its rank."""

    def __init__(self, backend: str | None = None):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.backend = backend
        if self.world > 1:
            import torch.distributed as dist
            if backend is None:
                import torch
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            self.backend = backend
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "max")

    def sum(self, x: float) -> float:
        return self._reduce(x, "sum")

    def _reduce(self, x: float, op: str) -> float:
        if self.pg is None:
            return float(x)
        import torch
        dev = "cuda" if self.backend == "nccl" else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def rank_seed(index: int, rank: int) -> int:
    """Rank r verifies its own batch: the named workload's seed, shifted per rank."""
    return 1000 + index + 100 * rank


def whole_job_value(units_per_rank: list, max_seconds: float) -> float:
    return float(sum(units_per_rank)) / max_seconds


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "25", "-i", self.gpu_id], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    def stop(self) -> dict:
        if self.proc is None:
            return {"unavailable": "nvidia-smi not runnable"}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[3], parts[4:]))
            except ValueError:
                continue
        os.unlink(self.file.name)
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        use = inside if inside else rows
        if not use:
            return {"unavailable": "no samples"}
        reasons = sorted({n for r in use for n, v in zip(self.NAMES, r[4]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "in_window": bool(inside)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device_index)


# ---------------------------------------------------------------------------
# Shared pieces
# ---------------------------------------------------------------------------


def measured_peaks() -> tuple:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def stats_traffic(w) -> float | None:
    """dram bytes per row-statistics launch from the committed ncu summary, if the kernel is unchanged and the
    summary covers this workload's logits."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    base = rec.get("workload_name")
    if w.kind == "sample_match_chain" or not (w.name == base or w.name.startswith("%s_sparse_q" % base)):
        return None
    h = hashlib.sha256()
    for p in STATS_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec.get("bytes_per_full_launch")


def make_workload(args, rank: int = 0):
    from reject_row_vocab_gb300 import workload as wl
    if args.q_cands > 0:  # the same chain shape with a K-candidate (selector) q instead of dense q rows
        if args.config not in (2, 4):
            raise SystemExit("--q-cands applies to the rejection-chain workloads (2, 4)")
        shape = {2: dict(batch=8, m=7, boost=6.0, temperature=0.8, noise_sigma=1.0, name="c2_rejection_chain"),
                 4: dict(batch=64, m=15, boost=0.0, temperature=1.0, noise_sigma=1.5, name="c4_dflash_block")}
        kw = dict(shape[args.config])
        kw["name"] += "_sparse_q%d" % args.q_cands
        return wl.rejection_chain_sparse(vocab=151936, dtype="bf16", K=args.q_cands, sigma=3.0,
                                         seed=rank_seed(args.config, rank), **kw)
    kw = {"seed": rank_seed(args.config, rank)}
    if args.match:
        if args.config not in (2, 4):
            raise SystemExit("--match applies to the rejection-chain workloads (2, 4)")
        import dataclasses
        w = wl.config(args.config, **kw)
        return dataclasses.replace(w, kind="sample_match_chain", q=None, name=w.name + "_sample_match")
    if args.config == 3:
        kw["mode"] = args.tree_mode
    return wl.config(args.config, **kw)


L2_BYTES = 129e6
FLUSH_BYTES = 256 << 20  # about twice the L2


def event_context(logits, flush_l2, cap, pairs: int = 20, replays: int = 5):
    """The statistics kernel's timing, applied to two other kernels in the same setting (the same L2 flush before
    each, the same event nodes in a CUDA graph when the bench uses one): an empty kernel, whose span is the fixed
    cost of the timing itself, and torch.sum over the same logits, what a plain library reduction reaches on the
    same bytes.  Medians in us; None when this torch cannot record event nodes inside a graph."""
    import torch
    try:
        evs = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
               for _ in range(pairs)]
    except TypeError:
        return None
    kernels = {"empty_kernel_us": lambda: torch.cuda._sleep(0),
               "torch_sum_us": lambda: torch.sum(logits, dtype=torch.float32)}
    res = {}
    for name, fn in kernels.items():
        def body():
            for a, b in evs:
                if flush_l2 is not None:
                    flush_l2()
                a.record()
                fn()
                b.record()
        if cap is not None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                body()
            run = g.replay
        else:
            run = body
        run()
        torch.cuda.synchronize()
        ts = []
        for _ in range(replays):
            run()
            torch.cuda.synchronize()
            ts += [a.elapsed_time(b) * 1e3 for a, b in evs]
        res[name] = statistics.median(ts)
    return res


def stats_event_slots(n: int, every: int) -> list:
    """For each of n launches, the index of the event pair recorded around its row-statistics kernel, or None:
    one launch in `every` (the first of each group) is instrumented, so most steps run without event nodes."""
    every = max(1, every)
    return [k // every if k % every == 0 else None for k in range(max(1, n))]


def flush_wanted(args, w) -> bool:
    if args.flush_l2 == "auto":
        return w.logit_bytes() < 2 * L2_BYTES
    return args.flush_l2 == "on"


def describe(w, flush: bool) -> dict:
    if flush:
        l2 = ("L2 flushed before every step (a %d MB write, then a read of as much); the step time is the span of flush + step minus "
              "that of the flushes alone, the row-statistics time its own events" % (FLUSH_BYTES >> 20))
    elif w.logit_bytes() > L2_BYTES:
        l2 = "inputs larger than L2 (%.0f MB of logits vs 129 MB L2)" % (w.logit_bytes() / 1e6)
    else:
        l2 = "inputs smaller than L2, not flushed: repeated steps may hit in L2"
    return {"workload": w.name, "kind": w.kind, "batch": w.batch, "rows": w.rows, "vocab": w.vocab,
            "max_len": w.max_len, "logit_dtype": w.dtype, "logit_bytes": w.logit_bytes(), "l2": l2,
            "seed": w.meta.get("seed")}


def oracle_run(w, threads: int):
    import oracle
    if w.kind == "greedy_chain":
        return oracle.verify_chain(w, greedy_all=True, threads=threads)
    if w.kind in ("rejection_chain", "rejection_ragged"):
        return oracle.verify_chain(w, threads=threads)
    if w.kind == "rejection_chain_sparse":
        return oracle.verify_chain_sparse(w, threads=threads)
    if w.kind == "sample_match_chain":
        from oracle import match
        return match.verify_chain_match(w)
    return oracle.verify_tree(w, "greedy" if w.kind == "greedy_tree" else "target_only", threads=threads)


def time_oracle(w, seconds: float, threads: int) -> dict:
    """The oracle, as it stands, on the host cores over the full batch, repeated for ~`seconds`."""
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_run(w, threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    if w.kind == "sample_match_chain":  # plain Python over the C++ row statistics: one host thread
        threads, how = 1, "Python loop over requests on one thread"
    elif w.kind == "rejection_chain_sparse":
        how = "candidate lists scattered by numpy on one thread, then std::thread over requests"
    else:
        how = "std::thread over requests"
    return {"value": w.rows * reps / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "full batch (%d requests, %d rows) x %d repetitions, %s" % (w.batch, w.rows, reps, how),
            "seconds": round(el, 3)}


def step_parity(w, res: dict, threads: int) -> dict:
    """The timed step's outputs (the last replay) against the oracle on the same inputs, under the parity rule:
    exact token decisions except from a decision within 1e-6 of its threshold on."""
    from oracle import parity
    c = parity.compare(w, res, oracle_run(w, threads), check=False)
    return {"requests": c["requests"], "exact": c["exact"], "flagged": c["flagged"],
            "draw_flagged": c["draw_flagged"], "test_flagged": c["test_flagged"], "differ": c["differ"],
            "mismatch": c["mismatch"], "rule": "bit-exact decisions; a request is compared up to its first "
                                              "decision within 1e-6 of its threshold, and must be valid after it"}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------


def run_ours(args):
    import torch
    ranks = Ranks()
    torch.cuda.set_device(ranks.local)
    from reject_row_vocab_gb300 import _build
    if ranks.local == 0:
        _build.build()
    ranks.barrier()
    from reject_row_vocab_gb300 import device_workload as dw
    from reject_row_vocab_gb300 import specverify as sv

    w = make_workload(args, ranks.rank)
    d = dw.DeviceInputs.from_workload(w)
    out = dw.outputs_for(w)
    ws = dw.workspace_for(w)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup
    flush = flush_wanted(args, w)
    flush_buf = torch.empty(FLUSH_BYTES if flush else 0, dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones((FLUSH_BYTES if flush else 0) // 4, dtype=torch.float32, device="cuda")

    def flush_l2():
        # The write evicts the previous step's lines; the read then evicts the written (dirty) lines, so their
        # write-back happens here and not inside the next step.
        flush_buf.fill_(1)
        flush_rd.sum()

    def step():
        if flush:
            flush_l2()
        dw.run(w, d, out=out, ws=ws)

    for _ in range(max(W, 3)):
        step()
    torch.cuda.synchronize()

    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    G = max(1, min(args.graph_steps, K))
    E = max(1, args.stats_events_every)  # one launch in E gets events around its row-statistics kernel
    slots = stats_event_slots(min(K, 1024) if args.eager else G, E)
    P = sum(1 for x in slots if x is not None)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(P)]
    for a, b in pairs:  # create the events on the device
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()

    graph = None
    if not args.eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            dw.run(w, d, out=out, ws=ws)  # populate per-device caches outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for k in range(G):
                if flush:
                    flush_l2()
                sv.set_stats_events(*(pairs[slots[k]] if slots[k] is not None else (None, None)))
                dw.run(w, d, out=out, ws=ws)
            sv.set_stats_events(None, None)
        torch.cuda.synchronize()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()

    clocks = ClockSampler(gpu_id_for(ranks.local))
    clocks.start()
    ranks.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ev_start.record(stream)
    if graph is None:
        for k in range(K):
            if flush:
                flush_l2()
            j = slots[k % len(slots)]
            sv.set_stats_events(*(pairs[j] if j is not None else (None, None)))
            dw.run(w, d, out=out, ws=ws)
        sv.set_stats_events(None, None)
        launched = K
    else:
        reps = max(1, K // G)
        for _ in range(reps):
            graph.replay()
        launched = reps * G
    ev_end.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    t1 = time.time()
    clocks.mark(t0, t1)
    clk = clocks.stop()

    elapsed_s = ev_start.elapsed_time(ev_end) / 1e3
    if flush:  # the same number of flushes alone, launched the same way, comes off the span
        fgraph = None
        if graph is not None:
            fgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(fgraph, stream=cap):
                for _ in range(G):
                    flush_l2()
            torch.cuda.synchronize()
            fgraph.replay()
        torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        if fgraph is None:
            for _ in range(launched):
                flush_l2()
        else:
            for _ in range(launched // G):
                fgraph.replay()
        f1.record(stream)
        torch.cuda.synchronize()
        elapsed_s -= f0.elapsed_time(f1) / 1e3
    max_s = ranks.max(elapsed_s)
    avg_stats_ms = statistics.mean(a.elapsed_time(b) for a, b in pairs)  # last recording of each pair
    floor = event_context(d["logits"], flush_l2 if flush else None, None if graph is None else cap)

    res = out.to_numpy()
    committed = int(res["num_out"].sum())
    rows_total = ranks.sum(w.rows * launched)
    value = rows_total / max_s
    tokens = ranks.sum(committed * launched) / max_s
    peak, peak_src = measured_peaks()
    alg_bytes = w.logit_bytes()
    achieved = alg_bytes / (avg_stats_ms / 1e3) / 1e9

    # end to end through the public call with host buffers: H2D inputs, verify, D2H results
    e2e = None
    if args.e2e_steps > 0:
        host = dw.DeviceInputs.from_workload(w, pin=True)
        out_names = ("accept_len", "num_out", "out_tokens", "bonus", "commit_cu", "commit_src_slot",
                     "commit_dst_pos", "dev_status")
        h_out = {n: torch.empty_like(getattr(out, n), device="cpu").pin_memory() for n in out_names}
        d2h = sum(t.numel() * t.element_size() for t in h_out.values())
        h2d = host.nbytes()
        for _ in range(2):
            d.copy_from(host)
            dw.run(w, d, out=out, ws=ws)
        torch.cuda.synchronize()
        ranks.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            d.copy_from(host)
            dw.run(w, d, out=out, ws=ws)
            for n in out_names:
                h_out[n].copy_(getattr(out, n), non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e_s = ranks.max(e0.elapsed_time(e1) / 1e3)
        e2e = {"value": ranks.sum(w.rows * args.e2e_steps) / e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * e_s / args.e2e_steps,
               "note": "bound by the host link: every input (dense q included) crosses it each step, and pinned "
                       "host->device copies measured 211 GB/s on this GPU, by copy engine or by SM loads alike"}

    cpu = parity = None
    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, args.cpu_seconds, os.cpu_count() or 1)
        one = time_oracle(w, args.cpu_seconds / 3.0, 1)  # the same oracle on one host thread
        cpu["single_thread"] = {"value": one["value"], "cores": 1, "seconds": one["seconds"]}
        parity = step_parity(w, res, os.cpu_count() or 1)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ranks.world, "steps": launched,
        "warmup": max(W, 3), "ms_per_step": 1e3 * max_s / launched, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(describe(w, flush), launch="eager" if graph is None else "cuda graph of %d steps" % G,
                       parallelism="replicas x%d (independent batches)" % ranks.world),
        "committed_tokens_per_s": tokens, "mean_accept_len": float(res["accept_len"].mean()),
        "logit_gbs_per_step": alg_bytes * launched / elapsed_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": stats_traffic(w), "kernel": "k_row_stats",
                     "timed_span": "k_row_stats alone (events recorded around its launch, in %s)"
                                   % ("every launch" if E == 1 else "one launch in %d; the others run without "
                                                                        "event nodes" % E),
                     "bytes_per_launch": alg_bytes,
                     "avg_launch_us": avg_stats_ms * 1e3, "peak_source": peak_src,
                     "event_context": None if floor is None else dict(
                         floor, torch_sum_frac=alg_bytes / (floor["torch_sum_us"] * 1e-6) / 1e9 / peak)},
        "clocks": clk, "gpu_launches": KERNELS_PER_STEP[w.kind] * launched,
        "e2e": e2e, "cpu_baseline": cpu, "parity": parity,
        "inputs_sha256": w.sha256(),  # first 16 hex digits per input array (rank 0's batch)
    }
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)
    ranks.close()


# ---------------------------------------------------------------------------
# Reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = make_workload(args, 0)
    threads = os.cpu_count() or 1
    K, W = args.steps, max(args.warmup, 3)
    t0 = time.perf_counter()
    oracle_run(w, threads)
    per_batch = time.perf_counter() - t0
    # each step verifies the full batch when the budget allows, else a prefix of its requests
    budget = args.ref_budget_s / (K + W)
    n = w.batch if per_batch <= budget else max(1, int(w.batch * budget / per_batch))
    sub = subset(w, n)
    for _ in range(W):
        oracle_run(sub, threads)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle_run(sub, threads)
    el = time.perf_counter() - t0
    value = sub.rows * K / el
    sample = "%d of %d requests (%d rows) per step, %d steps, std::thread over requests" % (n, w.batch, sub.rows, K)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": 1e3 * el / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": dict(describe(w, flush_wanted(args, w)), parallelism="host cores"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "inputs_sha256": w.sha256(),
    }
    print(json.dumps(line), flush=True)


def subset(w, n: int):
    """The first n requests of a workload (slicing only)."""
    import copy
    if n >= w.batch:
        return w
    s = copy.copy(w)
    if w.nodes:
        rows = n * w.nodes
        s.tokens, s.parents = w.tokens[:n], w.parents[:n]
        if w.first_child is not None:
            s.first_child, s.next_sibling = w.first_child[:n], w.next_sibling[:n]
    else:
        rows = int(w.cu_seqlens[n])
        s.cu_seqlens = w.cu_seqlens[: n + 1]
        s.verify_ids = w.verify_ids[:rows]
    s.batch, s.rows = n, rows
    s.logits = w.logits[:rows]
    for k in ("q", "u_accept", "row_slots"):
        if getattr(w, k) is not None:
            setattr(s, k, getattr(w, k)[:rows])
    for k in ("temperature", "u_final", "seq_lens"):
        if getattr(w, k) is not None:
            setattr(s, k, getattr(w, k)[:n])
    return s


# ---------------------------------------------------------------------------
# Scheduler and tree-input builder (their own small kernels, timed the same way)
# ---------------------------------------------------------------------------

# One lane compares two 64-bit keys in three 32-bit integer instructions (two compares with carry, one
# predicated add): 152 SMs x 128 lanes x 2.07 GHz / 3.
ALU_COMPARE_PEAK = 152 * 128 * 2.07e9 / 3.0
AUX = {"dspark": {"metric": "verify-length schedules/s", "unit": "schedules/s", "launches": 2},
       "tree-build": {"metric": "tree batches built/s", "unit": "batches/s", "launches": 1}}


def aux_inputs(kind: str, rank: int = 0) -> dict:
    from reject_row_vocab_gb300 import workload as wl
    if kind == "dspark":
        return wl.dspark_schedule(requests=256, drafts=15, seed=1006 + 100 * rank)
    return wl.random_trees(batch=64, nodes=64, fan=8, seed=1007 + 100 * rank)


def aux_config(kind: str, x: dict) -> dict:
    if kind == "dspark":
        R, D = x["survival"].shape
        return {"workload": "dspark_schedule_r%d_d%d" % (R, D), "requests": R, "drafts": D,
                "l2": "inputs of %d KB, L2-resident (a scheduling step, not a streaming pass)" % (R * D * 4 // 1024)}
    B, N = x["parents"].shape
    return {"workload": "tree_build_b%d_n%d" % (B, N), "batch": B, "nodes": N,
            "l2": "inputs and outputs of %d KB, L2-resident" % ((B * N * (N + 28) + 8 * B) // 1024)}


def run_aux(args):
    import numpy as np
    import torch
    ranks = Ranks()
    torch.cuda.set_device(ranks.local)
    from reject_row_vocab_gb300 import _build
    if ranks.local == 0:
        _build.build()
    ranks.barrier()
    from reject_row_vocab_gb300 import specverify as sv
    kind, spec = args.kernel, AUX[args.kernel]
    x = aux_inputs(kind, ranks.rank)
    dev = torch.device("cuda", ranks.local)
    if kind == "dspark":
        R, D = x["survival"].shape
        k_star = sv.dspark_budget(x["hist"], R, x["sps"])
        surv = torch.from_numpy(x["survival"]).to(dev)
        out = torch.empty(R, dtype=torch.int32, device=dev)
        ws = sv.dspark_workspace(R, dev)

        def call():
            sv.dspark_verify_lens(surv, k_star, out=out, ws=ws)
        work = float(R * D) ** 2  # pairwise key comparisons per call
    else:
        B, N = x["parents"].shape
        par = torch.from_numpy(x["parents"]).to(dev)
        sl = torch.from_numpy(x["seq_lens"]).to(dev)
        res = sv.build_tree(par, sl)

        def call():
            sv.build_tree(par, sl, out=res)
        # bytes per call: parents and seq_lens read; mask, positions, index, links and status written
        work = float(B * N * 4 + B * 8 + B * N * N + B * N * (8 + 4 + 4 + 4) + B * 4)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup
    for _ in range(max(W, 3)):
        call()
    torch.cuda.synchronize()
    G = max(1, min(args.graph_steps, K))
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for _ in range(G):
            call()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_id_for(ranks.local))
    clocks.start()
    ranks.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    e0.record(stream)
    reps = max(1, K // G)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    clocks.mark(t0, time.time())
    clk = clocks.stop()
    launched = reps * G
    el = ranks.max(e0.elapsed_time(e1) / 1e3)
    per_call = el / launched
    if kind == "dspark":
        roof = {"bound": "alu", "achieved": work / per_call / 1e9, "peak": ALU_COMPARE_PEAK / 1e9,
                "unit": "Gcompare/s", "frac": work / per_call / ALU_COMPARE_PEAK, "traffic": None,
                "kernel": "k_dspark_rank + k_dspark_lens", "compares_per_launch": work,
                "timed_span": "whole calls inside a CUDA graph", "peak_source": "derived (lanes x clock / 3)"}
    else:
        peak, src = measured_peaks()
        roof = {"bound": "hbm", "achieved": work / per_call / 1e9, "peak": peak, "unit": "GB/s",
                "frac": work / per_call / 1e9 / peak, "traffic": None, "kernel": "k_build_tree",
                "bytes_per_launch": work, "timed_span": "whole calls inside a CUDA graph", "peak_source": src}
    line = {
        "metric": spec["metric"], "value": ranks.sum(launched) / el, "unit": spec["unit"], "n_gpus": ranks.world,
        "steps": launched, "warmup": max(W, 3), "ms_per_step": 1e3 * per_call, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if kind == "dspark" else "int32",
        "data": "synthetic", "config": dict(aux_config(kind, x), launch="cuda graph of %d calls" % G,
                                            parallelism="replicas x%d (independent inputs)" % ranks.world),
        "roofline": roof, "clocks": clk, "gpu_launches": spec["launches"] * launched, "e2e": None,
        "cpu_baseline": None,
    }
    if kind == "dspark":
        line["budget"] = k_star
        line["verify_lens_sum"] = int(out.sum().item())
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)
    ranks.close()


def run_aux_reference(args):
    """The scheduler or the tree builder of the fp64 oracle, on the host, same inputs and config."""
    import oracle.dspark as od
    import oracle.tree_build as ot
    if int(os.environ.get("RANK", "0")) != 0:
        return
    kind, spec = args.kernel, AUX[args.kernel]
    x = aux_inputs(kind)
    if kind == "dspark":
        surv = x["survival"].astype("float64").tolist()
        R = len(surv)
        k_star = od.budget(x["hist"].astype("float64").tolist(), R, x["sps"].astype("float64").tolist())

        def call():
            od.verify_lens(surv, k_star)
    else:
        par, sl = x["parents"].tolist(), x["seq_lens"].tolist()

        def call():
            for b in range(len(par)):
                ot.build(par[b], sl[b], b)
    for _ in range(3):  # three untimed calls whatever --warmup asks (at least three, and a bounded CPU cost)
        call()
    budget = args.ref_budget_s
    t0 = time.perf_counter()
    n = 0
    while n < args.steps and time.perf_counter() - t0 < budget:
        call()
        n += 1
    el = time.perf_counter() - t0
    value = n / el
    sample = "%d calls on one host thread (the oracle is single-threaded here)" % n
    line = {
        "impl": "reference", "metric": spec["metric"], "value": value, "unit": spec["unit"], "n_gpus": 1,
        "steps": n, "warmup": 3, "ms_per_step": 1e3 * el / n, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(aux_config(kind, x), parallelism="host cores"),
        "cpu_baseline": {"value": value, "unit": spec["unit"], "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": spec["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.kernel != "step":
        run_aux_reference(args) if args.impl == "reference" else run_aux(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
