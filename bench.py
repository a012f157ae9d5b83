"""Benchmark of the triggered all-gather on one GB300 (replicas on N GPUs under torchrun).

A step is one round of the whole hot path on the 4-rank chunked workload: plan_start launches
the round's copier, the hashed-fill producer writes every rank's 32 MiB slice in 512-row
chunks and marks each one, the copier fans each ready chunk out to the three peers and signals
arrival, and plan_wait runs the completion check and returns to the host; next_round ends the
step.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

--impl reference times the CPU oracle (the plain restatement of the method in oracle/) on the
host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "delivered all-gather GB/s and % of HBM peak (1 GB300); gate-to-arrival latency"
DEFAULT_CONFIG = W.C2.name

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the named kernel from one ncu capture
# of the same workload and launch configuration (the summaries under profiles/); absent until
# taken, and dropped once the kernel changes.
NCU_TRAFFIC = {("c2_chunks_p4", "copier_bulk_kernel"): 474700544,
               # captured with 2000 rows per rank (--rows 2000) and scaled by the rows, 4x
               ("c3_tiles_p8", "copier_bulk_kernel"): 8009544192,
               ("c5_gemm_p4", "gemm2_producer_kernel"): 184814208,
               ("c5_gemm_p4", "copier_kernel"): 206209536,
               ("c4a_writers8_p8", "copier_bulk_kernel"): 205637888,
               # captured with 256 rows (--rows 256) and scaled by the rows, 10x
               ("c4b_bcast_p8", "copier_bulk_kernel"): 20848015360,
               # the two-shot all-reduce's reduce kernel (bench.py --allreduce --in-order), 256 threads
               ("allreduce_p4", "reduce_kernel"): 652057088}
# DRAM bytes (read, write) of one whole round, producer, copier and check together, from an
# ncu range-replay capture of three rounds of the benchmark's launch (--profile-rounds 3;
# c2 and c5 with overlapping rounds)
ROUND_TRAFFIC = {"c2_chunks_p4": (799317, 515392085), "c3_tiles_p8": (16352085, 8237216427),
                 "c5_gemm_p4": (272514048, 252129451)}


def describe(w, launch, copier=None) -> str:
    if w.kind == "chunks":
        sched = f"chunks() {w.num_chunks} x {w.M // w.num_chunks} rows, 1 writer each"
    elif w.kind == "whole":
        sched = f"whole() with {w.num_programs} writers"
    else:
        sched = (f"tile_chunks {w.BM}x{w.BN}, {w.num_programs} programs, "
                 f"{w.tiles_per_chunk} tiles per chunk, GROUP_M={w.group_m}")
    cl, grp = launch.get("cluster", 1), launch.get("group", 1)
    prod = ""
    if cl > 1:
        prod = f"; producer: {launch.get('programs') or 'one per chunk'} program(s) per rank of {cl}-CTA clusters"
    elif grp > 1:
        prod = (f"; producer: {launch.get('programs') or 'one per chunk'} program(s) per rank, each a "
                f"group of {grp} CTAs marking each chunk once")
    if launch.get("pace"):
        prod += (f"; producer paced: a program writes chunk k once chunk k-{launch['pace']} of its "
                 f"rank is delivered")
        if copier is not None and copier.get("overlap"):
            prod += " (the previous round's chunk n-%d+k for k < %d)" % (launch["pace"], launch["pace"])
    cop = ""
    if copier is not None:
        cop = ("; copier: bulk copies, %d CTA(s) per SM with %d x %d KiB stages each"
               % (copier["ctas_per_sm"], copier["stages"], copier["piece_bytes"] >> 10)
               if copier["method"] == 1 else
               "; copier: 16-byte vector copies, %d threads x %d CTA(s) per SM"
               % (copier["copier_threads"], copier["ctas_per_sm"]))
    kind = "broadcast from rank 0" if w.broadcast else "in-place all-gather"
    return (f"{w.name}: {kind}, P={w.P} virtual ranks, {w.dtype} [{w.buf_rows}, {w.N}] per "
            f"buffer, {sched}{prod}{cop}")


def l2_note(w, dev) -> str:
    """Whether the round's buffers exceed L2 (read from the device), as the timing rule asks."""
    import torch
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20)
    total = w.P * w.buf_bytes
    if total > l2:
        return "inputs larger than L2 (%d MiB of buffers, L2 %d MiB)" % (total >> 20, l2 >> 20)
    return ("inputs smaller than L2 (%d KiB of buffers, L2 %d MiB): an L2-resident, latency-bound "
            "workload; every round rewrites them, no flush" % (total >> 10, l2 >> 20))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_tensor_peak():
    """Dense bf16 tensor peak: the measured burst figure (a kernel timed on its own)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured burst"
    except Exception:
        return 1900.0, "fallback"


def load_tensor_peak_sustained():
    """Dense bf16 tensor peak under the power cap (a seconds-long matmul loop), or None."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return None


# ---- clocks ------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()
        return False

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


# ---- CPU oracle timing ---------------------------------------------------------------------------
def oracle_sample_workload(w):
    """A bounded sample of workload w for the CPU oracle: same P, row length, dtype and
    schedule kind, fewer rows (one chunk's worth per rank for the chunked workload)."""
    if w.kind == "chunks":
        rows = max(1, min(128, w.M // w.num_chunks))
        return W.small(w, M=rows, num_chunks=1), f"{rows} of {w.M} rows per rank, one chunk"
    if w.kind == "tile_chunks":
        rows = min(w.M, 2 * w.BM)
        return W.small(w, M=rows), f"{rows} of {w.M} rows per rank"
    rows = max(1, min(w.M, 256, (8 << 20) // w.row_bytes))      # at most 8 MiB per slice
    return W.small(w, M=rows, num_programs=min(w.num_programs, rows)), f"{rows} of {w.M} rows"


def time_oracle(w, budget_s: float = 10.0, max_rounds: int = 1000):
    """Run the oracle's sequential rounds on a sample of w until budget_s; GB/s delivered."""
    from oracle.run import make_plan as oracle_plan, run_round as oracle_round
    sw, what = oracle_sample_workload(w)
    o = oracle_plan(sw)
    n, t0 = 0, time.perf_counter()
    while n < max_rounds:
        status = oracle_round(o, sw)
        assert status[0] == "OK"
        o.next_round()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return sw.delivered_bytes_per_round() * n / dt / 1e9, n, dt, what


def time_oracle_threaded(w, budget_s: float = 10.0, max_rounds: int = 1000):
    """The threaded oracle (one producer thread per rank, one copier thread per (source, peer)
    queue, gate words under a lock) on the same sample as time_oracle; GB/s delivered and the
    thread count."""
    from oracle import hashfill as H
    from oracle.run import make_plan as oracle_plan
    from oracle.threaded import ThreadedRound
    sw, what = oracle_sample_workload(w)
    if w.kind == "tile_chunks":     # one tile row per rank: a round of many small regions
        sw, what = W.small(w, M=min(w.M, w.BM)), f"{min(w.M, w.BM)} of {w.M} rows per rank"
    o = oracle_plan(sw)
    n, t0 = 0, time.perf_counter()
    while n < max_rounds:
        data = {}

        def write_unit(rank, c, u, o=o, data=data):
            if rank not in data:        # the rank's slice for this round, computed by its thread
                data[rank] = H.fill_slice_bytes(sw.dtype, sw.seed, rank, o.round, sw.M, sw.N)
            base = sw.slice_offset(rank)
            regs = o.chunks[c].regions
            # one region per writer (tiles): writer u stores tile u; otherwise writer 0 stores
            # the chunk and the others only mark
            mine = [regs[u]] if len(regs) == o.chunks[c].writers else (regs if u == 0 else [])
            for (off, nb, rows, pitch) in mine:
                for i in range(rows):
                    a = off + i * pitch
                    o.bufs[rank][a:a + nb] = data[rank][a - base:a - base + nb]

        order = {r: [(c, u) for c in o.chunks_of(r) for u in range(o.chunks[c].writers)]
                 for r in sw.senders()}
        status = ThreadedRound(o, write_unit, order, max_polls=10 ** 6, poll_sleep=1e-5).run()
        assert status[0] == "OK", status
        o.next_round()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    threads = len(sw.senders()) * (sw.P - 1) + len(sw.senders())
    return sw.delivered_bytes_per_round() * n / dt / 1e9, n, dt, what, threads


def time_oracle_gemm(w, budget_s: float = 10.0, rows: int = 128):
    """The oracle on a sample of the GEMM workload: C_r for `rows` rows of every rank (fp64
    product of the bf16 operands, numpy's multithreaded BLAS), rounded to bf16 and copied to
    the P-1 peers.  GB/s delivered."""
    from oracle import gemm as OG
    from oracle import hashfill as H
    A, Bt = W.gemm_inputs(w.P, rows, w.N, w.K, w.seed)
    Bt64 = Bt.double().numpy()
    A64 = [A[r].double().numpy() for r in range(w.P)]
    peers = [np.zeros((w.P, rows, w.N), dtype=np.uint16) for _ in range(w.P)]
    n, t0 = 0, time.perf_counter()
    while True:
        for r in range(w.P):
            c = H.f32_to_bf16_bits(OG.product(A64[r], Bt64).astype(np.float32))
            for q in range(w.P):
                peers[q][r] = c
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return (w.P * rows * w.N * 2 * (w.P - 1) * n / dt / 1e9, n, dt,
            f"{rows} of {w.M} rows of C per rank")


# ---- distributed helpers ---------------------------------------------------------------------------
def time_oracle_allreduce(budget_s: float = 10.0, rows: int = 32):
    """The oracle's two-shot all-reduce (both plans and the reduce step on the plan model) on a
    sample of the benchmark's workload: P = 4 ranks of `rows` rows of 4096 bf16 per block, in
    the benchmark's sub-blocks.  Returns (GB/s of vector bytes per rank, rounds, seconds, sample)."""
    from oracle import allreduce as OA
    a = W.ALLREDUCE
    P, cols, J = a["P"], a["cols"], a["sub_blocks"]
    o = OA.TwoShot(P, rows, cols, a["dtype"], J)
    M = P * rows
    parts = [OA.hashed_partials(a["dtype"], a["seed"], P, M, cols, R) for R in (1, 2)]
    n, t0 = 0, time.perf_counter()
    while True:
        o.round(parts[n % 2])
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or n >= 1000:
            break
    S = M * cols * 2
    return S * n / dt / 1e9, n, dt, f"{rows} of {a['block_rows']} rows per block, P={P}, {J} sub-blocks"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def aggregate(elapsed_s: float, units: float, world: int):
    """Whole-job figures: max elapsed over ranks, units summed over ranks."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- the two arms ------------------------------------------------------------------------------------
def workload(args):
    """The workload named by --config, with --rows rows per rank when given."""
    w = W.CONFIGS[args.config]
    return W.small(w, M=args.rows, name=f"{w.name}_rows{args.rows}") if args.rows else w


def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    w = workload(args)
    sw, what = oracle_sample_workload(w)
    from oracle.run import make_plan as oracle_plan, run_round as oracle_round
    o = oracle_plan(sw)
    for _ in range(args.warmup):
        oracle_round(o, sw)
        o.next_round()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        assert oracle_round(o, sw)[0] == "OK"
        o.next_round()
    dt = time.perf_counter() - t0
    value = sw.delivered_bytes_per_round() * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": describe(w, {}), "sample": what},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": what},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def measure_workload(w, args, K, warmup, latency_rounds, isolated_rounds, with_e2e, world=1,
                     clocks_dev=None, early_us=None, method=None, overlap=None, pace=None):
    """Time K rounds of workload w in the launch the benchmark uses for it (runner.bench_launch),
    then the kernel-timing pass, the gate timestamps, the isolated kernels and (optionally) the
    host-buffer round.  overlap (None: the launch's choice): rounds two at a time (opts.overlap):
    each step starts its round, launches the producer, waits for the round before it and leaves
    its own round pending; the timed region ends with the wait for the last round.  pace: the
    fill producer's pacing (None: the launch's own).  Returns a dict of raw measurements
    (seconds, milliseconds, bytes)."""
    import torch
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner

    launch = dict(runner.bench_launch(w, overlap))
    # the copier runs on a stream the bench can put events on
    copy_stream = torch.cuda.Stream(priority=-1)
    # the headline pass records no per-launch events (a timed event between two launches on a
    # stream costs the round a few microseconds); the kernel-timing pass after it runs the same
    # launches on a plan that times each copier launch itself (CUDA events in the library)
    opts = launch.pop("opts", None) or D.dtt_plan_opts_default()
    if method is not None and method != opts.method:
        # another transport under the same producer: the copy engines need no copier kernel
        # (nothing to launch early, nothing to pace against)
        opts = D.dtt_plan_opts_default(method=method)
        launch.pop("pace", None)
    if args.deferred:
        opts.deferred_copier = 1
        opts.overlap = 0      # a round's producer would wait for a copier that runs after it
    if early_us is not None:
        opts.early_copier_us = early_us
    if getattr(args, "copier", None):            # launch overrides
        opts.method = {"vector": D.COPY_VEC16, "bulk": D.COPY_TMA}[args.copier]
    for k in ("piece_bytes", "stages", "ctas_per_sm", "copier_threads", "copier_ctas", "host_piece_bytes"):
        v = getattr(args, k, 0)
        if v:
            setattr(opts, k, v)
    overlap = bool(opts.overlap)
    if pace is not None and w.K == 0:
        launch["pace"] = pace
    opts.time_copier = 0
    copier_method = {"method": opts.method, "piece_bytes": opts.piece_bytes, "stages": opts.stages,
                     "copier_threads": opts.copier_threads, "ctas_per_sm": opts.ctas_per_sm,
                     "copier_ctas": opts.copier_ctas, "overlap": opts.overlap}
    gemm = w.K > 0
    if gemm:           # the GEMM producer: C_r = A_r . B, marking each tile's chunk
        A, Bt = W.gemm_inputs(w.P, w.M, w.N, w.K, w.seed)
        st = runner.make_gemm(w, A, Bt, opts=opts, copy_stream=copy_stream)
        w_sched = st.w

        def produce(h, deferred=False):
            D.dtt_gemm_producer(st.A, st.Bt, st.buf_ptrs, w.M, w.N, w.K, w.row_bytes, st.slice_offs,
                                st.num_programs, h, st.err, prod)
    else:
        st = runner.make(w, opts=opts, copy_stream=copy_stream, **launch)
        w_sched = w

        # a paced producer waits for the copier, so a plan whose copier starts only after the
        # producer gets the same producer without pacing
        desc_unpaced = type(st.desc).from_buffer_copy(st.desc)
        desc_unpaced.pace = 0

        def produce(h, deferred=False):
            D.dtt_fill_producer(st.buf_ptrs, desc_unpaced if deferred else st.desc, h, prod)
    prod = st.producer_stream

    def make_step(plan, deferred, overlapped=False, after_producer=False):
        """One round.  ev: two events around the producer launch (producer stream), or None.
        deferred: the plan's copier starts only after the producer.  overlapped: the round is
        left pending (its wait comes in the next step, or in drain).  after_producer: the
        plan's copier is launched right after the producer's launch (deferred_copier = 2)."""
        def step(ev=None):
            h = plan.start(prod)
            if ev is not None:
                ev[0].record(prod)
            produce(h, deferred)
            if ev is not None:
                ev[1].record(prod)
            if after_producer:
                plan.launch_copier()
            if overlapped:
                if plan.pending:
                    plan.wait()
                plan.next_round()
                return
            if deferred:      # the copier starts once the producer has finished
                plan.launch_copier()
            plan.wait()
            plan.next_round()
        return step

    def drain(plan):
        """Wait for a round still pending (overlapped steps)."""
        if plan.pending:
            plan.wait()

    def timed(plan, step, K, producer_events):
        """K steps between two events on the producer stream; returns (seconds, copier ms per
        launch from the plan's own events, producer ms per launch or None)."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)] \
            if producer_events else [None] * K
        c0 = plan.stats()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(prod)
        for i in range(K):
            step(evs[i])
        drain(plan)
        e1.record(prod)
        e1.synchronize()
        torch.cuda.synchronize()
        c1 = plan.stats()
        cop = (c1[1] - c0[1]) / max(1, c1[2] - c0[2])
        prod_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) if producer_events else None
        return e0.elapsed_time(e1) / 1e3, cop, prod_ms

    step = make_step(st.plan, opts.deferred_copier == 1, overlap, opts.deferred_copier == 2)
    for _ in range(warmup):
        step()
    drain(st.plan)
    torch.cuda.synchronize()
    out = {"w": w, "launch": launch, "copier_method": copier_method, "gemm": gemm,
           "deferred_copier": opts.deferred_copier, "early_copier_us": opts.early_copier_us,
           "overlap": overlap}
    if args.profile_rounds:
        # whole rounds (producer, copier and check together) inside one profiler range, for a
        # range-replay capture of their DRAM traffic; no timing
        torch.cuda.profiler.start()
        for _ in range(args.profile_rounds):
            step()
        drain(st.plan)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        st.plan.close()
        out["profiled"] = True
        return out
    barrier(world)
    torch.cuda.synchronize()
    e_before = st.plan.early_stats()
    if clocks_dev is not None:
        with ClockSampler(clocks_dev) as clocks:
            time.sleep(0.25)
            elapsed, _, _ = timed(st.plan, step, K, producer_events=False)
            time.sleep(0.25)
        out["clocks"] = clocks.summary()
    else:
        elapsed, _, _ = timed(st.plan, step, K, producer_events=False)
    e_after = st.plan.early_stats()
    out["early"] = {k: e_after[k] - e_before[k] for k in e_after}
    barrier(world)
    out["elapsed_s"] = elapsed

    def side_plan(**over):
        """A second plan over the same buffers with the same copier launch."""
        o = D.dtt_plan_opts_default(allgather=0 if w.broadcast else 1, **copier_method)
        for k, v in over.items():
            setattr(o, k, v)
        scheds = runner.schedules_for(w_sched)
        plan = D.Plan(st.bufs, w.buf_bytes, scheds, o, copy_stream=copy_stream)
        for sc in scheds:
            sc.free()
        return plan

    # kernel-timing pass: K more rounds of the same step, CUDA events around every copier launch
    # (in the library, on the copy stream) and, for the GEMM, around every producer launch.  A
    # timed plan launches its copier at plan_start, so each copier launch is one round's.
    if opts.method == D.COPY_ENGINE:      # no copier kernel: the round is the transport's time
        out.update(timing_pass_s=elapsed, copier_ms=elapsed / K * 1e3, producer_ms=None)
    else:
        plan3 = side_plan(time_copier=1, deferred_copier=opts.deferred_copier, overlap=opts.overlap)
        step3 = make_step(plan3, opts.deferred_copier == 1, overlap, opts.deferred_copier == 2)
        for _ in range(3):
            step3()
        drain(plan3)
        torch.cuda.synchronize()
        t3, copier_ms, producer_ms = timed(plan3, step3, K, producer_events=gemm)
        plan3.close()
        out.update(timing_pass_s=t3, copier_ms=copier_ms, producer_ms=producer_ms)

    # gate-to-arrival latency and the copier window, from the gate timestamps of extra rounds
    lat, windows, queue, xfer = [], [], [], []
    _, _, n_chunks_all, _ = st.plan.info()
    out["n_chunks_total"] = sum(n_chunks_all[r] for r in w.senders())
    for _ in range(latency_rounds):
        step()
        if overlap:           # a round whose producer ran beside the previous round's copier
            step()
            drain(st.plan)
        g = st.plan.read_gates()
        n_global, first, n_chunks, _ = st.plan.info()
        t_open_min, t_arr_max = None, 0
        for r in range(w.P):
            for c in range(first[r], first[r] + n_chunks[r]):
                to = int(g[r, c, D.GATE_T_OPEN])
                t_open_min = to if t_open_min is None else min(t_open_min, to)
                tc = int(g[r, c, D.GATE_T_ARRIVE])     # owner's row: when the copier began the chunk
                if tc >= to > 0:
                    queue.append(tc - to)
                for p in range(w.P):
                    if p != r:
                        ta = int(g[p, c, D.GATE_T_ARRIVE])
                        lat.append(ta - to)
                        t_arr_max = max(t_arr_max, ta)
                        if tc >= to > 0:
                            xfer.append(ta - tc)
        windows.append((t_arr_max - t_open_min) / 1e9)
    out.update(lat=lat, windows=windows, queue=queue, xfer=xfer)

    # e2e: the host-buffer round through the public API: H2D of every rank's slice from pinned
    # memory, the triggered fan-out, D2H of rank 0's gathered buffer
    out["e2e"] = None
    if with_e2e and not w.broadcast and not gemm:
        S = w.slice_bytes
        host_in = [torch.empty(S, dtype=torch.uint8).pin_memory() for _ in range(w.P)]
        for r in range(w.P):
            host_in[r].copy_(st.bufs[r][w.slice_offset(r):w.slice_offset(r) + S].cpu())
        host_out = torch.empty(w.buf_bytes, dtype=torch.uint8).pin_memory()
        e2e_steps = max(1, min(K, 20))
        if overlap:
            # rounds back to back in one call, pipelined: a round's slices go in while the round
            # before comes back (each round's copies in and back are all inside the timed region)
            def run_e2e(n):
                st.plan.allgather_host_rounds([host_in] * n, [host_out] * n, 0, prod)
        else:
            def run_e2e(n):
                for _ in range(n):
                    st.plan.allgather_host(host_in, host_out, 0, prod)
        run_e2e(2)
        torch.cuda.synchronize()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(prod)
        run_e2e(e2e_steps)
        x1.record(prod)
        torch.cuda.synchronize()
        out["e2e"] = {"elapsed_s": x0.elapsed_time(x1) / 1e3, "steps": e2e_steps,
                      "h2d_bytes_per_step": S * w.P, "d2h_bytes_per_step": w.buf_bytes,
                      "call": "dtt_allgather_host_rounds" if overlap else "dtt_allgather_host"}
    st.plan.close()

    # the same copier and producer one after the other (deferred plan): each kernel alone
    out["isolated"] = None
    if not args.deferred and isolated_rounds and opts.method != D.COPY_ENGINE:
        plan2 = side_plan(time_copier=1, deferred_copier=1, overlap=0)
        step2 = make_step(plan2, True)
        for _ in range(3):
            step2()
        _, c2, f2 = timed(plan2, step2, isolated_rounds, producer_events=True)
        plan2.close()
        out["isolated"] = {"copier_ms": c2, "producer_ms": f2}
    out["num_programs"] = getattr(st, "num_programs", None)
    del st
    torch.cuda.empty_cache()
    return out


def summarize(m, K, t_max, units, peak, peak_kind):
    """The JSON fields of one measured workload (see measure_workload)."""
    import device_triggered_transfers_gb300 as D
    w = m["w"]
    D_round = w.delivered_bytes_per_round()
    B_alg = w.algorithmic_bytes_per_round()
    copier_method = m["copier_method"]
    cop_s = m["copier_ms"] / 1e3
    achieved = B_alg / cop_s / 1e9
    kname = "copier_bulk_kernel" if copier_method["method"] == D.COPY_TMA else "copier_kernel"
    copier_roof = {"kernel": kname, "bound": "hbm", "achieved": achieved,
                   "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                   "traffic": NCU_TRAFFIC.get((w.name, kname)), "algorithmic_bytes_per_launch": B_alg,
                   "round_dram_read_write": ROUND_TRAFFIC.get(w.name)}
    if m["gemm"]:       # the dominant kernel is the tensor-core producer
        flops = 2.0 * w.P * w.M * w.N * w.K
        tf_peak, tf_kind = load_tensor_peak()
        prod_s = m["producer_ms"] / 1e3
        NP = m["num_programs"] or w.num_programs
        gname = "gemm2_producer_kernel" if (w.M % 256 == 0 and w.N % 256 == 0 and NP >= 2) \
            else "gemm_producer_kernel"
        sustained = load_tensor_peak_sustained()
        roofline = {"kernel": gname, "bound": "tensor",
                    "achieved": flops / prod_s / 1e12, "peak": tf_peak, "peak_kind": tf_kind,
                    "unit": "TFLOP/s", "frac": flops / prod_s / 1e12 / tf_peak,
                    "frac_of_sustained": (flops / prod_s / 1e12 / sustained) if sustained else None,
                    "traffic": NCU_TRAFFIC.get((w.name, gname)),
                    "flops_per_launch": flops}
    else:
        roofline = copier_roof
    def med_p99(xs):
        xs = sorted(xs) or [0]
        return xs[len(xs) // 2], xs[min(len(xs) - 1, int(len(xs) * 0.99))]
    lat_med, lat_p99 = med_p99(m["lat"])
    q_med, q_p99 = med_p99(m.get("queue") or [])
    x_med, x_p99 = med_p99(m.get("xfer") or [])
    # the ideal time of one chunk's fan-out at the measured copy peak: one read of the chunk and
    # P-1 writes of it, (S_c + (P-1) S_c) / peak
    chunk_mean = len(w.senders()) * w.slice_bytes / max(1, m["n_chunks_total"])
    ideal_ns = w.P * chunk_mean / (peak * 1e9) * 1e9
    iso = None
    if m["isolated"]:
        c2, f2 = m["isolated"]["copier_ms"], m["isolated"]["producer_ms"]
        iso = {"copier_ms": c2, "producer_ms": f2,
               "copier_gbs_algorithmic": B_alg / (c2 / 1e3) / 1e9,
               "copier_frac_of_measured": B_alg / (c2 / 1e3) / 1e9 / peak,
               "overlap_ratio": (t_max / K) / (max(c2, f2) / 1e3)}
    windows = m["windows"]
    e2e = None
    if m["e2e"]:
        e2e = {"value": D_round * m["e2e"]["steps"] / m["e2e"]["elapsed_s"] / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": m["e2e"]["h2d_bytes_per_step"],
               "d2h_bytes_per_step": m["e2e"]["d2h_bytes_per_step"], "call": m["e2e"]["call"]}
    return {
        "ms_per_round": t_max / K * 1e3,
        "gbs_delivered": units / t_max / 1e9,
        "hbm_frac_end_to_end": {"of_measured": B_alg * units / D_round / t_max / 1e9 / peak,
                                "of_spec_8000": B_alg * units / D_round / t_max / 1e9 / 8000.0},
        "roofline": roofline,
        "copier_roofline": copier_roof if m["gemm"] else None,
        "kernels_ms": {"copier_mean": m["copier_ms"], "producer_mean": m["producer_ms"],
                       "timing_pass_ms_per_step": m["timing_pass_s"] / K * 1e3},
        "isolated": iso,
        "copier_window": ({"gbs_delivered": D_round / statistics.median(windows) / 1e9,
                           "hbm_frac": B_alg / statistics.median(windows) / 1e9 / peak}
                          if windows else None),
        "gate_to_arrival_ns": {"median": lat_med, "p99": lat_p99, "samples": len(m["lat"]),
                               "chunk_bytes_mean": chunk_mean,
                               "ideal_chunk_ns": ideal_ns,
                               "median_over_ideal": lat_med / ideal_ns if ideal_ns else None,
                               "p99_over_ideal": lat_p99 / ideal_ns if ideal_ns else None,
                               # the same split in two: the chunk's wait in its queue (gate open to
                               # the copier beginning it) and its transfer (to each arrival)
                               "queue_median": q_med if m.get("queue") else None,
                               "queue_p99": q_p99 if m.get("queue") else None,
                               "transfer_median": x_med if m.get("xfer") else None,
                               "transfer_p99": x_p99 if m.get("xfer") else None},
        "early_copier": {"wait_us": m["early_copier_us"], **(m.get("early") or {})},
        "e2e": e2e,
    }


# workloads measured beside the headline in the default run, with the steps each is timed over
PER_CONFIG_STEPS = {"c1_whole_p2": 200, "c3_tiles_p8": 30, "c4a_writers8_p8": 100,
                    "c4b_bcast_p8": 5, "c5_gemm_p4": 50}


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.cuda.current_device()
    import device_triggered_transfers_gb300 as D  # noqa: F401

    w = workload(args)
    K = args.steps
    early = None if args.early_us < 0 else args.early_us
    pace = None if args.pace < 0 else args.pace
    m = measure_workload(w, args, K, args.warmup, args.latency_rounds, args.isolated_rounds,
                         with_e2e=not args.no_e2e, world=world, clocks_dev=dev, early_us=early,
                         overlap=args.overlap, pace=pace)
    if m.get("profiled"):
        if rank == 0:
            print(json.dumps({"profile_rounds": args.profile_rounds, "workload": w.name,
                              "algorithmic_bytes_per_round": w.algorithmic_bytes_per_round(),
                              "producer_bytes_per_round": len(w.senders()) * w.slice_bytes}))
        return 0
    D_round = w.delivered_bytes_per_round()
    t_max, units = aggregate(m["elapsed_s"], D_round * K, world)
    if m["e2e"]:
        e_t, e_units = aggregate(m["e2e"]["elapsed_s"], D_round * m["e2e"]["steps"], world)
        m["e2e"]["elapsed_s"], m["e2e"]["steps"] = e_t, e_units / D_round
    value = units / t_max / 1e9
    peak, peak_kind = load_peaks()
    s = summarize(m, K, t_max, units, peak, peak_kind)

    # the other workloads, each timed the same way over fewer steps (single GPU only)
    per_config = None
    if world == 1 and args.per_config and not args.rows:
        per_config = {}
        for name, steps in PER_CONFIG_STEPS.items():
            if name == w.name:
                continue
            wc = W.CONFIGS[name]
            mc = measure_workload(wc, args, steps, 3, 5, 5, with_e2e=False, early_us=early,
                                  overlap=args.overlap)
            Dc = wc.delivered_bytes_per_round()
            sc = summarize(mc, steps, mc["elapsed_s"], Dc * steps, peak, peak_kind)
            per_config[name] = {
                "steps": steps, "ms_per_round": sc["ms_per_round"], "gbs_delivered": sc["gbs_delivered"],
                "dominant_kernel": {k: sc["roofline"][k] for k in ("kernel", "bound", "achieved", "unit", "frac",
                                                                   "traffic")},
                "copier_frac_in_round": (sc["copier_roofline"] or sc["roofline"])["frac"],
                "hbm_frac_end_to_end": sc["hbm_frac_end_to_end"]["of_measured"],
                "copier_window_hbm_frac": (sc["copier_window"] or {}).get("hbm_frac"),
                "isolated": sc["isolated"],
                "gate_to_arrival_ns": {k: sc["gate_to_arrival_ns"][k] for k in
                                       ("median", "p99", "median_over_ideal", "p99_over_ideal",
                                        "queue_median", "transfer_median", "transfer_p99")},
                "early_copier": sc["early_copier"],
                "workload": describe(wc, mc["launch"], mc["copier_method"]),
                "l2": l2_note(wc, dev)}

        # the two-shot all-reduce, built from a reduce-scatter plan and an all-gather plan
        ma = measure_allreduce(20, 3, isolated_rounds=5, fill_rounds=5)
        sa = summarize_allreduce(ma, peak, peak_kind)
        per_config[W.ALLREDUCE["name"]] = {
            "steps": 20, "ms_per_round": sa["ms_per_round"], "algbw_gbs": sa["algbw_gbs"],
            "busbw_gbs": sa["busbw_gbs"], "hbm_frac_end_to_end": sa["hbm_frac_end_to_end"]["of_measured"],
            "with_fill_producer_ms_per_round": ma.get("fill_round_ms"),
            "dominant_kernel": {k: (sa.get("reduce_roofline") or {}).get(k)
                                for k in ("kernel", "bound", "achieved", "unit", "frac", "traffic")},
            "workload": (f"P={W.ALLREDUCE['P']} bf16 [{W.ALLREDUCE['P'] * W.ALLREDUCE['block_rows']}, "
                         f"{W.ALLREDUCE['cols']}] per rank, {W.ALLREDUCE['sub_blocks']} sub-blocks of "
                         f"{W.ALLREDUCE['block_rows'] // W.ALLREDUCE['sub_blocks']} rows per block "
                         "(bench.py --allreduce)")}

    if rank != 0:
        return 0
    gemm = m["gemm"]
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        if gemm:
            v, n, dt, what = time_oracle_gemm(w, budget_s=args.cpu_seconds)
            cores = os.cpu_count()
        else:
            v, n, dt, what = time_oracle(w, budget_s=args.cpu_seconds)
            cores = 1
        cpu = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{what}; {n} oracle round(s) in {dt:.1f} s"}
        if not gemm:    # the same sample with threads as ranks and copier queues
            vt, nt, dtt, what_t, threads = time_oracle_threaded(w, budget_s=args.cpu_seconds / 2)
            cpu["threaded"] = {"value": vt, "threads": threads, "host_cores": os.cpu_count(),
                               "sample": f"{what_t}; {nt} threaded oracle round(s) in {dtt:.1f} s"}
    mode = {0: "copier launched at plan_start, overlapping the producer",
            1: "copier launched after the producer (no overlap)",
            2: "copier launched right after the producer's launch, overlapping it"}[m["deferred_copier"]]
    if m["early_copier_us"] and m["deferred_copier"] != 1:
        mode += ("; each round's copier launched early, by the previous round's plan_wait, and "
                 "claimed by plan_start (waits up to %d us for it)" % m["early_copier_us"])
    if m["overlap"]:
        mode += ("; overlapping rounds: a round's producer runs while the previous round's copier "
                 "still copies (each chunk written once its previous copies landed), its copier "
                 "queued behind the previous one")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_max / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": describe(w, m["launch"], m["copier_method"]), "parallelism": f"replicas{world}",
                   "l2": l2_note(w, dev),
                   "step": (("plan_start + %s producer + copier + plan_wait of the previous round + "
                             "next_round (this round left pending); the timed region ends with the "
                             "last round's plan_wait" if m["overlap"] else
                             "plan_start + %s producer + copier + plan_wait + next_round")
                            % ("GEMM" if gemm else "fill")),
                   "mode": mode},
        "hbm_frac_end_to_end": s["hbm_frac_end_to_end"],
        "roofline": s["roofline"],
        "copier_roofline": s["copier_roofline"],
        "kernels_ms": s["kernels_ms"],
        "isolated": s["isolated"],
        "copier_window": s["copier_window"],
        "gate_to_arrival_ns": s["gate_to_arrival_ns"],
        "early_copier": s["early_copier"],
        "e2e": s["e2e"],
        "gpu_launches": 3 * K,
        "clocks": m.get("clocks"),
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    print(json.dumps(line))
    return 0


def run_consumer(args):
    """The consumer side of the plan: a GEMM over rank 0's gathered buffer, D = X . W^T with
    X [P*M, N] (the all-gather's output) and W^T [consumer_n, N], each 128-row block loaded as
    soon as its chunks have arrived.  Times the all-gather round alone, the GEMM alone (its
    chunks already delivered), and the two overlapped in one round; the copier is the bulk-copy
    one with a ring small enough to leave the GEMM room, or the vector one.  Both wait forms are
    timed: one wait per chunk of a block, and one wait per block on a chunk group."""
    import torch
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner
    w = workload(args)
    K, N2 = w.N, args.consumer_n
    rows = w.buf_bytes // (2 * K)
    g = torch.Generator().manual_seed(w.seed + 99)
    Wt = (torch.randn(N2, K, generator=g) / K ** 0.5).to(torch.bfloat16).cuda()
    out = torch.empty(rows, N2, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy_stream, cons = torch.cuda.Stream(priority=-1), torch.cuda.Stream()
    # the producer of the benchmark's launch (its chunks open one wave after another), with the
    # vector copier
    launch = {k: v for k, v in runner.bench_launch(w, overlap=False).items() if k != "opts"}
    if args.consumer_copier == "bulk":    # one CTA per SM with a ring small enough for the GEMM's
        copier_desc = "bulk copies, one CTA per SM, 2 x 32 KiB stages"
    else:
        copier_desc = f"vector (16-byte) path, {args.consumer_copier_threads} threads per CTA"

    def copts():
        if args.consumer_copier == "bulk":
            return D.dtt_plan_opts_default(method=D.COPY_TMA, piece_bytes=32768, stages=2)
        return D.dtt_plan_opts_default(copier_threads=args.consumer_copier_threads)

    def measure(grouped):
        st = runner.make(w, opts=copts(), copy_stream=copy_stream, **launch)
        n_groups = None
        if grouped:     # one group per 128-row block of X, before the first round
            n_groups, _ = st.plan.define_block_groups(128 * 2 * K)
        prod = st.producer_stream

        def ag():
            h = st.plan.start(prod)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, prod)
            st.plan.wait()
            st.plan.next_round()

        def overlapped():
            h = st.plan.start(prod)
            st.plan.gemm_consumer(0, Wt, out, N2, K, err, stream=cons)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, prod)
            st.plan.wait()
            prod.wait_stream(cons)
            st.plan.next_round()

        def timed(fn, K_):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(prod)
            for _ in range(K_):
                fn()
            e1.record(prod)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / K_

        K_ = max(3, min(args.steps, 50))
        ag_ms = timed(ag, K_)
        ov_ms = timed(overlapped, K_)
        gemm = []
        for _ in range(K_):                 # the GEMM alone: its chunks have all arrived
            h = st.plan.start(prod)
            D.dtt_fill_producer(st.buf_ptrs, st.desc, h, prod)
            torch.cuda.synchronize()        # producer and copier done
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cons)
            st.plan.gemm_consumer(0, Wt, out, N2, K, err, stream=cons)
            e1.record(cons)
            st.plan.wait()
            cons.synchronize()
            st.plan.next_round()
            gemm.append(e0.elapsed_time(e1))
        st.plan.close()
        assert int(err.item()) == 0
        return K_, ag_ms, ov_ms, statistics.median(gemm), n_groups

    K_, ag_ms, ov_ms, gemm_ms, _ = measure(False)
    _, ag_g, ov_g, gemm_g, n_groups = measure(True)
    flops = 2.0 * rows * N2 * K
    tf_peak, tf_kind = load_tensor_peak()
    line = {"metric": "all-gather + consumer GEMM round, overlapped (1 GB300)", "unit": "ms per round",
            "higher_is_better": False, "steps": K_, "value": ov_ms,
            "config": {"workload": describe(w, launch) + f"; consumer GEMM: rank 0's [{rows}, {K}] bf16 "
                                                           f"x W^T [{N2}, {K}], tcgen05, 148 CTAs",
                       "copier": copier_desc},
            "all_gather_ms": ag_ms, "gemm_alone_ms": gemm_ms,
            "sequential_ms": ag_ms + gemm_ms, "overlap_saving": 1.0 - ov_ms / (ag_ms + gemm_ms),
            "gemm_alone_tflops": flops / (gemm_ms / 1e3) / 1e12,
            "gemm_alone_frac": flops / (gemm_ms / 1e3) / 1e12 / tf_peak, "peak_kind": tf_kind,
            "group_waits": {"groups": n_groups, "overlapped_ms": ov_g, "all_gather_ms": ag_g,
                            "gemm_alone_ms": gemm_g,
                            "overlap_saving": 1.0 - ov_g / (ag_g + gemm_g)}}
    print(json.dumps(line))
    return 0


def run_ce_fanout(args):
    """Copy engines against the SM copier on the same fan-out: every rank's slice copied to the
    P-1 peers with one device-to-device cudaMemcpyAsync per (source, peer), spread over a few
    streams and not gated (the copy-engine transport the pages pre-arm), against this build's
    copier moving the same bytes with its gates already open (a deferred plan)."""
    import torch
    import device_triggered_transfers_gb300 as D
    from device_triggered_transfers_gb300 import runner
    w = workload(args)
    S = w.slice_bytes
    launch = dict(runner.bench_launch(w, overlap=False))
    launch.pop("pace", None)          # the copier starts after the producer here
    opts = launch.pop("opts", None) or D.dtt_plan_opts_default()
    opts.deferred_copier, opts.time_copier = 1, 1
    st = runner.make(w, opts=opts, **launch)
    prod = st.producer_stream
    res = {}
    for n_streams in (1, w.P - 1, w.P * (w.P - 1)):
        streams = [torch.cuda.Stream() for _ in range(n_streams)]

        def fan_out():
            i = 0
            for r in w.senders():
                src = st.bufs[r][w.slice_offset(r):w.slice_offset(r) + S]
                for q in range(w.P):
                    if q == r:
                        continue
                    with torch.cuda.stream(streams[i % n_streams]):
                        st.bufs[q][w.slice_offset(r):w.slice_offset(r) + S].copy_(src, non_blocking=True)
                    i += 1
        for _ in range(3):
            fan_out()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        reps = 20
        for _ in range(reps):
            fan_out()
        torch.cuda.synchronize()
        dt = (time.perf_counter() - t0) / reps
        res[f"ce_{n_streams}_streams_ms"] = dt * 1e3
        res[f"ce_{n_streams}_streams_gbs_delivered"] = w.delivered_bytes_per_round() / dt / 1e9
    for _ in range(3):                  # the SM copier alone: producer first, then the copier
        runner.run_round(st)
        st.plan.next_round()
    c0 = st.plan.stats()
    for _ in range(20):
        runner.run_round(st)
        st.plan.next_round()
    c1 = st.plan.stats()
    st.plan.close()
    cop_ms = (c1[1] - c0[1]) / (c1[2] - c0[2])
    res["sm_copier_ms"] = cop_ms
    res["sm_copier_gbs_delivered"] = w.delivered_bytes_per_round() / (cop_ms / 1e3) / 1e9
    del st
    torch.cuda.empty_cache()
    # whole gated rounds, the benchmark's producer each time: the copy engines driven by the
    # plan's host proxy (poll, copy, atomic per chunk) against the benchmark's SM copier launch
    peak, peak_kind = load_peaks()
    K = max(3, min(args.steps, 100))
    gated = {}
    for name, method in (("copy_engines", D.COPY_ENGINE), ("sm_copier", None)):
        m = measure_workload(w, args, K, 3, 5, 0, with_e2e=False, method=method)
        sm = summarize(m, K, m["elapsed_s"], w.delivered_bytes_per_round() * K, peak, peak_kind)
        gated[name] = {"ms_per_round": sm["ms_per_round"], "gbs_delivered": sm["gbs_delivered"],
                       "hbm_frac_end_to_end": sm["hbm_frac_end_to_end"]["of_measured"],
                       "gate_to_arrival_ns": {k: sm["gate_to_arrival_ns"][k] for k in
                                              ("median", "p99", "median_over_ideal", "p99_over_ideal")}}
    res["gated_rounds"] = gated
    line = {"metric": "fan-out of one all-gather round: copy engines vs the SM copier (1 GB300)",
            "unit": "GB/s delivered", "higher_is_better": True,
            "config": {"workload": describe(w, launch)}, **res}
    print(json.dumps(line))
    return 0


def measure_allreduce(K: int, warmup: int, isolated_rounds: int = 10, e2e_steps: int = 0,
                      clocks_dev=None, rows: int = 0, in_order: bool = False, ctas_per_sm: int = 0,
                      stages: int = 0, piece_bytes: int = 0, fill_rounds: int = 0, reduce_ctas: int = 0,
                      reduce_threads: int = 0, gather: bool = True, ag_ctas_per_sm: int = 0,
                      host_piece_bytes: int = 0):
    """The two-shot all-reduce of W.ALLREDUCE.  The collective: K rounds of start + a producer that
    only marks (dtt_publish: the vectors were written before the timed region, as an all-reduce
    benchmark's inputs are) + reduce kernel + wait + next_round (both plans' copiers launched at
    start), CUDA events on the producer stream with a synchronize on both sides -- in place, so
    each round's result is the next round's input (the values grow by P a round, finite over
    these rounds).  Then fill_rounds rounds whose producer is the fill (writing every rank's
    whole vector), the reduce kernel alone (launched once the reduce-scatter copier has finished,
    on a stream of its own), and (e2e_steps > 0) rounds fed from pinned host memory through
    dtt_publish with rank 0's result read back.  in_order: both plans with deferred_copier = 1,
    every kernel after its inputs (for profilers that serialise launches; the isolated reduce
    then includes its wait for the copier)."""
    import torch
    import device_triggered_transfers_gb300 as D
    a = W.ALLREDUCE
    P, cols, J, dtype = a["P"], a["cols"], a["sub_blocks"], a["dtype"]
    Mb = rows or a["block_rows"]
    M = P * Mb
    rb = cols * W.ELEM_BYTES[dtype]
    S = M * rb                      # one rank's vector
    buf_bytes = 2 * S               # the vector, then the P slots
    dev = torch.device("cuda")
    bufs = [torch.zeros(buf_bytes, dtype=torch.uint8, device=dev) for _ in range(P)]
    prod, side = torch.cuda.Stream(), torch.cuda.Stream()
    rs_cs, ag_cs = torch.cuda.Stream(priority=-1), torch.cuda.Stream(priority=-1)
    opts = ag_opts = None
    if in_order or ctas_per_sm or stages or piece_bytes or ag_ctas_per_sm or host_piece_bytes:
        opts = D.dtt_plan_opts_default(method=D.COPY_TMA, ctas_per_sm=ctas_per_sm or 3,
                                       piece_bytes=piece_bytes or 16384, stages=stages or 2,
                                       deferred_copier=1 if in_order else 0,
                                       host_piece_bytes=host_piece_bytes)
        ag_opts = D.dtt_plan_opts_default(method=D.COPY_TMA, ctas_per_sm=ag_ctas_per_sm or ctas_per_sm or 3,
                                          piece_bytes=piece_bytes or 16384, stages=stages or 2,
                                          deferred_copier=1 if in_order else 0)
    ar = D.AllReduce(bufs, buf_bytes, dtype, Mb, cols, sub_blocks=J, rs_opts=opts, ag_opts=ag_opts,
                     reduce_ctas=reduce_ctas, reduce_threads=reduce_threads,
                     rs_copy_stream=rs_cs, ag_copy_stream=ag_cs, gather=gather)
    Mj = Mb // J
    counters = torch.zeros(P * (M // Mj), dtype=torch.int32, device=dev)
    desc = D.fill_desc(dtype, a["seed"], M, cols, rb, buf_bytes, [0] * P, Mj, cols, 1, 1,
                       mark_mode=D.MARK_PER_STEP, group=a["fill_group"], group_counters=counters)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    n_rs = ar.rs.info()[0]

    def one(fill=False):
        h = ar.start(prod)
        if fill:
            D.dtt_fill_producer(bufs, desc, h, prod)
        else:
            D.dtt_publish(h, 0, n_rs, 0, prod)      # every reduce-scatter chunk's marks
        ar.reduce(err, prod)
        ar.wait()
        ar.next_round()

    for _ in range(warmup):
        one(fill=True)
    one(fill=True)                                   # fresh inputs for the timed rounds
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {}
    sampler = ClockSampler(clocks_dev) if clocks_dev is not None else None
    if sampler:
        sampler.__enter__()
    e0.record(prod)
    for _ in range(K):
        one()
    e1.record(prod)
    torch.cuda.synchronize()
    if sampler:
        sampler.__exit__(None, None, None)
        out["clocks"] = sampler.summary()
    out["round_ms"] = e0.elapsed_time(e1) / K
    assert int(err.item()) == 0
    if fill_rounds:
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(prod)
        for _ in range(fill_rounds):
            one(fill=True)
        f1.record(prod)
        torch.cuda.synchronize()
        out["fill_round_ms"] = f0.elapsed_time(f1) / fill_rounds

    # the reduce kernel alone, on an all-reduce over the same buffers whose kernels run in order:
    # its reduce-scatter copier (launched here, after the fill) has finished before the reduce
    # starts on a stream of its own, and its all-gather copier starts after the reduce
    iso = []
    if isolated_rounds:
        serial = D.dtt_plan_opts_default(method=D.COPY_TMA, ctas_per_sm=ctas_per_sm or 3,
                                         piece_bytes=piece_bytes or 16384, stages=stages or 2, deferred_copier=1)
        ars = D.AllReduce(bufs, buf_bytes, dtype, Mb, cols, sub_blocks=J, rs_opts=serial, ag_opts=serial,
                          reduce_ctas=reduce_ctas, reduce_threads=reduce_threads,
                          rs_copy_stream=rs_cs, ag_copy_stream=ag_cs)
        for i in range(isolated_rounds + 2):
            h = ars.start(prod)
            D.dtt_fill_producer(bufs, desc, h, prod)
            ars.rs.launch_copier()
            ev = torch.cuda.Event()
            ev.record(rs_cs)
            side.wait_event(ev)
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            r0.record(side)
            ars.reduce(err, side)
            r1.record(side)
            ars.wait()
            ars.next_round()
            torch.cuda.synchronize()
            if i >= 2:
                iso.append(r0.elapsed_time(r1))
        ars.close()
    out["reduce_isolated_ms"] = statistics.median(iso) if iso else None
    assert int(err.item()) == 0

    if e2e_steps:
        g = torch.Generator().manual_seed(a["seed"])
        host = [torch.randn(M, cols, generator=g).to(torch.bfloat16).view(torch.uint8).reshape(-1).pin_memory()
                for _ in range(P)]
        host_out = torch.empty(S, dtype=torch.uint8).pin_memory()

        def host_round():
            # dtt_allreduce_host: the partials go in sub-block by sub-block, each reduce-scatter
            # chunk marked once its rows have landed, the reduce running meanwhile, and rank 0's
            # result coming back as the all-gather delivers it
            ar.host_round(host, err, host_out=host_out, out_rank=0, stream=prod)

        for _ in range(2):
            host_round()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_round()
        torch.cuda.synchronize()
        out["e2e_round_ms"] = (time.perf_counter() - t0) / e2e_steps * 1e3
        out["e2e_bytes"] = (P * S, S)
        assert int(err.item()) == 0
    ar.close()
    out.update(P=P, S=S, Mb=Mb, cols=cols, J=J, dtype=dtype)
    return out


def summarize_allreduce(m, peak, peak_kind):
    """Bandwidths and roofline fractions of measure_allreduce's numbers.  Algorithmic HBM bytes
    of a round (the producer's writes aside, as for the all-gathers): the reduce-scatter copies
    read and write (P-1) S, the reduce reads P S and writes S, the all-gather copies read S and
    write (P-1) S: (4P - 1) S in all, S = one rank's vector."""
    P, S = m["P"], m["S"]
    t = m["round_ms"] * 1e-3
    alg = (4 * P - 1) * S
    red = (P + 1) * S               # the reduce kernel: P parts of every block read, one written
    algbw = S / t / 1e9
    res = {"ms_per_round": m["round_ms"], "algbw_gbs": algbw, "busbw_gbs": algbw * 2 * (P - 1) / P,
           "algorithmic_bytes_per_round": alg,
           "hbm_frac_end_to_end": {"of_measured": alg / t / 1e9 / peak, "peak_kind": peak_kind}}
    if m.get("reduce_isolated_ms"):
        achieved = red / (m["reduce_isolated_ms"] * 1e-3) / 1e9
        res["reduce_roofline"] = {"kernel": "reduce_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                                  "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                                  "traffic": NCU_TRAFFIC.get(("allreduce_p4", "reduce_kernel")),
                                  "algorithmic_bytes_per_launch": red, "ms": m["reduce_isolated_ms"]}
    return res


def run_allreduce(args):
    """One JSON line for the two-shot all-reduce (W.ALLREDUCE)."""
    import torch
    dev = torch.cuda.current_device()
    K = args.steps
    m = measure_allreduce(K, args.warmup, isolated_rounds=10, e2e_steps=0 if args.no_e2e else 10,
                          clocks_dev=dev, rows=args.rows, in_order=args.in_order,
                          ctas_per_sm=args.ctas_per_sm, stages=args.stages, piece_bytes=args.piece_bytes,
                          fill_rounds=20, reduce_ctas=args.reduce_ctas, reduce_threads=args.reduce_threads,
                          ag_ctas_per_sm=args.ag_ctas_per_sm, host_piece_bytes=args.host_piece_bytes)
    peak, peak_kind = load_peaks()
    s = summarize_allreduce(m, peak, peak_kind)
    # the reduce-scatter alone (the first shot: no all-gather plan), the same way
    mr = measure_allreduce(K, args.warmup, isolated_rounds=0, rows=args.rows, in_order=args.in_order,
                           ctas_per_sm=args.ctas_per_sm, stages=args.stages, piece_bytes=args.piece_bytes,
                           reduce_ctas=args.reduce_ctas, reduce_threads=args.reduce_threads, gather=False)
    t_rs = mr["round_ms"] * 1e-3
    reduce_scatter = {"ms_per_round": mr["round_ms"], "algbw_gbs": mr["S"] / t_rs / 1e9,
                      "algorithmic_bytes_per_round": (3 * mr["P"] - 1) * mr["S"],
                      "hbm_frac_of_measured": (3 * mr["P"] - 1) * mr["S"] / t_rs / 1e9 / peak}
    a = W.ALLREDUCE
    cpu = None
    if not args.no_cpu_baseline:
        v, n, dt, what = time_oracle_allreduce(budget_s=args.cpu_seconds)
        cpu = {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{what}; {n} oracle round(s) in {dt:.1f} s"}
    e2e = None
    if "e2e_round_ms" in m:
        e2e = {"value": m["S"] / (m["e2e_round_ms"] * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": m["e2e_bytes"][0], "d2h_bytes_per_step": m["e2e_bytes"][1],
               "call": ("dtt_allreduce_host: partials from pinned host memory in sub-block pieces, each "
                        "reduce-scatter chunk marked as its rows land, the reduce meanwhile, rank 0's "
                        "result copied back as the all-gather delivers it")}
    line = {
        "metric": "two-shot all-reduce algorithm GB/s (one rank's vector bytes per round, 1 GB300)",
        "value": s["algbw_gbs"], "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": s["ms_per_round"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 sums of bf16", "data": "synthetic",
        "config": {"workload": (f"{a['name']}: P={m['P']} virtual ranks, {m['dtype']} [{m['P'] * m['Mb']}, {m['cols']}] "
                                f"per rank, blocks of {m['Mb']} rows in {m['J']} sub-blocks; reduce-scatter into "
                                "staging slots after each vector, reduce kernel, in-place all-gather; both "
                                "plans bulk-copy copiers of 3 CTAs x 2 x 16 KiB per SM; fill producer a group "
                                f"of {a['fill_group']} CTAs per rank"),
                   "step": ("start (both plans) + marks of every reduce-scatter chunk (inputs resident, "
                            "in place) + reduce + wait (both) + next_round"),
                   "l2": f"inputs larger than L2 ({m['P'] * 2 * m['S'] >> 20} MiB of buffers)"},
        "busbw_gbs": s["busbw_gbs"],
        "hbm_frac_end_to_end": s["hbm_frac_end_to_end"],
        "with_fill_producer_ms_per_round": m.get("fill_round_ms"),
        "reduce_scatter": reduce_scatter,
        "roofline": s.get("reduce_roofline"),
        "e2e": e2e,
        "gpu_launches": 6 * K,      # marks, 2 copiers, reduce, 2 checks per round
        "clocks": m.get("clocks"),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    return 0


def run_barrier(args):
    """Latency of the N-rank notify/wait barrier and the builtin reveal (P = 8 virtual ranks,
    reveal SIZE = 256): one cooperative launch per barrier, CUDA events around K of them."""
    import torch
    import device_triggered_transfers_gb300 as D
    P, size = W.BARRIER_P, W.BARRIER_SIZE
    sig = [torch.zeros(P, dtype=torch.int32, device="cuda") for _ in range(P)]
    y = [torch.zeros(P, dtype=torch.int32, device="cuda") for _ in range(P)]
    status = torch.zeros(P, dtype=torch.int32, device="cuda")
    x_np = W.barrier_payload(P, size)
    x = [torch.from_numpy(x_np[r].copy()).cuda() for r in range(P)]
    data = [torch.zeros(size, dtype=torch.int32, device="cuda") for _ in range(P)]
    yr = [torch.zeros(size, dtype=torch.int32, device="cuda") for _ in range(P)]
    b = D.Barrier(P)
    s = torch.cuda.current_stream()
    out = {}
    gen = 0
    # arguments checked and marshalled once, as a caller that reuses its windows would do
    hargs = D.HandrolledArgs(sig, y, status)
    rargs = D.RevealArgs(x, data, yr, size, status)
    for name in ("handrolled", "reveal"):
        def one():
            nonlocal gen
            if name == "handrolled":
                gen += 1
                D.dtt_barrier_handrolled(hargs, gen=gen, max_polls=1 << 24, stream=s)
            else:
                b.reveal(rargs, max_polls=1 << 24, stream=s)
        for _ in range(args.warmup):
            one()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(args.steps):
            one()
        e1.record(s)
        torch.cuda.synchronize()
        assert int(status.abs().sum()) == 0
        out[name] = e0.elapsed_time(e1) / args.steps * 1e3
    b.destroy()
    print(json.dumps({"metric": "N-rank barrier latency (P=8 virtual ranks)", "unit": "us per barrier",
                      "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
                      "handrolled_us": out["handrolled"], "reveal_us": out["reveal"],
                      "config": {"workload": "barrier: int32 [8,1] signal windows; reveal [1,256]",
                                 "launch": "one cooperative launch per barrier, 8 CTAs"}}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(W.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deferred", action="store_true",
                    help="launch each round's copier after its producer (for profilers that "
                         "serialise kernels)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--overlap", dest="overlap", action="store_const", const=True, default=None,
                    help="overlapping rounds (opts.overlap) for every workload: each round's "
                         "producer runs while the previous round's copier still copies (default: "
                         "where the benchmark's launch uses them)")
    ap.add_argument("--sequential", dest="overlap", action="store_const", const=False,
                    help="rounds one at a time for every workload")
    ap.add_argument("--copier", choices=["vector", "bulk"], default=None,
                    help="copier data path (default: the launch's)")
    ap.add_argument("--piece-bytes", type=int, default=0, help="copier piece size (default: the launch's)")
    ap.add_argument("--stages", type=int, default=0, help="bulk copier stages per CTA (default: the launch's)")
    ap.add_argument("--ctas-per-sm", type=int, default=0, help="copier CTAs per SM (default: the launch's)")
    ap.add_argument("--copier-threads", type=int, default=0, help="vector copier threads per CTA")
    ap.add_argument("--copier-ctas", type=int, default=0, help="copier CTAs in all (default: per SM)")
    ap.add_argument("--host-piece-bytes", type=int, default=0,
                    help="host-buffer round: bytes per host-to-device copy (default: the plan's)")
    ap.add_argument("--pace", type=int, default=-1,
                    help="the fill producer's pacing in chunks (default: the launch's own)")
    ap.add_argument("--latency-rounds", type=int, default=20)
    ap.add_argument("--isolated-rounds", type=int, default=20)
    ap.add_argument("--barrier", action="store_true",
                    help="time the N-rank barrier and the builtin reveal instead")
    ap.add_argument("--ce-fanout", action="store_true",
                    help="time the fan-out with copy engines (device-to-device memcpy) against the SM copier")
    ap.add_argument("--allreduce", action="store_true",
                    help="time the two-shot all-reduce (reduce-scatter plan, reduce kernel, all-gather plan)")
    ap.add_argument("--ag-ctas-per-sm", type=int, default=0,
                    help="--allreduce: the all-gather plan's copier CTAs per SM (default: --ctas-per-sm, else 3)")
    ap.add_argument("--reduce-ctas", type=int, default=0, help="--allreduce: reduce kernel CTAs (default: one per SM)")
    ap.add_argument("--reduce-threads", type=int, default=0, help="--allreduce: threads per reduce CTA (default 256)")
    ap.add_argument("--in-order", action="store_true",
                    help="--allreduce: each kernel after its inputs (deferred copiers), for profiler captures")
    ap.add_argument("--consumer", action="store_true",
                    help="time the all-gather with a consumer GEMM over its output, overlapped")
    ap.add_argument("--consumer-n", type=int, default=4096)
    ap.add_argument("--consumer-copier-threads", type=int, default=256)
    ap.add_argument("--consumer-copier", choices=["vector", "bulk"], default="vector")
    ap.add_argument("--profile-rounds", type=int, default=0,
                    help="run this many rounds after the warm-up inside a profiler range "
                         "(cudaProfilerStart/Stop) and exit, for ncu --replay-mode app-range")
    ap.add_argument("--early-us", type=int, default=-1,
                    help="opts.early_copier_us for the timed plans (-1: the launch's own setting, "
                         "0: off)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="time only the named workload (default: also the other workloads, "
                         "reported under per_config)")
    ap.add_argument("--rows", type=int, default=0,
                    help="rows per rank instead of the workload's (a smaller case of the same "
                         "shape, for profiler captures; the default runs the workload as named)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.barrier and args.impl == "ours":
        return run_barrier(args)
    if args.consumer and args.impl == "ours":
        return run_consumer(args)
    if args.allreduce and args.impl == "ours":
        return run_allreduce(args)
    if args.ce_fanout and args.impl == "ours":
        return run_ce_fanout(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
