"""Benchmark: decode attention over a quantized KV cache on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long] [--impl reference]

A step = one pass of the whole decode path over one batch: the newest token(s)
of every cache are appended and every cache is decoded, by one
kvq_decode_attn_multi call with the appends fused into the attention kernel
(split-KV attention + log-sum-exp combine).  The same step through kvq_append
and kvq_decode_attn per cache is timed beside it.  The default workload is the long-context
decode: a main cache (40 query / 8 kv heads) and a draft cache (16 / 4), each
131072 positions built in 4 append-only segments, q4_0 V, one query token each.

Timed region (value): CUDA-graph replays of the step, rotating between enough
independent copies of the caches that their total exceeds L2 several times, so
no step reads KV left in L2 by the previous one; CUDA events on the launching
stream, synchronize + barrier on both sides; max over ranks.  Multi-GPU runs
are independent replicas (the path needs no exchange).

The reference arm (--impl reference) times the fp64 CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn tokens/s and KV HBM GB/s (% of 8 TB/s) at 128k ctx, 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
L2_BYTES = 129 * 1024 * 1024
SPREAD_MIN_REPLAYS = 5      # replays behind the step-time spread
SPREAD_MAX_REPLAYS = 4000
SPREAD_SECONDS = 1.0        # length of the spread pass (clock samples every 100 ms)
PRE_SLEEP_CYCLES = 4_000_000   # ~2 ms at 2 GHz, untimed, ahead of the timed region

WORKLOADS = {
    "long": "long-context decode: main 40q/8kv heads + draft 16q/4kv heads, 131072 positions each "
            "in 4 append-only segments, head_dim 128, K int8 per-32 fp16 scale, V q4_0, 1 query token",
    "single": "single-sequence decode: 32q/8kv heads, 8192 positions, V q4_0, 4 outlier channels x10",
    "batched": "batched decode: 64 sequences, lengths U[1024, 32768], 32q/8kv heads, V q8_0, outliers x10",
    "verify": "multi-token verify: 16 sequences x 4 causal query tokens, 32768 positions, 64q/8kv heads, V q4_0",
    "tiny": "tiny: 1 kv head, 4 query heads, 256 positions, V q8_0",
    "long_f16k": "long-context decode with F16 K (K kept as fp16 values, query unquantized) and q4_0 V: "
                 "main 40q/8kv + draft 16q/4kv heads, 131072 positions each in 4 segments, 1 query token",
    "prefill": "chunked prefill: one 512-token chunk (causal among its tokens) over 32768 positions, "
               "32q/8kv heads, V q4_0; the chunk is appended by kvq_append, then attended",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30000)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--workload", default="long", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--graph-passes", type=int, default=8,
                    help="passes over the rotating cache copies captured in one timed CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="time budget of the reference arm (warm-up + timed steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", default="bench", choices=["bench", "profile"],
                    help="profile: one cache copy, a few directly launched steps, no timing (for ncu)")
    ap.add_argument("--ctx", type=int, default=None, help="shrink the workload's context (profile mode)")
    ap.add_argument("--layout", default="auto", choices=["auto", "tiles", "rows"],
                    help="segment layouts: auto = kvq_choose_layout per segment (the library's cost model), "
                         "or every segment in tiles / rows")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def job_rate(ms_local, world, steps, tokens_per_step, device=None):
    """Whole-job timing across ranks: the max of the ranks' timed milliseconds
    (all-reduce MAX when world > 1) -> (ms per step, tokens/s of all ranks)."""
    ms = float(ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_per_step = ms / steps
    return ms_per_step, tokens_per_step * world / (ms_per_step * 1e-3)


def timing_plan(steps, n_rot, graph_passes):
    """How exactly `steps` timed steps run as CUDA-graph replays: a graph of
    per_replay steps (at most graph_passes whole passes over the n_rot cache
    copies, and at most `steps`), replayed `reps` times, then one graph of the
    remaining rem < per_replay steps.  When per_replay is below `steps` it is
    a multiple of n_rot, so consecutive steps never decode the same copy."""
    k = max(1, int(steps))
    per = min(k, max(1, n_rot) * max(1, graph_passes))
    reps, rem = divmod(k, per)
    return per, reps, rem


def measured_peaks(kind="hbm_gbs"):
    """(peak, 'measured'|'fallback'): HBM copy GB/s, or the bf16 GEMM TFLOP/s
    sustained over seconds (kind='bf16_tflops_sustained')."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get(kind):
            return float(d[kind]), "measured"
    return (FALLBACK_HBM_GBS if kind == "hbm_gbs" else FALLBACK_BF16_TFLOPS_SUSTAINED), "fallback"


# Source files that define each profiled kernel: a committed ncu summary stays
# valid while these are unchanged.
KERNEL_SOURCES = {
    "split_attn": ["csrc/kvq_attn.cuh", "csrc/kvq_attn_q4.cu", "csrc/kvq_attn_q8.cu", "csrc/kvq_internal.cuh"],
    "prefill_attn": ["csrc/kvq_prefill.cuh", "csrc/kvq_prefill_q4.cu", "csrc/kvq_prefill_q8.cu",
                     "csrc/kvq_internal.cuh"],
}


_COMMENT = re.compile(rb"/\*.*?\*/|//[^\n]*", re.S)
_SPACE = re.compile(rb"\s+")


def kernel_source_hash(kernel="split_attn"):
    """Hash of the kernel's source files with C comments removed and every run
    of white space collapsed to one blank, so that counters taken on a kernel
    stay valid across comment-only and layout-only edits."""
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "quantized_kv_cache_03_gb300")
    for f in KERNEL_SOURCES[kernel] + ["../include/kvq.h"]:
        with open(os.path.normpath(os.path.join(pkg, f)), "rb") as fh:
            h.update(_SPACE.sub(b" ", _COMMENT.sub(b"", fh.read())).strip())
            h.update(b"\n")
    return h.hexdigest()[:16]


def launches_of(grp, fused):
    """Kernels one step launches: the fused call's split kernel (one per launch
    group of <= 64 sequences / 64 segments / 8 work groups; the appends run
    inside it) and, when any sequence is split, its combine; plus one append
    per cache when the appends are not fused."""
    seqs = sum(ds.B for ds in grp)
    segs = sum(len(x) for ds in grp for x in ds.spec.segments)
    groups = max(-(-seqs // 64), -(-segs // 64), -(-len(grp) // 8))
    return (0 if fused.append else len(grp)) + groups * (2 if fused.call.ws is not None else 1)


def profiled_traffic(workload, kernel="split_attn"):
    """DRAM bytes per step of the dominant kernel from the committed ncu
    record profiles/<kernel>_<workload>.json (written beside each ncu
    summary), if it was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "%s_%s.json" % (kernel, workload))
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    tr = rec.get("traffic_bytes_per_step")
    return None if tr is None else float(tr)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 hw=f[5], hwt=f[6], swt=f[7], pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [r["sm"] for r in rows]
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------------------ oracle --

def _oracle_caches(specs_data):
    import oracle
    caches = []
    for d in specs_data:
        s = d.spec
        for b in range(s.n_seqs):
            k, v = d.kv[b]
            caches.append((s, b, oracle.quantize_kv(k, v, s.v_type), d.q[b]))
    return caches


def run_oracle(specs_data, seconds, threads):
    """The fp64 oracle on the host: quantize the caches (untimed), then time
    whole decode steps over all caches until `seconds` have passed."""
    import oracle
    caches = _oracle_caches(specs_data)
    tokens_per_step = sum(d.spec.n_seqs * d.spec.t_q for d in specs_data)
    n = 0
    t0 = time.perf_counter()
    while True:
        for s, b, c, q in caches:
            oracle.decode_seq(c, q, oracle.default_head_map(s.n_q_heads, s.n_kv_heads), s.causal,
                              1.0 / np.sqrt(128.0), s.v_type, n_threads=threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return tokens_per_step * n / el, n, el


def run_oracle_rows(specs_data, steps, warmup, threads, budget_s):
    """Reference arm: the oracle on a bounded sample of the workload.  A step
    decodes `threads` query rows (cycling over every row of every cache, one
    OpenMP thread per row); a whole decode step of the workload is all its rows,
    so tokens/s = rows done * (tokens per step / rows per step) / seconds.
    Warm-up and timed steps stop early when the time budget is spent."""
    import oracle
    caches = _oracle_caches(specs_data)
    rows = [(ci, r) for ci, (s, b, c, q) in enumerate(caches) for r in range(s.t_q * s.n_q_heads)]
    tokens_per_step = sum(d.spec.n_seqs * d.spec.t_q for d in specs_data)
    pos = 0

    def one_step():
        nonlocal pos
        pick = [rows[(pos + i) % len(rows)] for i in range(min(threads, len(rows)))]
        pos = (pos + len(pick)) % len(rows)
        by_cache = {}
        for ci, r in pick:
            by_cache.setdefault(ci, []).append(r)
        for ci, rs in by_cache.items():
            s, b, c, q = caches[ci]
            mask = np.zeros(s.t_q * s.n_q_heads, np.uint8)
            mask[rs] = 1
            oracle.decode_seq(c, q, oracle.default_head_map(s.n_q_heads, s.n_kv_heads), s.causal,
                              1.0 / np.sqrt(128.0), s.v_type, row_mask=mask, n_threads=threads)
        return len(pick)

    t_start = time.perf_counter()
    w = 0
    while w < warmup and time.perf_counter() - t_start < 0.2 * budget_s:
        one_step()
        w += 1
    n, done_rows = 0, 0
    t0 = time.perf_counter()
    while n < max(1, steps):
        done_rows += one_step()
        n += 1
        if time.perf_counter() - t0 >= 0.8 * budget_s:
            break
    el = time.perf_counter() - t0
    return done_rows * tokens_per_step / len(rows) / el, n, w, el, done_rows, len(rows)


# ---------------------------------------------------------------- GPU arm --

def main():
    args = parse()
    rank, world, local = dist_env()
    from quantized_kv_cache_03_gb300 import workloads as W

    specs = W.make_spec(args.workload, ctx=args.ctx)
    kv_bytes = W.step_kv_bytes(specs)
    tokens_per_step = sum(s.n_seqs * s.t_q for s in specs)
    threads = os.cpu_count() or 1

    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        from quantized_kv_cache_03_gb300.harness import HostData
        import oracle
        oracle.build()
        data = [HostData(s) for s in specs]
        tps, n, w, el, done_rows, n_rows = run_oracle_rows(data, args.steps, args.warmup, threads,
                                                           max(10.0, args.ref_seconds))
        sample = ("%d steps of %d query rows each (%d of the workload's %d rows per decode step, cycling), "
                  "fp64 oracle, OpenMP over rows, %.1f s timed" % (n, min(threads, n_rows), done_rows, n_rows, el))
        line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": n, "warmup": w, "ms_per_step": 1e3 * el / n, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": WORKLOADS[args.workload], "oracle_threads": threads},
                "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_kv_cache_03_gb300 import kvq
    from quantized_kv_cache_03_gb300.harness import DecodeSet, HostData, StepSet

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    data = [HostData(s) for s in specs]
    # the step's appends run inside the attention kernel when every cache
    # takes at most KVQ_MAX_T_Q_APPEND tokens per step; else kvq_append first
    fusable = all(s.t_q <= kvq.MAX_T_Q_APPEND and s.k_type == W.K_I8 for s in specs)
    layout = {"auto": "auto", "tiles": kvq.LAYOUT_TILES, "rows": kvq.LAYOUT_ROWS}[args.layout]
    if args.mode == "profile":
        grp = [DecodeSet(d, dev, layout=layout) for d in data]
        for ds in grp:
            ds.staging = None
        fused = StepSet(grp, append=fusable)
        for _ in range(max(1, args.warmup) + max(1, args.steps)):
            if not fusable:
                for ds in grp:
                    ds.append_step()
            fused.decode()
            for ds in grp:
                ds.rewind()
        torch.cuda.synchronize()
        print(json.dumps({"mode": "profile", "workload": args.workload, "ctx": args.ctx,
                          "steps": max(1, args.warmup) + max(1, args.steps),
                          "launches_per_step": launches_of(grp, fused),
                          "kv_bytes_per_step": kv_bytes}), flush=True)
        return
    n_rot = max(3, -(-3 * L2_BYTES // max(1, kv_bytes)))
    n_rot = min(n_rot, 64)
    first = [DecodeSet(d, dev, layout=layout) for d in data]
    sets = [first] + [[DecodeSet(d, dev, staging=f.staging, layout=layout) for d, f in zip(data, first)]
                      for _ in range(n_rot - 1)]
    for f in first:
        f.staging = None
    for grp in sets:
        for ds in grp:
            ds.staging = None
    torch.cuda.synchronize()
    fused = [StepSet(grp, append=fusable) for grp in sets]
    launches_per_step = launches_of(sets[0], fused[0])

    stream = torch.cuda.Stream(device=dev)

    def step(grp, fz=None):
        """One step: append every cache's new tokens and decode all caches --
        one kvq_decode_attn_multi call with the appends fused (fz), or per cache
        a kvq_append and a kvq_decode_attn (fz None) -- then rewind."""
        if fz is not None:
            if not fz.append:
                for ds in grp:
                    ds.append_step(stream=stream)
            fz.decode(stream=stream)
        else:
            for ds in grp:
                ds.append_step(stream=stream)
            for ds in grp:
                ds.decode(stream=stream)
        for ds in grp:
            ds.rewind()

    # ---- capture one graph that runs one step on every rotation copy ----
    with torch.cuda.stream(stream):
        for grp, fz in zip(sets, fused):   # warm-up outside capture (first call sets device attributes)
            step(grp, fz)
            step(grp)
    stream.synchronize()
    # The K timed steps run as replays of a graph of per_replay steps (whole
    # passes over the rotation copies, at most --graph-passes of them, at most
    # K) plus one graph of the remaining rem < per_replay steps, so exactly K
    # steps are timed.  Step i of a graph decodes copy i % n_rot, so no two
    # consecutive steps read the same copy.  PDL chains the launches inside a
    # graph only: long graphs are what a decode loop capturing many layers has.
    per_replay, reps, rem = timing_plan(args.steps, n_rot, args.graph_passes)
    warm_steps = max(3, args.warmup)

    def capture(n_steps, body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                body(i % n_rot)
        return g

    g_all = capture(per_replay, lambda r: step(sets[r], fused[r]))
    g_rem = capture(rem, lambda r: step(sets[r], fused[r])) if rem else None
    g_warm = capture(warm_steps, lambda r: step(sets[r], fused[r]))
    # the same steps through kvq_append + kvq_decode_attn per cache (reported beside the fused number)
    g_sep = capture(per_replay, lambda r: step(sets[r]))

    # the step's appends alone: kvq_append per cache, no attention
    def app_only(r):
        for ds in sets[r]:
            ds.append_step(stream=stream)
            ds.rewind()

    g_app = capture(per_replay, app_only)
    # decode timing graph: events around each step's fused decode call (separate pass);
    # external event nodes, so their timestamps can be read after each replay
    g_ev = torch.cuda.CUDAGraph()
    ev_pairs = [(torch.cuda.Event(enable_timing=True, external=True),
                 torch.cuda.Event(enable_timing=True, external=True)) for _ in sets]
    with torch.cuda.graph(g_ev, stream=stream):
        for grp, fz, (a, b) in zip(sets, fused, ev_pairs):
            if not fz.append:
                for ds in grp:
                    ds.append_step(stream=stream)
            a.record(stream)
            fz.decode(stream=stream)
            b.record(stream)
            for ds in grp:
                ds.rewind()

    with torch.cuda.stream(stream):
        g_warm.replay()
    stream.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # An event at every replay boundary of the timed region gives the spread of
    # the step time when the region holds several replays.  With fewer than
    # SPREAD_MIN_REPLAYS (a short --steps), the spread comes from a pass of
    # replays of the same graph right after the timed region, at least
    # SPREAD_MIN_REPLAYS of them and ~SPREAD_SECONDS long, so that the clock
    # sampler also sees several samples under load.
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    spread_reps = 0
    with ClockSampler(local) as clk:
        t_region = time.perf_counter()
        with torch.cuda.stream(stream):
            # a short device-side sleep ahead of the start event keeps the
            # GPU busy while the host enqueues the replays, so the timed
            # region holds the K steps and not the host's launch latency
            torch.cuda._sleep(PRE_SLEEP_CYCLES)
            e0.record(stream)
            for i in range(reps):
                g_all.replay()
                evs[i].record(stream)
            if g_rem is not None:
                g_rem.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        if reps < SPREAD_MIN_REPLAYS:
            region_ms = e0.elapsed_time(e1)
            spread_reps = int(min(SPREAD_MAX_REPLAYS, max(SPREAD_MIN_REPLAYS,
                                                           SPREAD_SECONDS * 1e3 * max(1, reps) / max(region_ms, 1e-3))))
            sev = [torch.cuda.Event(enable_timing=True) for _ in range(spread_reps + 1)]
            with torch.cuda.stream(stream):
                sev[0].record(stream)
                for i in range(spread_reps):
                    g_all.replay()
                    sev[i + 1].record(stream)
            torch.cuda.synchronize()
        clk.region_s = time.perf_counter() - t_region
    if reps >= SPREAD_MIN_REPLAYS:
        marks = [e0] + evs
        rep_ms = np.array([a.elapsed_time(b) for a, b in zip(marks[:-1], marks[1:])]) / per_replay
        spread_src = "replay boundaries of the timed region"
        n_spread = reps
    else:
        rep_ms = np.array([a.elapsed_time(b) for a, b in zip(sev[:-1], sev[1:])]) / per_replay
        spread_src = "replays of the timed graph right after the timed region"
        n_spread = spread_reps
    step_pct = {"p10": float(np.percentile(rep_ms, 10)), "p50": float(np.percentile(rep_ms, 50)),
                "p90": float(np.percentile(rep_ms, 90)), "replays": int(n_spread),
                "steps_per_replay": int(per_replay), "source": spread_src}
    if world > 1:
        torch.distributed.barrier()
    steps = reps * per_replay + rem
    ms_per_step, value = job_rate(e0.elapsed_time(e1), world, steps, tokens_per_step, dev)

    # ---- one decode call per cache instead of the fused call (same steps) ----
    sreps = max(1, min(max(SPREAD_MIN_REPLAYS, reps), 2000 // per_replay))
    with torch.cuda.stream(stream):
        g_sep.replay()
        e0.record(stream)
        for _ in range(sreps):
            g_sep.replay()
        e1.record(stream)
    stream.synchronize()
    sep_ms_per_step = e0.elapsed_time(e1) / (sreps * per_replay)
    with torch.cuda.stream(stream):
        g_app.replay()
        e0.record(stream)
        for _ in range(sreps):
            g_app.replay()
        e1.record(stream)
    stream.synchronize()
    app_ms_per_step = e0.elapsed_time(e1) / (sreps * per_replay)

    # ---- kernel-level timing pass (decode = the split kernel + its combine) ----
    kreps = max(SPREAD_MIN_REPLAYS, min(reps * per_replay // n_rot, 2000 // n_rot))
    tot = 0.0
    with torch.cuda.stream(stream):
        for _ in range(kreps):
            g_ev.replay()
            stream.synchronize()
            for a, b in ev_pairs:
                tot += a.elapsed_time(b)
    dec_ms = tot / (kreps * n_rot)                     # per step (all caches)
    dec_bytes = float(kv_bytes)
    # The split kernel runs once per step (one launch for all caches): its
    # average launch duration is at most the timed region's time per step,
    # which also holds the small combine; that bound gives the achieved rate.
    achieved = float(dec_bytes / (ms_per_step * 1e-3) / 1e9)
    peak, peak_kind = measured_peaks()
    # Long query chunks (prefill) make the attention a dense contraction: each
    # KV byte feeds t_q x group query rows.  Above the machine balance
    # (measured bf16 FLOP/s over copy bytes/s) the kernel is bound by the
    # tensor pipe, and its roofline is FLOPs over the bracketed attention call
    # (the chunk's kvq_append launch is outside the brackets).
    flops = W.step_attn_flops(specs)
    tpeak, tpeak_kind = measured_peaks("bf16_tflops_sustained")
    tensor_bound = flops / max(1, kv_bytes) > tpeak * 1e12 / (peak * 1e9)

    # ---- end to end through the public API with host buffers ----
    # A step's inputs (q, new K, new V of every cache) sit in one pinned host
    # buffer and go over in one H2D copy; its results (out, lse of every
    # cache) come back in one D2H copy.  Each piece starts on a 256-byte
    # boundary (the API wants 16).  The stagings are double-buffered, as a
    # serving loop keeps them: the copies run on a second stream, so step
    # i + 1's inputs go over and step i's results come back while the
    # kernels run; events order every copy against the steps that write or
    # read its buffer.  Steps rotate over the cache copies like the timed
    # region, and the region holds every step's copies.
    grp = sets[0]

    def pack(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += -(-(t.numel() * t.element_size()) // 256) * 256
        return offs, n

    ins = [t for ds in grp for t in (ds.q16, ds.k_new, ds.v_new)]
    outs = [t for ds in grp for t in (ds.out, ds.lse)]
    in_offs, in_bytes = pack(ins)
    out_offs, out_bytes = pack(outs)
    NBUF = 2
    h_in = [torch.zeros(in_bytes, dtype=torch.uint8).pin_memory() for _ in range(NBUF)]
    for hb in h_in:
        for t, o in zip(ins, in_offs):
            nb = t.numel() * t.element_size()
            hb[o:o + nb].copy_(t.detach().contiguous().view(-1).view(torch.uint8).cpu())
    d_in = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    d_out = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    h_out = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(NBUF)]

    def view(buf, t, off):
        nb = t.numel() * t.element_size()
        return buf[off:off + nb].view(t.dtype).view(t.shape)

    h2d, d2h = in_bytes, out_bytes
    e2e_calls = []   # [copy r][buffer j]
    for r in range(n_rot):
        row = []
        for j in range(NBUF):
            dv_in = [view(d_in[j], t, o) for t, o in zip(ins, in_offs)]
            dv_out = [view(d_out[j], t, o) for t, o in zip(outs, out_offs)]
            kv_in = list(zip(dv_in[1::3], dv_in[2::3]))
            row.append((StepSet(sets[r], q16=dv_in[0::3], append=fusable, kv_new=kv_in,
                                outs=list(zip(dv_out[0::2], dv_out[1::2]))), kv_in))
        e2e_calls.append(row)
    cs = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(NBUF)]     # inputs of the buffer's step on the device
    ev_done = [torch.cuda.Event() for _ in range(NBUF)]   # the buffer's step finished
    ev_out = [torch.cuda.Event() for _ in range(NBUF)]    # its results are on the host

    def e2e_run(n, start=None):
        with torch.cuda.stream(cs):
            if start is not None:
                cs.wait_event(start)
            d_in[0].copy_(h_in[0], non_blocking=True)
            ev_in[0].record(cs)
        for i in range(n):
            j, r = i % NBUF, i % n_rot
            fz, kv_in = e2e_calls[r][j]
            stream.wait_event(ev_in[j])
            if i >= NBUF:
                stream.wait_event(ev_out[j])    # step i - 2's results have left d_out[j]
            with torch.cuda.stream(stream):
                if not fusable:
                    for ds, (k, v) in zip(sets[r], kv_in):
                        ds.append_step(k_new=k, v_new=v, stream=stream)
                fz.decode(stream=stream)
                ev_done[j].record(stream)
            for ds in sets[r]:
                ds.rewind()
            with torch.cuda.stream(cs):
                if i + 1 < n:
                    jn = (i + 1) % NBUF
                    if i >= 1:
                        cs.wait_event(ev_done[jn])   # step i - 1 has read d_in[jn]
                    d_in[jn].copy_(h_in[jn], non_blocking=True)
                    ev_in[jn].record(cs)
                cs.wait_event(ev_done[j])
                h_out[j].copy_(d_out[j], non_blocking=True)
                ev_out[j].record(cs)
        stream.wait_event(ev_out[(n - 1) % NBUF])

    e2e_run(6)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(PRE_SLEEP_CYCLES)
        a.record(stream)
    e2e_run(args.e2e_steps, start=a)
    with torch.cuda.stream(stream):
        b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / args.e2e_steps

    # ---- CPU baseline: the oracle on this host's cores (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        tps, n, el = run_oracle(data, args.cpu_seconds, threads)
        cpu = {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": "%d whole decode steps of this workload (fp64, OpenMP over query rows), %.1f s"
                         % (n, el)}

    if rank != 0:
        return
    kv_gbs = kv_bytes / (ms_per_step * 1e-3) / 1e9   # per GPU
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warm_steps, "ms_per_step": ms_per_step, "ms_per_step_spread": step_pct,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8+fp32", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "parallelism": "replicas" if world > 1 else "single",
                   "segment_layout": args.layout if args.layout != "auto" else
                   "auto: kvq_choose_layout per segment -> " + "/".join(sorted({
                       {kvq.LAYOUT_TILES: "tiles", kvq.LAYOUT_ROWS: "rows"}[ds.cache.seg(b, k).layout]
                       for grp in sets for ds in grp for b in range(ds.B) for k in range(ds.cache.n_segs(b))})),
                   "l2": "rotating %d independent cache copies (%.0f MB each, L2 129 MB); CUDA-graph replays"
                         " of %d steps" % (n_rot, kv_bytes / 1e6, per_replay),
                   "timed": "%d replays of a %d-step graph + a %d-step graph; warm-up: %d steps in a graph after"
                            " %d eager steps (first calls and capture)" % (reps, per_replay, rem, warm_steps,
                                                                            3 * n_rot),
                   "kv_bytes_per_step": kv_bytes, "tokens_per_step": tokens_per_step},
        "kv_gbs": kv_gbs, "kv_frac_of_8tbs": kv_gbs / NOMINAL_HBM_GBS,
        "kv_frac_of_measured_copy": kv_gbs / peak,
        "roofline": ({"bound": "hbm", "kernel": "split_attn (appends fused), all caches in one launch per step",
                      "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                      "frac": achieved / peak, "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                      "traffic": profiled_traffic(args.workload),
                      "duration_us": 1e3 * ms_per_step,
                      "duration_basis": "timed region / split launches (the per-step combine included)",
                      "decode_call_us_event_bracketed": 1e3 * dec_ms, "algorithmic_bytes": int(dec_bytes)}
                     if not tensor_bound else
                     {"bound": "tensor",
                      "kernel": "prefill_attn (tcgen05 MMAs, TMEM accumulators, 128-row tiles) + combine"
                      if os.environ.get("KVQ_PREFILL", "1") != "0" else "split_attn over 32-row tiles (mma.sync)",
                      "achieved": flops / (dec_ms * 1e-3) / 1e12, "peak": tpeak,
                      "peak_kind": tpeak_kind + " bf16 cuBLAS sustained (fp16 has the same nominal rate)",
                      "unit": "TFLOP/s", "frac": flops / (dec_ms * 1e-3) / 1e12 / tpeak,
                      "traffic": profiled_traffic(args.workload, "prefill_attn"
                                                  if os.environ.get("KVQ_PREFILL", "1") != "0" else "split_attn"),
                      "duration_us": 1e3 * dec_ms,
                      "duration_basis": "event-bracketed attention call (split + combine), appends outside",
                      "algorithmic_flops": int(flops), "kv_bytes": int(dec_bytes)}),
        "steps_per_s": 1e3 / ms_per_step,
        "per_cache_calls_ms_per_step": sep_ms_per_step,
        "append_alone_ms_per_step": app_ms_per_step,
        "e2e": {"value": tokens_per_step / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "method": "kvq_decode_attn_multi per step (appends fused), eager launches; pinned host "
                          "stagings double-buffered, H2D / D2H on a second stream ordered by events"},
        "gpu_launches": launches_per_step * steps,
        "clocks": dict(clk.summary(), window="timed region + the spread pass after it (%.2f s)"
                       % (clk.region_s,)),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
