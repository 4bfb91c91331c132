"""Throughput of the decode-step DSA indexer on one GB300 (or N replicas).

One step = one pass of the whole indexer over one decode batch through the C
ABI's fused entry point: the scores kernel (page-table lookup, page gather, QK
on the tensor cores, relu-weighted head sum, -inf fill of the full-width row)
followed by the top-k kernel.  The scores kernel is also timed alone (scores
entry point) for the roofline.  Default workload: B=64 requests, 128K max context, every
request 131072 tokens long (32768 live C4 positions per row), keys with 1%
x8 outliers, k=2048, 32768 distinct pages in a shuffled pool (268 MB of live
keys, twice the L2).  The metric is live C4 positions scored and selected per
second; the roofline is live key bytes / scores-kernel time against the
measured HBM copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own replica of the workload on its own GPU
(weak scaling, no data-path collective); rank 0 prints one JSON line.
``--impl reference`` times the fp64 CPU oracle on the host cores on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "C4 positions scored+top-k per sec and HBM GB/s (% of roofline), B=64 @128K"
UNIT = "positions/s"
KEY_BYTES_PER_POSITION = 128          # 64 bf16 dims of one C4 index key
FP8_KEY_BYTES_PER_POSITION = 68       # 64 e4m3 codes + one fp32 scale (fp8 key cache)
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20               # > 2x the 129 MB L2
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "scores_kernel_b64_ctx128k_dense.md")
PROFILE_SUMMARY_FP8 = os.path.join(ROOT, "profiles", "scores_fp8_kernel_b64_ctx128k_dense.md")
SCORES_SRC = os.path.join(ROOT, "sparse_attention_paged_dsa_gb300", "csrc", "scores_kernel.cu")
SCORES_FP8_SRC = os.path.join(ROOT, "sparse_attention_paged_dsa_gb300", "csrc", "scores_fp8_kernel.cu")
SCORES_COMMON_SRC = os.path.join(ROOT, "sparse_attention_paged_dsa_gb300", "csrc", "scores_common.cuh")
PTX_SRC = os.path.join(ROOT, "sparse_attention_paged_dsa_gb300", "csrc", "sm103_ptx.cuh")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="b64_ctx128k_dense")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-sample-rows", type=int, default=64,
                    help="rows of the workload the one-core CPU baseline times (a few seconds)")
    ap.add_argument("--reference-rows-per-step", type=int, default=0,
                    help="rows of the workload the reference arm (the oracle) scores per step (0: one per host core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context-scaling", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload table (all five workloads)")
    ap.add_argument("--no-fp8", action="store_true", help="skip the fp8 key-cache measurement")
    ap.add_argument("--no-mtp", action="store_true", help="skip the multi-token (next_n = 2, 4) measurement")
    ap.add_argument("--no-proj", action="store_true", help="skip the q/w projection measurement")
    ap.add_argument("--proj-d-model", type=int, default=7168, help="model width of the synthetic projection")
    ap.add_argument("--no-mla", action="store_true", help="skip the sparse-MLA decode measurement")
    ap.add_argument("--literal-pool", action="store_true",
                    help="dense workload on its literal 8192-page pool (each page in four rows): a small device "
                         "footprint for profiler captures, not for reported numbers")
    ap.add_argument("--l2-flush", action="store_true",
                    help="read a 512 MiB buffer (evicting L2) before every timed launch (default: back-to-back steps; "
                         "the live keys are twice the L2)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ ranks
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_units: float, local_seconds: float, group=None):
    """Whole-job units and the slowest rank's time (max over ranks)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return local_units, local_seconds
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    s = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(s, op=dist.ReduceOp.MAX, group=group)
    return float(u.item()), float(s.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        else:
            self.lines = []
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- helpers
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(summary, src):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged since."""
    try:
        text = open(summary).read()
    except OSError:
        return None
    h = hashlib.sha256()
    for f in (src, SCORES_COMMON_SRC, PTX_SRC):  # the kernel and the headers it is built from
        h.update(open(f, "rb").read())
    sha = h.hexdigest()
    fields = dict(l.split(":", 1) for l in text.splitlines() if l.startswith(("source_sha256:", "dram_bytes_per_launch:")))
    if fields.get("source_sha256", "").strip() != sha:
        return None
    try:
        return float(fields["dram_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


def host_cores():
    """Host cores this process may run on (read at run time)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rows(case, rows, threads):
    """The oracle as it stands (scores, then the full-sort top-k) on the given rows of a workload,
    one row per call, `threads` calls at a time.  The oracle keeps no state and ctypes releases the
    GIL during each call, so the calls run on `threads` host cores.  Returns (live positions, s)."""
    import concurrent.futures as cf
    from oracle import oracle
    from sparse_attention_paged_dsa_gb300.inputs import IndexerCase
    oracle.build()

    def one(b):
        sub = IndexerCase("row", case.q[b:b + 1], case.w[b:b + 1], case.key_pool, case.page_table[b:b + 1],
                          case.seq_lens[b:b + 1], case.max_context, case.k)
        oracle.case_topk(sub, oracle.case_scores(sub))
        return int(sub.live_positions().sum())

    t0 = time.perf_counter()
    if threads <= 1:
        pos = sum(one(b) for b in rows)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            pos = sum(ex.map(one, rows))
    return pos, time.perf_counter() - t0


def cpu_baseline(case, rows: int, min_wall_s: float = 0.75, max_passes: int = 8):
    """The fp64 oracle as it stands on the host's cores: all of them (one row per core at a time),
    repeated passes over every row of the workload until `min_wall_s` of wall time (about ten
    seconds of CPU work on 16 cores), and one core on the first `rows` rows."""
    cores = host_cores()
    pos_all, dt_all, passes = 0, 0.0, 0
    while passes < max_passes and (passes == 0 or dt_all < min_wall_s):
        pos, dt = oracle_rows(case, list(range(case.batch)), cores)
        pos_all, dt_all, passes = pos_all + pos, dt_all + dt, passes + 1
    rows = max(1, min(rows, case.batch))
    pos_one, dt_one = oracle_rows(case, list(range(rows)), 1)
    return {"value": pos_all / dt_all, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{passes} pass(es) over all {case.batch} rows ({pos_all} live positions), fp64 scores + "
                      f"full-sort top-k, one row per call on {cores} threads, {dt_all:.2f} s",
            "single_core": {"value": pos_one / dt_one, "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": f"first {rows} rows ({pos_one} live positions), {dt_one:.2f} s"}}


def evict_l2(buf):
    """Evict L2 by reading a buffer larger than it.  A read (not a memset) leaves the lines
    clean, so the next kernel's misses cost no write-backs of the flush's data."""
    import torch
    torch.amax(buf)


def device_preroll(stream):
    """Keep the device busy for about 100 us on `stream` (a spin kernel), so that the host has
    submitted the start event and the graph behind it before the device reaches them: the event
    pair then brackets the device's execution of the steps, not the host's graph submission."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        with torch.cuda.stream(stream):
            sleep(200_000)


def time_loop(fn, n, stream, flush=None):
    """CUDA-event time of `n` back-to-back calls of `fn` on `stream`.

    Without `flush`: the `n` calls are captured in one CUDA graph (a serving loop's
    form: no host launch cost between calls, consecutive launches overlap through
    programmatic dependent launch), replayed once untimed, then once between one
    event pair, behind a device pre-roll that keeps the host's graph submission out of
    the region; returns (mean seconds per call, None).  With `flush` (a callable
    that evicts L2): events around every call, the flush outside them; returns
    (mean, per-call list)."""
    import torch
    if flush is None:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        device_preroll(stream)
        e0.record(stream)
        with torch.cuda.stream(stream):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / n, None
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        flush()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) * 1e-3 for a, b in ev]
    return statistics.fmean(per), per


def per_call_events(fn, n, stream):
    """Per-call CUDA-event times (an event between calls; for percentiles only)."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in ev]


def graph_us_per_call(fn, reps=20, replays=20):
    """GPU time per call of `fn`: `reps` calls captured in one CUDA graph and replayed (no host launch cost)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        device_preroll(torch.cuda.current_stream())
        e0.record()
        g.replay()
        e1.record()
        times.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) * 1e3 / reps for a, b in times)


def context_scaling(binding, inputs, device):
    """Fused indexer without the full-width row on 64 requests of 512 tokens: max_context 1M vs 8K.

    The same requests (same keys, same page ids) are scored with a page table 4096 pages wide and
    one 32 pages wide; the ratio of GPU times is the cost of the larger fixed capture shape.
    """
    import torch
    big = inputs.workload("b64_ctx1m_seq512")
    small = inputs.IndexerCase("b64_ctx8k_seq512", big.q, big.w, big.key_pool,
                               big.page_table[:, :8192 // inputs.PAGE_TOKENS].copy(), big.seq_lens, 8192, big.k)
    out = {}
    for label, c in (("1m", big), ("8k", small)):
        q, w, pool, table, seq = binding.to_device(c, device)
        ws = binding.new_workspace(c.batch, c.max_context, c.k, device)
        topk = torch.empty((c.batch, c.k), dtype=torch.int32, device=device)
        out[label] = graph_us_per_call(lambda: binding.dsa_indexer_fused(q, w, pool, table, seq, c.max_context, c.k,
                                                                         topk_idx=topk, workspace=ws))
        if binding.get_error(ws) != 0:
            raise RuntimeError("device error word set in the context-scaling run")
    return {"t_fused_no_row_1m_us": out["1m"], "t_fused_no_row_8k_us": out["8k"],
            "ratio_1m_over_8k": out["1m"] / out["8k"],
            "workload": "64 requests x 512 tokens, k=2048, same keys and page ids; CUDA-graph replay"}


CONFIG_WORKLOADS = ["b1_ctx8k_seq512", "b16_ctx8k_mixed", "b64_ctx128k_loguniform", "b64_ctx1m_seq512",
                    "b64_ctx128k_dense"]


def run_configs(args, binding, inputs, device, stream, main_case, main_dev):
    """Every named workload through the three call shapes: the fused call with the full-width scores
    row, the fused call without it (live scores in the workspace), and the scores entry point alone.
    Each is timed twice: warm (20 calls captured in one CUDA graph, median of 20 replays: back to back,
    as in a decode loop) and with L2 evicted before every call (a 512 MiB read outside the events,
    median of 30 isolated calls).  Every warm timing runs before any eviction: the keys are loaded
    evict-first, so after a flush the flush buffer's lines would keep them out of L2 and a "warm"
    loop that follows one is not back to back."""
    import torch
    peak, peak_kind = measured_hbm_peak()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    out = {"timing": "warm: CUDA-graph replay of 20 calls, median of 20; l2_evicted: CUDA events around each of "
                     "30 calls, a 512 MiB read before each (outside the events), median",
           "peak_gbs": peak, "peak_kind": f"{peak_kind} (HBM copy bandwidth)"}

    deferred = []  # (result dict, call): the evicted timings, run after every warm one
    workspaces = []

    def time_both(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        res = {"warm": graph_us_per_call(fn)}
        deferred.append((res, fn))
        return res

    for name in CONFIG_WORKLOADS:
        case = main_case if name == main_case.name else inputs.workload(name)
        q, w, pool, table, seq = main_dev if case is main_case else binding.to_device(case, device)
        B, M, K = case.batch, case.max_context // 4, case.k
        live = int(case.live_positions().sum())
        scores = torch.empty((B, M), dtype=torch.float32, device=device)
        topk = torch.empty((B, K), dtype=torch.int32, device=device)
        ws = binding.new_workspace(B, case.max_context, K, device)
        # (partial binds this workload's tensors: the evicted timings run after the loop)
        fused_row = time_both(functools.partial(binding.dsa_indexer_fused, q, w, pool, table, seq, case.max_context,
                                                K, topk_idx=topk, scores=scores, workspace=ws))
        fused_no_row = time_both(functools.partial(binding.dsa_indexer_fused, q, w, pool, table, seq,
                                                   case.max_context, K, topk_idx=topk, workspace=ws))
        scores_only = time_both(functools.partial(binding.dsa_indexer_scores, q, w, pool, table, seq,
                                                  case.max_context, scores=scores, workspace=ws))
        workspaces.append((name, ws))
        key_bytes = live * KEY_BYTES_PER_POSITION
        entry = {
            "batch": B, "max_context": case.max_context, "k": K, "live_positions": live, "live_key_bytes": key_bytes,
            "fused_row_us": fused_row, "fused_no_row_us": fused_no_row, "scores_us": scores_only,
            "scores_row_bytes": B * M * 4,
        }
        if name == "b64_ctx1m_seq512":
            # The scores entry point writes the whole [B, max_context / 4] row: its -inf fill at this
            # width against the same requests at an 8K width (same keys and page ids).
            small = inputs.IndexerCase("b64_ctx8k_seq512", case.q, case.w, case.key_pool,
                                       case.page_table[:, :8192 // inputs.PAGE_TOKENS].copy(), case.seq_lens,
                                       8192, case.k)
            q8, w8, pool8, table8, seq8 = binding.to_device(small, device)
            scores8 = torch.empty((B, 8192 // 4), dtype=torch.float32, device=device)
            ws8 = binding.new_workspace(B, 8192, K, device)
            s8 = time_both(functools.partial(binding.dsa_indexer_scores, q8, w8, pool8, table8, seq8, 8192,
                                             scores=scores8, workspace=ws8))
            workspaces.append((name + " at 8K width", ws8))
            entry["scores_api_fill"] = {
                "width_1m": {"row_bytes": B * M * 4, "us": scores_only},
                "width_8k": {"row_bytes": B * 2048 * 4, "us": s8},
                "note": "the scores entry point is O(max_context) by contract (it writes the full-width row); "
                        "the O(live) bound is the fused call without a row (context_scaling)"}
        out[name] = entry
    for res, fn in deferred:  # the evicted timings (the warm ones are all done)
        _, per = time_loop(fn, 30, stream, lambda: evict_l2(flush))
        res["l2_evicted"] = 1e6 * statistics.median(per)
    for name, ws in workspaces:
        if binding.get_error(ws) != 0:
            raise RuntimeError(f"device error word set in the {name} run")
    for name in CONFIG_WORKLOADS:  # the ratios that need both timings
        e = out[name]
        key_bytes = e["live_key_bytes"]
        gbs = lambda us: key_bytes / (us * 1e-6) / 1e9
        e["positions_per_s"] = {t: e["live_positions"] / (e["fused_row_us"][t] * 1e-6) for t in ("warm", "l2_evicted")}
        e["step_gbs"] = {t: gbs(e["fused_row_us"][t]) for t in ("warm", "l2_evicted")}
        e["step_frac"] = {t: gbs(e["fused_row_us"][t]) / peak for t in ("warm", "l2_evicted")}
        e["scores_kernel_frac"] = {t: gbs(e["scores_us"][t]) / peak for t in ("warm", "l2_evicted")}
        e["fused_over_scores"] = {t: e["fused_row_us"][t] / e["scores_us"][t] for t in ("warm", "l2_evicted")}
        fill = e.get("scores_api_fill")
        if fill:
            for w in ("width_1m", "width_8k"):
                fill[w]["row_gbs"] = {t: fill[w]["row_bytes"] / (fill[w]["us"][t] * 1e-6) / 1e9 for t in fill[w]["us"]}
            fill["ratio_1m_over_8k"] = {t: fill["width_1m"]["us"][t] / fill["width_8k"]["us"][t]
                                        for t in ("warm", "l2_evicted")}
    del flush
    return out


def run_fp8(args, case, binding, inputs, device, stream, live):
    """The same workload on the fp8 key cache: fused step (events, back-to-back) and scores kernel alone."""
    import torch
    f = inputs.with_fp8_keys(case)
    q, w, _, table, seq = binding.to_device(f, device)
    codes, scales = binding.to_device_fp8(f, device)
    B, M, K = f.batch, f.max_context // 4, f.k
    scores = torch.empty((B, M), dtype=torch.float32, device=device)
    topk = torch.empty((B, K), dtype=torch.int32, device=device)
    ws = binding.new_workspace(B, f.max_context, K, device)

    def step():
        binding.dsa_indexer_fused_fp8(q, w, codes, scales, table, seq, f.max_context, K, topk_idx=topk,
                                      scores=scores, workspace=ws)

    def scores_only():
        binding.dsa_indexer_scores_fp8(q, w, codes, scales, table, seq, f.max_context, scores=scores, workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
        scores_only()
    torch.cuda.synchronize(device)
    # Secondary legs are timed by CUDA-graph replay (one launch sequence per replay, no host in the
    # loop), so that a busy host late in the run cannot inflate them; the back-to-back loop of the main
    # leg's form is reported too.
    t_step = graph_us_per_call(step) * 1e-6
    t_scores = graph_us_per_call(scores_only) * 1e-6
    n = max(10, min(args.steps, 500))
    t_step_loop, _ = time_loop(step, n, stream)
    # The codes and scales (142 MB) are about the size of L2: also time isolated launches of the
    # scores kernel with L2 evicted before each, so that no key of the previous call is in L2.
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    t_scores_cold, _ = time_loop(scores_only, 50, stream, lambda: evict_l2(flush))
    del flush
    if binding.get_error(ws) != 0:
        raise RuntimeError("device error word set in the fp8 run")
    peak, peak_kind = measured_hbm_peak()
    traffic = profiled_traffic(PROFILE_SUMMARY_FP8, SCORES_FP8_SRC)
    achieved = live * FP8_KEY_BYTES_PER_POSITION / t_scores / 1e9
    return {"value": live / t_step, "unit": UNIT, "ms_per_step": 1e3 * t_step,
            "scores_kernel_us": 1e6 * t_scores, "timing": "CUDA-graph replay, 20 calls per graph, median of 20",
            "back_to_back_ms_per_step": 1e3 * t_step_loop, "back_to_back_steps": n,
            "scores_kernel_us_l2_flushed": 1e6 * t_scores_cold,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "kernel": "scores_fp8_kernel",
                         "peak_kind": f"{peak_kind} (HBM copy bandwidth)",
                         "algorithmic_bytes_per_launch": live * FP8_KEY_BYTES_PER_POSITION,
                         "l2_share_back_to_back": 0.06,
                         "note": "back to back about 6 % of the 142.6 MB are still in L2 (ncu without cache "
                                 "control: 134 MB from DRAM per launch); scores_kernel_us_l2_flushed times isolated "
                                 "launches after an L2 eviction"},
            "cache": "e4m3 codes [pages, 64, 64] + fp32 scale per key (max|k| / 448), made from the bf16 keys",
            "step": "dsa_indexer_fused_fp8 with the full-width scores row"}


def run_mtp(args, case, binding, inputs, device, stream, live, pool, table, seq):
    """The same workload with next_n query tokens per request (keys read once for all tokens)."""
    import torch
    out = {}
    peak, peak_kind = measured_hbm_peak()
    for Q in (2, 4):
        c = inputs.with_next_n(case, Q)
        q = torch.from_numpy(c.q.view("int16")).to(device).view(torch.bfloat16)
        w = torch.from_numpy(c.w).to(device)
        B, M, K = c.batch, c.max_context // 4, c.k
        scores = torch.empty((B, Q, M), dtype=torch.float32, device=device)
        topk = torch.empty((B, Q, K), dtype=torch.int32, device=device)
        ws = torch.zeros(binding.workspace_size_mtp(B, Q, c.max_context, K), dtype=torch.uint8, device=device)

        def step():
            binding.dsa_indexer_fused_mtp(q, w, pool, table, seq, c.max_context, K, topk_idx=topk, scores=scores,
                                          workspace=ws)

        def scores_only():
            binding.dsa_indexer_scores_mtp(q, w, pool, table, seq, c.max_context, scores=scores, workspace=ws)

        for _ in range(max(3, args.warmup)):
            step()
            scores_only()
        torch.cuda.synchronize(device)
        t_step = graph_us_per_call(step) * 1e-6
        t_scores = graph_us_per_call(scores_only) * 1e-6
        if binding.get_error(ws) != 0:
            raise RuntimeError("device error word set in the multi-token run")
        tok_positions = sum((max(int(L) - (Q - 1 - j), 0) + 3) // 4 for L in c.seq_lens for j in range(Q))
        achieved = live * KEY_BYTES_PER_POSITION / t_scores / 1e9
        out[str(Q)] = {"value": tok_positions / t_step, "unit": "token-positions/s", "ms_per_step": 1e3 * t_step,
                       "scores_kernel_us": 1e6 * t_scores,
                       "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                                    "frac": achieved / peak, "peak_kind": f"{peak_kind} (HBM copy bandwidth)",
                                    "algorithmic_bytes_per_launch": live * KEY_BYTES_PER_POSITION}}
    out["step"] = ("dsa_indexer_fused_mtp with full-width rows: next_n query tokens per request, token j "
                   "scores its causal prefix of seq_len - (next_n - 1 - j) tokens; keys read once")
    out["timing"] = "CUDA-graph replay, 20 calls per graph, median of 20"
    return out


def run_proj(args, binding, device, batch):
    """q/w projection from a bf16 hidden state [batch, d] with synthetic weights (the pages give no shapes)."""
    import torch
    d = args.proj_d_model
    g = torch.Generator(device="cpu").manual_seed(4242)
    x = torch.randn((batch, d), generator=g).to(torch.bfloat16).to(device)
    wq = (torch.randn((2048, d), generator=g) / d ** 0.5).to(torch.bfloat16).to(device)
    ww = (torch.randn((32, d), generator=g) / d ** 0.5).to(torch.bfloat16).to(device)
    q = torch.empty((batch, 32, 64), dtype=torch.bfloat16, device=device)
    w = torch.empty((batch, 32), dtype=torch.float32, device=device)
    ws = torch.zeros(binding.qw_proj_workspace_size(batch, d), dtype=torch.uint8, device=device)
    fn = lambda: binding.dsa_indexer_qw_proj(x, wq, ww, q_out=q, w_out=w, workspace=ws)
    for _ in range(5):
        fn()
    # The weights (30 MB at d = 7168) fit in L2; a model's layers each bring their own, so every
    # timed call starts with L2 evicted (a 512 MiB read, outside the events).
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    t, _ = time_loop(fn, 50, stream, lambda: evict_l2(flush))
    t_warm = graph_us_per_call(fn) * 1e-6
    if binding.get_error(ws) != 0:
        raise RuntimeError("device error word set in the projection run")
    wbytes = (2048 + 32) * d * 2
    peak, peak_kind = measured_hbm_peak()
    achieved = wbytes / t / 1e9
    return {"value": batch / t, "unit": "tokens/s", "us_per_call": 1e6 * t, "batch": batch, "d_model": d,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "kernel": "proj_kernel", "peak_kind": f"{peak_kind} (HBM copy bandwidth)",
                         "algorithmic_bytes_per_launch": wbytes},
            "timing": "CUDA events around each of 50 calls, L2 evicted before each by a 512 MiB read (weights from HBM)",
            "us_per_call_l2_warm": 1e6 * t_warm,
            "weights": "synthetic N(0, 1/d) bf16: w_q [2048, d], w_w [32, d]; x N(0,1) bf16"}


def run_mla(args, case, binding, device, topk, step):
    """Sparse-MLA decode (64 heads, 576-wide entries) over the indexer's own top-k rows of the
    workload, on a synthetic cache with one 64-entry page per index-key page; also the indexer
    step and the attention chained in one graph."""
    import torch
    g = torch.Generator(device=device).manual_seed(4343)
    heads, dim, dv = binding.MLA_HEADS, binding.MLA_DIM, binding.MLA_DV
    q = torch.randn((case.batch, heads, dim), generator=g, device=device).to(torch.bfloat16)
    kv = torch.empty((case.num_pages, 64, dim), dtype=torch.bfloat16, device=device)
    for p0 in range(0, case.num_pages, 4096):  # N(0, 1) in slices (bounded temporary memory)
        p1 = min(case.num_pages, p0 + 4096)
        kv[p0:p1] = torch.randn((p1 - p0, 64, dim), generator=g, device=device).to(torch.bfloat16)
    table = torch.from_numpy(case.page_table).to(device)
    seq = torch.from_numpy(case.seq_lens).to(device)
    out = torch.empty((case.batch, heads, dv), dtype=torch.float32, device=device)
    lse = torch.empty((case.batch, heads), dtype=torch.float32, device=device)
    ws = torch.zeros(binding.sparse_mla_workspace_size(case.batch, case.k), dtype=torch.uint8, device=device)
    scale = dim ** -0.5
    step()  # the indexer's top-k rows of this workload
    torch.cuda.synchronize(device)
    used = int((topk >= 0).sum().item())

    def attn():
        binding.dsa_sparse_mla_decode(q, kv, table, seq, case.max_context, topk, scale, out=out, lse=lse,
                                      workspace=ws)

    def chained():
        step()
        attn()

    for _ in range(max(3, args.warmup)):
        attn()
    torch.cuda.synchronize(device)
    t = graph_us_per_call(attn) * 1e-6
    t_chain = graph_us_per_call(chained) * 1e-6
    if binding.get_error(ws) != 0:
        raise RuntimeError("device error word set in the sparse-MLA run")
    splits = max(1, min(32, (case.k + 63) // 64, torch.cuda.get_device_properties(device).multi_processor_count
                        // case.batch))
    algo = used * dim * 2 + q.numel() * 2 + out.numel() * 4 + lse.numel() * 4
    peak, peak_kind = measured_hbm_peak()
    achieved = algo / t / 1e9
    return {"value": case.batch / t, "unit": "requests/s", "us_per_call": 1e6 * t,
            "entries_per_s": used / t, "used_entries": used, "splits_per_request": splits,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "kernel": "mla_decode_kernel + mla_merge_kernel",
                         "peak_kind": f"{peak_kind} (HBM copy bandwidth)", "algorithmic_bytes_per_launch": algo,
                         "bytes": "used entries x 1152 B + q + o + lse (split partials not counted)"},
            "indexer_plus_mla_us": 1e6 * t_chain,
            "timing": "CUDA-graph replay, 20 calls per graph, median of 20",
            "inputs": "64 heads, 576-dim bf16 q and cache ~ N(0,1) (torch generator on the device), "
                      "one cache page per index-key page; top-k rows from this workload's indexer step; "
                      "sm_scale 576^-1/2"}


def workload_config(case, world, l2_flush=False):
    live = int(case.live_positions().sum())
    return {"workload": case.name, "batch": case.batch, "max_context": case.max_context,
            "seq_len": int(case.seq_lens.max()), "k": case.k, "pool_pages": case.num_pages,
            "live_positions": live, "live_key_bytes": live * KEY_BYTES_PER_POSITION,
            "l2": ("evicted before every timed launch (512 MiB read, outside the events)" if l2_flush else
                   "not flushed: back-to-back steps, live keys 268 MB = 2x the 129 MB L2 (DRAM bytes per "
                   "launch = algorithmic, ncu with --cache-control none)"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ----------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from sparse_attention_paged_dsa_gb300 import inputs
    case = inputs.workload(args.workload)
    cores = host_cores()
    r = max(1, min(args.reference_rows_per_step or cores, case.batch))

    def step(i):  # r rows of the workload, one per host core at a time
        b0 = (i * r) % case.batch
        return oracle_rows(case, [(b0 + j) % case.batch for j in range(r)], min(r, cores))[0]

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    pos = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    value = pos / dt
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(case, 1), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(r, cores), "kind": "oracle",
                             "sample": f"{r} rows of {case.batch} per step (fp64 oracle, one row per call on "
                                       f"{min(r, cores)} host threads)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)

    from sparse_attention_paged_dsa_gb300 import binding, inputs
    binding.load()
    case = inputs.workload(args.workload, literal_pool=args.literal_pool)
    B, M, K = case.batch, case.max_context // 4, case.k
    live = int(case.live_positions().sum())

    q, w, pool, table, seq = binding.to_device(case, device)
    scores = torch.empty((B, M), dtype=torch.float32, device=device)
    topk = torch.empty((B, K), dtype=torch.int32, device=device)
    ws = binding.new_workspace(B, case.max_context, K, device)
    flush = torch.empty(FLUSH_BYTES if args.l2_flush else 1, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        binding.dsa_indexer_fused(q, w, pool, table, seq, case.max_context, K, topk_idx=topk, scores=scores,
                                  workspace=ws)

    def scores_only():
        binding.dsa_indexer_scores(q, w, pool, table, seq, case.max_context, scores=scores, workspace=ws)

    def maybe_flush():
        if args.l2_flush:
            evict_l2(flush)

    for _ in range(max(3, args.warmup)):
        maybe_flush()
        step()
        maybe_flush()
        scores_only()
    torch.cuda.synchronize(device)
    if binding.get_error(ws) != 0:
        raise RuntimeError("device error word set during warm-up")

    n = args.steps
    flush_fn = (lambda: evict_l2(flush)) if args.l2_flush else None
    with ClockSampler(device.index) as clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)
        clocks.mark_start()
        wall0 = time.perf_counter()
        mean_step, per_step = time_loop(step, n, stream, flush_fn)
        if world > 1:
            dist.barrier()
        wall1 = time.perf_counter()
        clocks.mark_end()
    total_units, max_seconds = aggregate(live * n, mean_step * n)
    value = total_units / max_seconds
    if per_step is None:  # percentiles from a separate loop with an event between steps
        per_step = per_call_events(step, max(10, min(n, 200)), stream)

    # The dominant kernel alone: the scores entry point launches the same scores kernel the fused call
    # launches first; same workload, same L2 setting between launches.
    n_k = max(200, min(n, 500))  # enough launches to amortise the one graph launch
    mean_scores, per_scores = time_loop(scores_only, n_k, stream, flush_fn)
    if per_scores is None:
        per_scores = per_call_events(scores_only, max(10, min(n, 200)), stream)
    if binding.get_error(ws) != 0:
        raise RuntimeError("device error word set during the timed steps")

    # e2e: the step's host (pinned) inputs -> device, both kernels, top-k back to the host, every
    # step (key cache resident); beside it, the same with the whole key pool copied every step.
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, case, binding, scores, topk, ws, device, stream, world, live)
        e2e["with_key_pool_copied"] = run_e2e(args, case, binding, scores, topk, ws, device, stream, world, live,
                                              cache_copied=True)

    scaling_1m = context_scaling(binding, inputs, device) if not args.no_context_scaling else None
    configs = (run_configs(args, binding, inputs, device, stream, case, (q, w, pool, table, seq))
               if not args.no_configs else None)
    fp8 = run_fp8(args, case, binding, inputs, device, stream, live) if not args.no_fp8 else None
    mtp = (run_mtp(args, case, binding, inputs, device, stream, live, pool, table, seq)
           if not args.no_mtp else None)
    proj = run_proj(args, binding, device, case.batch) if not args.no_proj else None
    mla = run_mla(args, case, binding, device, topk, step) if not args.no_mla else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, args.cpu_sample_rows)

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0

    peak, peak_kind = measured_hbm_peak()
    achieved = live * KEY_BYTES_PER_POSITION / mean_scores / 1e9
    traffic = profiled_traffic(PROFILE_SUMMARY, SCORES_SRC)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n, "warmup": args.warmup,
        "ms_per_step": 1e3 * mean_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(case, world, args.l2_flush),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "kernel": "scores_kernel",
                     "peak_kind": f"{peak_kind} (HBM copy bandwidth)",
                     "algorithmic_bytes_per_launch": live * KEY_BYTES_PER_POSITION},
        "kernels_us": {"scores_mean": 1e6 * mean_scores,
                       "scores_median_with_events_between": 1e6 * statistics.median(per_scores),
                       "scores_launches_timed": n_k,
                       "step_p10": 1e6 * float(np.percentile(per_step, 10)),
                       "step_p50": 1e6 * float(np.percentile(per_step, 50)),
                       "step_p90": 1e6 * float(np.percentile(per_step, 90)),
                       "percentiles": "per-step events" + ("" if args.l2_flush else
                                                           " (separate loop, an event between steps)")},
        "step_gbs_live_keys": live * KEY_BYTES_PER_POSITION / mean_step / 1e9,
        "timing": ("events around every step, L2 flushed outside them" if args.l2_flush else
                   "the K back-to-back steps captured in one CUDA graph, one replay between one CUDA-event pair (a ~100 us device spin before the start event keeps the host's graph submission out of the region)"),
        "cpu_baseline": cpu,
        "context_scaling": scaling_1m,
        "configs": configs,
        "fp8_key_cache": fp8,
        "multi_token": mtp,
        "qw_projection": proj,
        "sparse_mla_decode": mla,
        "e2e": e2e,
        "gpu_launches": 2 * n * world,
        "step": "dsa_indexer_fused with the full-width scores row (scores kernel, then top-k kernel)",
        "clocks": clocks.summary(),
        "wall_s_timed_region": wall1 - wall0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(args, case, binding, scores, topk, ws, device, stream, world, live, cache_copied=False):
    """The same step through the C ABI with host buffers: H2D of the step's inputs from pinned memory,
    the fused call, D2H of the top-k, all inside the timed region.  The step's inputs are the query,
    head weights, page table and lengths, staged as one pinned buffer (256-byte aligned pieces) and
    copied in with one transfer, the way a serving loop stages a step; the call takes device views of
    the pieces.  The paged key cache is the model's resident state (a decode step appends one C4 key
    per 4 tokens per request, 64 B-256 B, not modelled) and is uploaded once before the timed region.
    With cache_copied the whole key pool is copied every step as well (a second transfer)."""
    import torch
    import torch.distributed as dist
    B, K = case.batch, case.k
    pieces = [torch.from_numpy(np.ascontiguousarray(a))
              for a in (case.q.view("int16"), case.w, case.page_table, case.seq_lens)]
    offs, total = [], 0
    for t in pieces:
        offs.append(total)
        total = (total + t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(pieces, offs):
        n = t.numel() * t.element_size()
        host[o:o + n].copy_(t.view(torch.uint8).reshape(-1))
    dev = torch.empty(total, dtype=torch.uint8, device=device)
    qd, wd, td, sd = (dev[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                      for t, o in zip(pieces, offs))
    pool_host = torch.from_numpy(case.key_pool.view("int16")).pin_memory()
    pd = torch.empty(pool_host.shape, dtype=pool_host.dtype, device=device)
    pd.copy_(pool_host)
    out_host = torch.empty((B, K), dtype=torch.int32).pin_memory()
    h2d = total + (pool_host.numel() * pool_host.element_size() if cache_copied else 0)
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        dev.copy_(host, non_blocking=True)
        if cache_copied:
            pd.copy_(pool_host, non_blocking=True)
        binding.dsa_indexer_fused(qd.view(torch.bfloat16), wd, pd.view(torch.bfloat16), td, sd,
                                  case.max_context, K, topk_idx=topk, scores=scores, workspace=ws)
        out_host.copy_(topk, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_units, e2e_seconds = aggregate(live * args.e2e_steps, e0.elapsed_time(e1) * 1e-3)
    if not np.array_equal(out_host.numpy(), topk.cpu().numpy()):
        raise RuntimeError("e2e top-k read-back mismatch")
    return {"value": e2e_units / e2e_seconds, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "inputs": "q, w, page table, seq_lens every step, staged as one pinned buffer and one copy"
                      + (", and the whole key pool" if cache_copied else "; key cache resident")}


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
