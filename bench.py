"""Benchmark: two-phase Block AttnRes throughput on GB300.

Default workload (the headline metric): one block of the two-phase Block
scheme over 9 cached block summaries [B=8, T=4096, D=4096] bf16 with S = 24
sublayer queries -- phase 1 batched, then 23 phase-2 merges, each sublayer
followed by the running-partial update with the synthetic sublayer
f(h) = 0.5 tanh(u h).  One step = one such block pass over all B*T tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload NAME] [--rows R]

Prints one JSON line (rank 0).  Multi-GPU (torchrun): every rank runs the
same per-GPU workload on its own token rows (no data-path collective);
value = all ranks' tokens / max-over-ranks time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from transformer_depth_wise_gb300 import accounting  # noqa: E402
from transformer_depth_wise_gb300 import workloads as wk  # noqa: E402

METRIC = "Block AttnRes tokens/s and achieved HBM GB/s (% of GB300 peak), two-phase path"
FALLBACK_HBM_GBS = 6800.0
# GB300's nominal HBM3e bandwidth.  Every fraction is reported against both
# denominators: `frac` against the measured copy bandwidth (the roofline
# peak), `frac_nominal` against this figure (the >= 80 % target's "~8 TB/s").
NOMINAL_HBM_GBS = 8000.0


# ---------------------------------------------------------------------------
# process group / timing helpers
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            j = json.load(fh)
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_traffic(kernel: str, workload: str, rows: int):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is
    unchanged.  A summary captured on fewer token rows than the workload's (to keep
    the capture small) is scaled by rows: these kernels stream every row once."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.txt")
    src = {"phase1": "phase1_tc.cu", "merge": "merge.cu", "merge_update": "merge.cu", "update": "merge.cu",
           "aggregate": "aggregate.cu"}.get(kernel)
    if not src or not os.path.exists(path):
        return None
    info = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            info[k.strip()] = v.strip()
    with open(os.path.join(ROOT, "transformer_depth_wise_gb300", "csrc", src), "rb") as fh:
        sha = hashlib.sha256(fh.read()).hexdigest()
    if info.get("source_sha256") != sha:
        return None
    try:
        per_launch = float(info["traffic_bytes_per_launch"])
        captured = int(info.get("rows_captured", rows))
    except (KeyError, ValueError):
        return None
    return round(per_launch * rows / captured)


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_block_rows_per_s(wl, rows_target_s: float = 12.0, max_rows: int = 4096):
    """Time the oracle's two-phase block chain on a bounded sample of token rows."""
    import numpy as np
    import oracle
    inp = wk.two_phase_inputs(wl, rows=256, device="cpu")
    blocks = [b.reshape(-1, wl.D).double().numpy() for b in inp["blocks"]]
    W, G, U = (inp["queries"].double().numpy(), inp["gains"].double().numpy(),
               inp["u"].double().numpy())
    t0 = time.perf_counter()
    oracle.block_two_phase_chain([b[:8] for b in blocks], W, G, U, inp["eps"], oracle.BF16)
    per_row = (time.perf_counter() - t0) / 8
    rows = int(min(max_rows, max(16, rows_target_s / max(per_row, 1e-6))))
    rows = min(rows, 256)
    reps = max(1, int(rows_target_s / max(per_row * rows, 1e-6)))
    reps = min(reps, 64)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.block_two_phase_chain([b[:rows] for b in blocks], W, G, U, inp["eps"], oracle.BF16)
    dt = time.perf_counter() - t0
    sample = f"{reps} x {rows} token rows of the {wl.name} block chain (phase 1 + {wl.S - 1} merges + {wl.S} updates), fp64 oracle, 1 thread"
    return reps * rows / dt, dt, sample


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
EVENT_EVERY = 5  # per-kernel events on one block pass in five


def time_block(blk, K, dev, world, stream, fused, label="timed"):
    """Run K block passes, every EVENT_EVERY-th with per-kernel events; returns (elapsed max over ranks,
    events of the instrumented passes, clocks).  An event recorded between two dependent launches keeps the
    second from starting early, so instrumenting every pass would add about 2 % to the step; the per-kernel
    averages come from the instrumented passes inside the same timed region.  The passes sit in an NVTX
    range named `label`, which a profiler can select."""
    S = blk.S
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    events = [{"phase1": (ev(), ev()), "merge": [(ev(), ev()) for _ in range(S - 1)],
               "update": [(ev(), ev()) for _ in range(1 if fused else S)]}
              for k in range(K) if k % EVENT_EVERY == 0]
    t_start, t_end = ev(), ev()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.nvtx.range_push(label)
    t_start.record(stream)
    for k in range(K):
        blk.run(events=events[k // EVENT_EVERY] if k % EVENT_EVERY == 0 else None)
    t_end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(world)
    return max_over_ranks(t_start.elapsed_time(t_end), world, dev), events, clk


def time_passes(run, K, dev, world, stream, label):
    """K back-to-back block passes without per-kernel events (elapsed ms, max over ranks)."""
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    torch.cuda.nvtx.range_push(label)
    t_start.record(stream)
    for _ in range(K):
        run()
    t_end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    barrier(world)
    return max_over_ranks(t_start.elapsed_time(t_end), world, dev)


def run_two_phase(args, wl, dev, rank, world):
    from transformer_depth_wise_gb300 import api
    if args.rows:
        wl = wk.Workload(wl.name, 1, args.rows, wl.D, wl.n, wl.dtype, wl.scale_lo, wl.scale_hi,
                         S=wl.S, seed=wl.seed)
    n_blocks = wl.n if wl.name == "two_phase_bf16" else wl.n - 1
    inp = wk.two_phase_inputs(wl, device=dev, n=n_blocks)
    stream = torch.cuda.current_stream(dev)
    rows, D, S, elt = wl.B * wl.T, wl.D, wl.S, 2
    K = args.steps

    blk = api.TwoPhaseBlock(inp["blocks"], inp["queries"], inp["gains"], inp["u"], inp["eps"], fused=True)
    for _ in range(args.warmup):
        blk.run()
    torch.cuda.synchronize(dev)
    elapsed_ms, events, clk = time_block(blk, K, dev, world, stream, fused=True)

    p1 = [e["phase1"][0].elapsed_time(e["phase1"][1]) for e in events]
    mg = [a.elapsed_time(b) for e in events for a, b in e["merge"]]
    up = [a.elapsed_time(b) for e in events for a, b in e["update"]]
    b = accounting.two_phase_block_bytes(n_blocks, S, rows, D, elt, fused=True)
    kern = {
        "phase1": {"launches": K, "avg_ms": statistics.mean(p1), "bytes": b["phase1"]},
        "merge_update": {"launches": K * (S - 1), "avg_ms": statistics.mean(mg),
                         "bytes": b["merges"] / (S - 1)},
        "update": {"launches": K, "avg_ms": statistics.mean(up), "bytes": b["updates"]},
    }
    peak, peak_src = measured_peak()
    for name, k in kern.items():
        k["total_ms"] = k["avg_ms"] * k["launches"]
        k["gbs"] = k["bytes"] / (k["avg_ms"] * 1e-3) / 1e9
        k["frac"] = k["gbs"] / peak
        k["frac_nominal"] = k["gbs"] / NOMINAL_HBM_GBS
    dom = max(kern, key=lambda n: kern[n]["total_ms"])
    d = kern[dom]
    traffic = kernel_traffic(dom, wl.name, rows)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(d["gbs"], 1), "peak": peak,
                "unit": "GB/s", "frac": round(d["frac"], 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": d["bytes"],
                "peak_source": peak_src + " hbm_gbs (copy bandwidth)",
                "frac_nominal": round(d["gbs"] / NOMINAL_HBM_GBS, 4),
                "nominal_peak": NOMINAL_HBM_GBS}

    tokens = rows * K * world
    value = tokens / (elapsed_ms * 1e-3)
    launches_per_step = blk.launches_per_run

    # The same block pass without the fused update+merge, for comparison.
    blk_u = api.TwoPhaseBlock(inp["blocks"], inp["queries"], inp["gains"], inp["u"], inp["eps"],
                              fused=False)
    for _ in range(args.warmup):
        blk_u.run()
    torch.cuda.synchronize(dev)
    el_u, ev_u, _ = time_block(blk_u, K, dev, world, stream, fused=False, label="timed_unfused")
    bu = accounting.two_phase_block_bytes(n_blocks, S, rows, D, elt, fused=False)
    mg_u = [a.elapsed_time(c) for e in ev_u for a, c in e["merge"]]
    up_u = [a.elapsed_time(c) for e in ev_u for a, c in e["update"]]
    unfused = {"value": round(rows * K * world / (el_u * 1e-3), 1), "ms_per_step": round(el_u / K, 4),
               "merge_gbs": round(bu["merges"] / (S - 1) / (statistics.mean(mg_u) * 1e-3) / 1e9, 1),
               "update_gbs": round(bu["updates"] / S / (statistics.mean(up_u) * 1e-3) / 1e9, 1),
               "launches_per_step": blk_u.launches_per_run}
    del blk_u

    # The fused pass with each sublayer's pre-norm formed inside the
    # update+merge (norm weights drawn like the gains), for comparison.
    nw = wk.queries_and_gains(wk.generator(wl.seed + 7, dev), S, D, dev)[1]
    blk_n = api.TwoPhaseBlock(inp["blocks"], inp["queries"], inp["gains"], inp["u"], inp["eps"],
                              fused=True, norm_weights=nw, norm_eps=1e-6)
    for _ in range(args.warmup):
        blk_n.run()
    torch.cuda.synchronize(dev)
    el_n, ev_n, _ = time_block(blk_n, K, dev, world, stream, fused=True, label="timed_prenorm")
    mg_n = [a.elapsed_time(c) for e in ev_n for a, c in e["merge"]]
    prenorm = {"value": round(rows * K * world / (el_n * 1e-3), 1), "ms_per_step": round(el_n / K, 4),
               "merge_update_ms": round(statistics.mean(mg_n), 5),
               "launches_per_step": blk_n.launches_per_run,
               "step": "as the headline, each sublayer reading rms_norm(h) (.) w_n formed in the same pass"}
    del blk_n, nw

    # The same block pass with the batch's sequences in two groups on two
    # streams (TwoPhaseBlock(groups=2)): one group's phase-1 scores overlap
    # the other's outputs kernel; the values are bitwise those of one pass.
    groups = None
    if wl.B % 2 == 0:
        blk_g = api.TwoPhaseBlock(inp["blocks"], inp["queries"], inp["gains"], inp["u"], inp["eps"], fused=True,
                                  groups=2)
        for _ in range(args.warmup):
            blk_g.run()
        torch.cuda.synchronize(dev)
        el_g = time_passes(blk_g.run, K, dev, world, stream, "timed_groups")
        groups = {"groups": 2, "value": round(rows * K * world / (el_g * 1e-3), 1),
                  "ms_per_step": round(el_g / K, 4),
                  "frac_step": round(b["total"] / (el_g / K * 1e-3) / 1e9 / peak, 4),
                  "launches_per_step": blk_g.launches_per_run,
                  "step": "as the headline, the batch's sequences in two groups of B/2 on two streams"}
        del blk_g

    # End to end through the public API: pinned host inputs -> device, block
    # pass, final partial (the new block summary) -> pinned host, every step.
    e2e = run_two_phase_e2e(args, wl, dev, inp, n_blocks, world)
    headline = wl.name == "two_phase_bf16" and not args.rows
    del blk, inp
    torch.cuda.empty_cache()
    decode = run_decode(dev) if headline else None
    backward = run_backward(dev) if headline else None
    configs = run_configs(dev) if headline and not args.no_configs else None

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "D": D, "n_blocks": n_blocks, "S": S,
                   "step": f"phase 1 + {S - 1} fused partial-update+merge + 1 partial update "
                           f"(= phase 1 + {S - 1} merges + {S} updates)",
                   "l2": "inputs larger than L2 (every kernel streams >= 268 MB); no flush",
                   "parallelism": f"dp{world} (token rows; no collective)"},
        "achieved_hbm_gbs_step": round(b["total"] / (elapsed_ms / K * 1e-3) / 1e9, 1),
        "frac_step": round(b["total"] / (elapsed_ms / K * 1e-3) / 1e9 / peak, 4),
        "frac_nominal_step": round(b["total"] / (elapsed_ms / K * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
        "roofline": roofline,
        "kernels": {n: {kk: (round(v, 5) if isinstance(v, float) else v) for kk, v in k.items()}
                    for n, k in kern.items()},
        "unfused": unfused,
        "prenorm": prenorm,
        "two_groups": groups,
        "decode": decode,
        "backward": backward,
        "configs": configs,
        "e2e": e2e,
        "gpu_launches": K * launches_per_step,
        "clocks": clk,
    }
    return res


def run_decode(dev, reps: int = 60):
    """The D = 7168 decode block pass ([256, 1, 7168], 9 summaries, S = 24): eager
    launches, one CUDA graph, and the graph with the side-stream inter-block pass.
    Each pass is timed alone with events, L2 flushed (and the stream idle) before it;
    the median is reported."""
    from transformer_depth_wise_gb300 import api
    wl = wk.WORKLOADS["decode_bf16"]
    tp = wk.two_phase_inputs(wl, device=dev)
    args = (tp["blocks"], tp["queries"], tp["gains"], tp["u"], tp["eps"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def time_pass(fn, host_ahead):
        ts = []
        for _ in range(reps):
            flush.fill_(1)
            torch.cuda.synchronize(dev)
            a, b = ev(), ev()
            if host_ahead:
                torch.cuda._sleep(HOST_AHEAD_CYCLES)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts)

    eager = api.TwoPhaseBlock(*args)
    graph = api.TwoPhaseBlock(*args)
    graph.capture()
    ov = api.TwoPhaseBlock(*args, overlap=True)
    ov.capture()
    for _ in range(3):
        eager.run(), graph.replay(), ov.replay()
    res = {"workload": wl.name, "tokens": wl.B * wl.T, "eager_launches": eager.launches_per_run,
           "eager_us": round(time_pass(eager.run, False), 2), "graph_us": round(time_pass(graph.replay, False), 2),
           "graph_side_stream_us": round(time_pass(ov.replay, False), 2),
           "device_us": {"eager": round(time_pass(eager.run, True), 2),
                         "graph": round(time_pass(graph.replay, True), 2),
                         "graph_side_stream": round(time_pass(ov.replay, True), 2)},
           "timing": "one pass per sample, median of %d; L2 flushed before each; *_us from an idle GPU "
                     "(host submission included), device_us with the submission hidden behind a device-side "
                     "wait queued first" % reps}
    res["tokens_per_s_graph"] = round(wl.B * wl.T / (min(res["graph_us"], res["graph_side_stream_us"]) * 1e-6), 1)
    del eager, graph, ov, flush
    return res


def run_two_phase_e2e(args, wl, dev, inp, n_blocks, world):
    """End to end through the public API: every step copies its summaries,
    queries, gains and u from pinned host memory, runs the fused block pass
    and reads its final partial back into pinned host memory.  The steps are
    pipelined by api.TwoPhaseStream (step k+1's host->device copies overlap
    step k's kernels; step k's partial returns while step k+1 runs); the
    timed region holds every copy of every timed step."""
    from transformer_depth_wise_gb300 import api
    host = {
        "blocks": [b.cpu().pin_memory() for b in inp["blocks"]],
        "queries": inp["queries"].cpu().pin_memory(),
        "gains": inp["gains"].cpu().pin_memory(),
        "u": inp["u"].cpu().pin_memory(),
    }
    ref = inp["blocks"][0]
    pipe = api.TwoPhaseStream(len(host["blocks"]), tuple(ref.shape), ref.dtype, wl.S, dev, inp["eps"])
    outs = [torch.empty(tuple(ref.shape), dtype=ref.dtype).pin_memory() for _ in range(2)]
    h2d = sum(b.numel() * b.element_size() for b in host["blocks"]) + sum(
        host[k].numel() * host[k].element_size() for k in ("queries", "gains", "u"))
    d2h = outs[0].numel() * outs[0].element_size()

    def step(k):
        return pipe.submit(host["blocks"], host["queries"], host["gains"], host["u"], outs[k % 2])

    for k in range(max(2, args.warmup)):
        step(k)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    K = max(2, args.steps // 2)
    barrier(world)
    torch.cuda.synchronize(dev)
    a.record(stream)
    pipe.copy_stream.wait_event(a)
    last = None
    for k in range(K):
        last = step(k)
    stream.wait_event(last)
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    tokens = wl.B * wl.T * K * world
    del pipe
    return {"value": round(tokens / (ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "ms_per_step": round(ms / K, 4),
            "pipelining": "two buffer sets; step k+1's H2D overlaps step k's block pass, step k's D2H step k+1's"}


def run_backward(dev, reps: int = 20):
    """Backward of the block_single_bf16 aggregation (10 x [4, 4096, 2048] bf16):
    source, query and gain gradients; L2 flushed before each timed call."""
    from transformer_depth_wise_gb300 import api
    wl = wk.WORKLOADS["block_single_bf16"]
    inp = wk.single_aggregation_inputs(wl, device=dev)
    dh = wk.upstream_grad(wk.generator(wl.seed + 11, dev), (wl.B, wl.T, wl.D), wl.dtype, dev)
    grads = [torch.empty_like(s) for s in inp["sources"]]
    ws = torch.empty((api.depth_aggregate_backward_workspace_rows(wl.D, wl.dtype), wl.D), dtype=torch.float32,
                     device=dev)
    call = lambda: api.depth_aggregate_backward(inp["sources"], inp["query"], inp["gain"], inp["eps"], dh,  # noqa
                                                grad_sources=grads, workspace=ws)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        call()
    ts = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        torch.cuda.synchronize(dev)
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    rows = wl.B * wl.T
    byts = accounting.aggregate_backward_bytes(wl.n, rows, wl.D, 2)
    peak, src = measured_peak()
    gbs = byts / (ms * 1e-3) / 1e9
    del inp, grads, ws, flush, dh
    return {"workload": wl.name, "ms": round(ms, 5), "tokens_per_s": round(rows / (ms * 1e-3), 1),
            "algorithmic_bytes": byts, "achieved_gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
            "peak_source": src, "launches": 2,
            "timing": "backward kernel + partial-sum reduce, median of %d, L2 flushed before each" % reps}


def run_single(args, wl, dev, world):
    """Single depth aggregation workloads (for profiling; not the headline line)."""
    from transformer_depth_wise_gb300 import api
    inp = wk.single_aggregation_inputs(wl, device=dev, rows=args.rows or None)
    out = torch.empty_like(inp["sources"][0])
    for _ in range(args.warmup):
        api.depth_aggregate(inp["sources"], inp["query"], inp["gain"], inp["eps"], out=out)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    times = []
    for _ in range(args.steps):
        flush.zero_()  # L2 flush between timed launches
        torch.cuda.synchronize(dev)
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        torch.cuda.nvtx.range_push("timed")
        a.record()
        api.depth_aggregate(inp["sources"], inp["query"], inp["gain"], inp["eps"], out=out)
        b.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    rows = inp["sources"][0].numel() // wl.D
    byts = accounting.aggregate_bytes(len(inp["sources"]), rows, wl.D, inp["sources"][0].element_size())
    ms = statistics.median(times)
    peak, src = measured_peak()
    gbs = byts / (ms * 1e-3) / 1e9
    n_src = len(inp["sources"])
    del inp, out, flush
    backward = run_backward(dev) if wl.name == "block_single_bf16" and not args.rows else None
    return {"metric": "depth aggregation tokens/s", "value": round(rows / (ms * 1e-3), 1),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32",
            "data": "synthetic", "config": {"workload": wl.name, "rows": rows, "D": wl.D,
                                            "n": n_src, "l2": "flushed between launches"},
            "roofline": {"bound": "hbm", "kernel": "aggregate", "achieved": round(gbs, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                         "traffic": None, "peak_source": src},
            "backward": backward}


def run_merge_update_only(args, wl, dev):
    """One fused update+merge launch per step on its own (profiling): the two-phase
    workload's width and dtype at --rows token rows (default 16384), holding only
    what the launch touches (o_k, p_in, the sublayer row, p_out, h; 0.7 GB at
    D = 4096), L2 flushed before each timed launch."""
    from transformer_depth_wise_gb300 import api
    rows = args.rows or 16384
    g = wk.generator(wl.seed, dev)
    (o, pin, sub), _ = wk.scaled_normal_sources(g, 3, (1, rows, wl.D), 0.5, 3.0, wl.dtype, dev)
    W, G = wk.queries_and_gains(g, 1, wl.D, dev)
    u = wk.sublayer_u(g, 1, wl.D, dev)[0].contiguous()
    lse = torch.empty(rows, device=dev).normal_(0.0, 2.0, generator=g)
    p_out, h = torch.empty_like(o), torch.empty_like(o)
    call = lambda: api.block_merge_update(o, lse, pin, sub, u, W[0], G[0], 1e-8, partial_out=p_out,  # noqa
                                          h_out=h)
    for _ in range(args.warmup):
        call()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)
    torch.cuda.nvtx.range_push("timed")
    ms = _event_median_ms(call, args.steps, flush)
    torch.cuda.nvtx.range_pop()
    peak, src = measured_peak()
    byts = accounting.merge_update_bytes(rows, wl.D, o.element_size(), first=False)
    r = _rate(byts, ms, peak)
    del o, pin, sub, p_out, h, flush
    return {"metric": "fused update+merge launch", "kernel": "merge_update", "rows": rows, "D": wl.D,
            "dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32", "steps": args.steps,
            "warmup": args.warmup, "peak_source": src, **r,
            "timing": "one launch per sample, L2 flushed before each, median of %d" % args.steps}


def run_full_stack(args, wl, dev, world):
    from transformer_depth_wise_gb300 import api
    inp = wk.full_stack_inputs(wl, device=dev, rows=args.rows or None)
    srcs = [inp["v0"]] + [torch.empty_like(inp["v0"]) for _ in range(wl.L)]
    y = torch.empty_like(inp["v0"])
    for _ in range(args.warmup):
        api.full_stack_forward(inp["v0"], inp["queries"], inp["gains"], inp["u"], inp["eps"], srcs, y)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    a.record()
    for _ in range(args.steps):
        api.full_stack_forward(inp["v0"], inp["queries"], inp["gains"], inp["u"], inp["eps"], srcs, y)
    b.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / args.steps
    rows = inp["v0"].numel() // wl.D
    byts = accounting.full_stack_bytes(wl.L, rows, wl.D, 2)
    peak, src = measured_peak()
    gbs = byts / (ms * 1e-3) / 1e9
    # The same stack with the two-phase schedule of block size S.
    S = args.schedule_block_size
    ws = torch.empty(int(api._lib.lib().attnres_full_stack_two_phase_workspace_bytes(
        wl.L, S, 1, rows, wl.D, 1)), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        api.full_stack_two_phase(inp["v0"], inp["queries"], inp["gains"], inp["u"], S, inp["eps"], srcs, y, ws)
    torch.cuda.synchronize(dev)
    torch.cuda.nvtx.range_push("timed_two_phase")
    a.record()
    for _ in range(args.steps):
        api.full_stack_two_phase(inp["v0"], inp["queries"], inp["gains"], inp["u"], S, inp["eps"], srcs, y, ws)
    b.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    ms2 = a.elapsed_time(b) / args.steps
    b2 = accounting.full_two_phase_bytes(wl.L, S, rows, wl.D, 2)
    two_phase = {"schedule_block_size": S, "ms_per_step": round(ms2, 4),
                 "tokens_per_s": round(rows / (ms2 * 1e-3), 1), "algorithmic_bytes": b2,
                 "achieved_gbs": round(b2 / (ms2 * 1e-3) / 1e9, 1), "frac": round(b2 / (ms2 * 1e-3) / 1e9 / peak, 4),
                 "speedup_vs_naive": round(ms / ms2, 3)}
    del ws
    return {"metric": "Full AttnRes stack forward tokens/s", "value": round(rows / (ms * 1e-3), 1),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "rows": rows, "D": wl.D, "L": wl.L},
            "roofline": {"bound": "hbm", "kernel": "aggregate (fused f)", "achieved": round(gbs, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                         "traffic": None, "peak_source": src},
            "two_phase": two_phase}


# Cycles of a device-side wait queued before each timed call (about 1 ms at
# 2 GHz): the host marshals and launches fn() while the GPU waits, so the
# events bracket the device's work alone, not the Python call around it.
HOST_AHEAD_CYCLES = 2_000_000


def _event_median_ms(fn, reps, flush=None):
    """Median CUDA-event time of fn() over reps calls, each alone on the
    stream (after an L2 flush when `flush` is given), with the host's launch
    work hidden behind a device-side wait queued before the first event."""
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.fill_(1)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def _rate(byts, ms, peak):
    gbs = byts / (ms * 1e-3) / 1e9
    return {"algorithmic_bytes": int(byts), "ms": round(ms, 5), "achieved_gbs": round(gbs, 1),
            "frac": round(gbs / peak, 4), "frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4)}


def run_configs(dev):
    """Every other workload of the benchmark recipe, each timed on its own:
    CUDA events around the launches, L2 flushed before each timed call where
    the inputs would otherwise sit in L2, median over the repetitions.
    `frac` divides the algorithmic bytes per second by the measured copy
    bandwidth, `frac_nominal` by the nominal 8 TB/s."""
    from transformer_depth_wise_gb300 import api
    peak, _ = measured_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    res = {}

    # Full single aggregation, fp32 (393 KB): launch-latency bound.  Both runs:
    # the drawn query and the zero query (the mean of the sources).
    wl = wk.WORKLOADS["full_single_f32"]
    one = {}
    for zero in (False, True):
        inp = wk.single_aggregation_inputs(wl, device=dev, zero_query=zero)
        out = torch.empty_like(inp["sources"][0])
        call = lambda: api.depth_aggregate(inp["sources"], inp["query"], inp["gain"], inp["eps"], out=out)  # noqa
        for _ in range(3):
            call()
        ms = _event_median_ms(call, 200, flush)
        r = _rate(accounting.aggregate_bytes(wl.n, wl.rows, wl.D, 4), ms, peak)
        r["us"] = round(ms * 1e3, 2)
        one["zero_query" if zero else "query"] = r
    one.update({"workload": wl.name, "bound": "launch latency (0.39 MB moves in 0.06 us at 8 TB/s)",
                "timing": "one launch per sample, L2 flushed before each, median of 200"})
    res[wl.name] = one

    # Block single aggregation, bf16 (738 MB).
    wl = wk.WORKLOADS["block_single_bf16"]
    inp = wk.single_aggregation_inputs(wl, device=dev)
    out = torch.empty_like(inp["sources"][0])
    call = lambda: api.depth_aggregate(inp["sources"], inp["query"], inp["gain"], inp["eps"], out=out)  # noqa
    for _ in range(3):
        call()
    ms = _event_median_ms(call, 30, flush)
    r = _rate(accounting.aggregate_bytes(wl.n, wl.rows, wl.D, 2), ms, peak)
    r.update({"workload": wl.name, "tokens_per_s": round(wl.rows / (ms * 1e-3), 1), "bound": "hbm",
              "timing": "one launch per sample, L2 flushed before each, median of 30"})
    res[wl.name] = r
    del inp, out

    # Full 186-sublayer stack, plain and with the two-phase schedule (S = 16, the fastest block size on a GB300).
    wl = wk.WORKLOADS["full_stack_bf16"]
    inp = wk.full_stack_inputs(wl, device=dev)
    srcs = [inp["v0"]] + [torch.empty_like(inp["v0"]) for _ in range(wl.L)]
    y = torch.empty_like(inp["v0"])
    plain = lambda: api.full_stack_forward(inp["v0"], inp["queries"], inp["gains"], inp["u"], inp["eps"], srcs, y)  # noqa
    S = 16
    ws = torch.empty(int(api._lib.lib().attnres_full_stack_two_phase_workspace_bytes(wl.L, S, 1, wl.rows, wl.D, 1)),
                     dtype=torch.uint8, device=dev)
    two = lambda: api.full_stack_two_phase(inp["v0"], inp["queries"], inp["gains"], inp["u"], S, inp["eps"],  # noqa
                                           srcs, y, ws)
    for _ in range(2):
        plain(), two()
    ms_p = _event_median_ms(plain, 5, flush)
    ms_t = _event_median_ms(two, 5, flush)
    # the same stacks as one CUDA graph each (api.FullStack)
    graphs = {}
    for name, S_g in (("plain", None), ("two_phase", S)):
        fs = api.FullStack(inp["v0"], inp["queries"], inp["gains"], inp["u"], inp["eps"], S=S_g)
        fs.capture()
        graphs[name] = round(_event_median_ms(fs.replay, 5, flush), 4)
        del fs
    rp = _rate(accounting.full_stack_bytes(wl.L, wl.rows, wl.D, 2), ms_p, peak)
    rt = _rate(accounting.full_two_phase_bytes(wl.L, S, wl.rows, wl.D, 2), ms_t, peak)
    rt.update({"schedule_block_size": S, "tokens_per_s": round(wl.rows / (ms_t * 1e-3), 1),
               "speedup_vs_plain": round(ms_p / ms_t, 3)})
    rp.update({"workload": wl.name, "tokens_per_s": round(wl.rows / (ms_p * 1e-3), 1), "launches": wl.L + 1,
               "two_phase": rt, "graph_ms": graphs,
               "timing": "one whole stack per sample, L2 flushed before each, median of 5"})
    res[wl.name] = rp
    del inp, srcs, y, ws

    # Long prefill, D = 7168: the single aggregation (n = 10) and the two-phase
    # block pass (9 summaries, S = 24) with per-kernel events.
    wl = wk.WORKLOADS["long_prefill_bf16"]
    inp = wk.single_aggregation_inputs(wl, device=dev)
    out = torch.empty_like(inp["sources"][0])
    call = lambda: api.depth_aggregate(inp["sources"], inp["query"], inp["gain"], inp["eps"], out=out)  # noqa
    for _ in range(2):
        call()
    ms = _event_median_ms(call, 5)
    single = _rate(accounting.aggregate_bytes(wl.n, wl.rows, wl.D, 2), ms, peak)
    del inp, out
    tp = wk.two_phase_inputs(wl, device=dev)
    blk = api.TwoPhaseBlock(tp["blocks"], tp["queries"], tp["gains"], tp["u"], tp["eps"], fused=True)
    for _ in range(2):
        blk.run()
    torch.cuda.synchronize()
    K = 3
    el, events, _ = time_block(blk, K, dev, 1, torch.cuda.current_stream(dev), fused=True, label="timed_long_prefill")
    n_blocks = len(tp["blocks"])
    b = accounting.two_phase_block_bytes(n_blocks, wl.S, wl.rows, wl.D, 2, fused=True)
    p1 = statistics.mean(e["phase1"][0].elapsed_time(e["phase1"][1]) for e in events)
    mg = statistics.mean(a.elapsed_time(c) for e in events for a, c in e["merge"])
    block = _rate(b["total"], el / K, peak)
    block.update({"tokens_per_s": round(wl.rows / (el / K * 1e-3), 1), "launches": blk.launches_per_run,
                  "phase1": _rate(b["phase1"], p1, peak),
                  "merge_update": _rate(b["merges"] / (wl.S - 1), mg, peak)})
    res[wl.name] = {"workload": wl.name, "single_aggregation": single, "two_phase_block": block,
                    "timing": "inputs far larger than L2; mean of %d block passes, median of 5 aggregations" % K}
    del tp, blk, flush
    torch.cuda.empty_cache()
    return res


def cpu_baseline_block(wl):
    v, dt, sample = oracle_block_rows_per_s(wl)
    return {"value": round(v, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": sample, "seconds": round(dt, 2)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="two_phase_bf16", choices=sorted(wk.WORKLOADS))
    ap.add_argument("--rows", type=int, default=0, help="shrink to B=1, T=rows (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="headline only: skip the per-workload measurements of the other configs")
    ap.add_argument("--kernel", default="", choices=["", "merge_update", "aggregate"],
                    help="time one kernel alone at --rows token rows (profiling; no headline line): the fused "
                         "update+merge at the workload's width, or the workload's single aggregation")
    ap.add_argument("--schedule-block-size", type=int, default=16,
                    help="Full stack: block size S of the two-phase schedule timed beside the plain stack")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = wk.WORKLOADS[args.workload]

    if args.impl == "reference":
        # The reference arm is the fp64 CPU oracle, on rank 0 only; under torchrun the
        # other ranks exit at once, and no process group is formed for it.
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if rank == 0:
            rates = []
            for _ in range(args.warmup):      # untimed: loads the oracle and touches its inputs
                oracle_block_rows_per_s(wl, rows_target_s=0.05, max_rows=16)
            t_total = 0.0
            for _ in range(max(1, args.steps)):
                v, dt, sample = oracle_block_rows_per_s(wl, rows_target_s=max(1.0, 60.0 / max(1, args.steps)))
                rates.append(v)
                t_total += dt
            value = statistics.mean(rates)
            line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
                    "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": round(t_total / max(1, args.steps) * 1e3, 2),
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                    "data": "synthetic",
                    "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "D": wl.D, "S": wl.S},
                    "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1,
                                     "kind": "oracle", "sample": sample},
                    "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        return

    rank, local, world = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CUDA path has no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from transformer_depth_wise_gb300 import _lib
    _lib.lib()

    if args.kernel == "merge_update":
        res = run_merge_update_only(args, wl, dev)
    elif args.kernel == "aggregate":
        res = run_single(args, wl, dev, world)
    elif wl.name in ("two_phase_bf16", "long_prefill_bf16", "decode_bf16"):
        res = run_two_phase(args, wl, dev, rank, world)
    elif wl.name == "full_stack_bf16":
        res = run_full_stack(args, wl, dev, world)
    else:
        res = run_single(args, wl, dev, world)

    if rank == 0:
        if not args.no_cpu_baseline and not args.kernel and not args.rows and "two_phase" in wl.name and world == 1:
            res["cpu_baseline"] = cpu_baseline_block(wl)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
