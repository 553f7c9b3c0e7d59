"""Benchmark: microseconds per decode layer-step (and the scan's HBM roofline).

One step = one decode layer-step of the whole hot path (key scan, exact top-K,
split-K softmax.V over the selected rows and the window, gamma merge) through
the C ABI, on seeded synthetic data shaped like the pages' workloads.  The
default workload is the Llama-3-8B layer at 128K context (32 query / 8 KV
heads, K = 2048, window 128 + 512); --workload picks another one.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

The default run (llama128k at N = 1) also times, in the same process and
reported under "secondary", the 1M-token decode step (the metric's second
context), the same two decode workloads through the int8 key codes with exact
rescoring (sparse_attn_decode_q8; each step codes its newest key) and the 64K
ReTopK reuse stream (CUDA-graph timed over its 512 steps); --no-secondary
skips them.  --q8 times the quantised path alone.  cpu_baseline is the fp64 oracle on one
host core, cpu_baseline_parallel the same code with one thread per query head.

--impl reference times the fp64 CPU oracle (the test oracle, as it stands) on
a bounded sample of the same workload, on the host cores.

Under torchrun (N > 1) every rank runs its own replica of the layer-step
(independent problems, no data-path collective): scaling is weak and the
value is the aggregate microseconds per layer-step over all ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "us per decode layer-step (scan + top-K + gather + merge)"
UNIT = "us/layer-step"
L2_BYTES = 126 * 1024 * 1024


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Maximum of a per-rank scalar (timing plumbing only)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int, device=None) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        import tempfile
        self.index = index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"tsa_clocks_{index}_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            if os.path.exists(self.path):
                os.remove(self.path)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t_end = time.time() + 3.0  # wait for the first sample before the work starts
        while time.time() < t_end:
            if os.path.exists(self.path) and os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)  # one more sample after the timed region
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        if not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        os.remove(self.path)
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workloads
def algorithmic_bytes(wl) -> dict:
    """Bytes the method must move per layer-step: every K row of the cache once
    per KV head, the V rows of the selected set once per query head, the V rows
    of the window once per KV head, q in and the fp32 output and lse out."""
    d = wl.d
    lens = wl.lens(0)
    k_bytes = sum(lens) * wl.Hkv * d * 2
    win = sum(min(wl.n_init + wl.n_recent, L) for L in lens)
    pool = [L - min(wl.n_init + wl.n_recent, L) for L in lens]
    sel = sum(min(wl.K, p) for p in pool)
    v_bytes = sel * wl.Hq * d * 2 + win * wl.Hkv * d * 2
    io = wl.B * wl.Hq * (d * 2 + d * 4 + 4)
    return {"scan": k_bytes, "gather": v_bytes, "io": io, "total": k_bytes + v_bytes + io}


SCAN_SOURCES = ("scan.cu", "tsa_internal.cuh", "tsa_kernels.h")


def scan_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in SCAN_SOURCES:
        with open(os.path.join(ROOT, "top_retrieval_sparse_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def scan_traffic(wl, rows_per_launch: int, record: str = "scan_llama128k.json"):
    """DRAM bytes (read + write) of one scan launch from a tracked ncu record
    (profiles/scan_llama128k.json, or scan_q8_llama128k.json for the
    quantised scan), or None when the scan sources changed since it was
    captured.  Its per-row traffic is scaled to this launch's key rows."""
    path = os.path.join(ROOT, "profiles", record)
    if not os.path.exists(path):
        return None, "no ncu record"
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != scan_sources_sha256():
        return None, "scan sources changed since the ncu capture"
    per_row = rec["traffic_bytes_per_launch"] / rec["key_rows_per_launch"]
    note = "ncu capture of llama128k" if wl.name == "llama128k" else \
        "llama128k ncu capture scaled by key rows"
    return int(round(per_row * rows_per_launch)), note


def run_ours(args, ws, rank, local):
    import torch
    import top_retrieval_sparse_gb300 as tsa
    from workloads.gen import make_decode

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    name = args.workload
    wl = make_decode(name, device=dev, seed=rank)  # each rank: its own replica
    paged = wl.page_table is not None
    kv = (tsa.kv_paged(wl.k_pages, wl.v_pages, wl.page_table) if paged
          else tsa.kv_contiguous(wl.k, wl.v))
    if paged:  # the contiguous copy is not needed on the device
        wl.k = wl.k.cpu() if args.cpu_baseline else None
        wl.v = wl.v.cpu() if args.cpu_baseline else None
        torch.cuda.empty_cache()
    B, Hq, d, K = wl.B, wl.Hq, wl.d, wl.K
    q8 = getattr(args, "q8", False)
    size_fn = tsa.decode_q8_workspace_size if q8 else tsa.decode_workspace_size
    nb = size_fn(B, Hq, wl.Hkv, d, kv.l_cap, K, wl.n_init, wl.n_recent)
    work = torch.zeros(nb, dtype=torch.uint8, device=dev)  # zeroed once, then reused
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    lens_all = torch.tensor([wl.lens(t) for t in range(wl.steps)], dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    codes = None
    if q8:  # scales fitted on the prefill rows; each step codes its newest key
        codes = tsa.KeyCodes(kv, B=B)
        tsa.quantize_keys(kv, codes, lens_all[0] - 1, fit=True, stream=stream)

    def step(i):
        t = i % wl.steps
        if q8:
            tsa.sparse_attn_decode_q8(wl.q_all[t], kv, codes, lens_all[t], K, wl.n_init,
                                      wl.n_recent, n_new=1, scale=wl.scale, out=out,
                                      lse_out=lse, workspace=work, stream=stream)
        else:
            tsa.sparse_attn_decode(wl.q_all[t], kv, lens_all[t], K, wl.n_init, wl.n_recent,
                                   wl.scale, out=out, lse_out=lse, workspace=work, stream=stream)

    clocks = Clocks(torch.cuda.current_device() if ws == 1 else local)
    if not args.device_only:
        clocks.start()  # sampling spans the warm-up and the timed region
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # ---- device-timed region: whole layer-steps, CUDA events on the launching stream ----
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    n_launch0 = tsa.kernel_launches()
    t0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    t1.record(stream)
    torch.cuda.synchronize()
    n_launches = tsa.kernel_launches() - n_launch0
    if ws > 1:
        torch.distributed.barrier()

    # ---- second timed region: the same steps with per-stage events (the events
    # between kernels cost the launch overlap, so this region only splits time) ----
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e4 in ev:  # torch tracks recording itself; the library re-records these
        for e in e4:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        tsa.set_stage_events(ev[i])
        step(args.warmup + i)
    tsa.set_stage_events(None)
    torch.cuda.synchronize()
    clk = clocks.stop() if not args.device_only else None
    total_ms = t0.elapsed_time(t1)
    total_ms = max_over_ranks(total_ms, ws, dev)
    scan_ms = [e[0].elapsed_time(e[1]) for e in ev]
    sel_ms = [e[1].elapsed_time(e[2]) for e in ev]
    att_ms = [e[2].elapsed_time(e[3]) for e in ev]
    ms_per_step = total_ms / args.steps
    us_per_layer_step = 1000.0 * ms_per_step / ws  # aggregate over all replicas

    ab = algorithmic_bytes(wl)
    if q8:  # the quantised scan reads one byte per key element
        ab["scan"] //= 2
    hbm, peak_kind = peaks()
    scan_avg = statistics.mean(scan_ms)
    achieved = ab["scan"] / (scan_avg * 1e-3) / 1e9
    path_gbs = ab["total"] / (ms_per_step * 1e-3) / 1e9

    if args.trace:  # per-CTA timeline of a few more steps (after the timed region)
        trace_summary = run_trace(args, step, tsa, torch, dev)
    else:
        trace_summary = None
    if args.device_only:  # profiling mode: the device path only
        return {"workload": name, "us_per_layer_step": round(us_per_layer_step, 3),
                "stages_ms": {"scan": round(scan_avg, 5),
                              "topk+attend+merge": round(statistics.mean(sel_ms)
                                                         + statistics.mean(att_ms), 5)},
                "scan_gbs": round(achieved, 1), "trace": trace_summary} if rank == 0 else None
    traffic, traffic_note = scan_traffic(
        wl, ab["scan"] // (wl.d * (1 if q8 else 2)),
        "scan_q8_llama128k.json" if q8 else "scan_llama128k.json")
    # ---- end to end through the public API with host buffers ----
    e2e = run_e2e(args, wl, kv, work, tsa, torch, dev, ws, codes=codes)

    res = {
        "metric": METRIC, "value": round(us_per_layer_step, 3), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": name, "B": B, "Hq": Hq, "Hkv": wl.Hkv, "d": d,
            "context": wl.L0 if B > 1 else wl.L0[0], "K": K,
            "window": [wl.n_init, wl.n_recent], "layout": "paged16" if paged else "contiguous",
            "decode_steps_cycled": wl.steps,
            "l2": f"inputs larger than L2 (K cache {ab['scan'] / 2**20:.0f} MiB > 126 MiB); no flush",
            "parallelism": f"replicas{ws}" if ws > 1 else "single",
            "keys": ("int8 codes (scan) + bf16 rows (exact rescoring); scales fitted on the "
                     "prefill rows, each step codes its newest key") if q8 else "bf16",
        },
        "stages_ms": {"scan": round(scan_avg, 5),
                      "topk+attend+merge": round(statistics.mean(sel_ms) + statistics.mean(att_ms), 5),
                      "note": "second timed region with per-stage events"},
        "path_algorithmic_gbs": round(path_gbs, 1),
        "roofline": {"kernel": ("scan_kernel<q8> (query preparation + code scan, pair emission)"
                                if q8 else "scan_kernel (GQA key scan, pair emission)"),
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "frac_of_8tbs": round(achieved / 8000.0, 4),
                     "traffic": traffic, "traffic_source": traffic_note,
                     "algorithmic_bytes_per_launch": ab["scan"]},
        "e2e": e2e,
        "gpu_launches": n_launches,
        "clocks": clk,
    }
    if args.cpu_baseline and rank == 0:
        res["cpu_baseline"] = oracle_baseline(wl, budget_s=args.cpu_budget)
        res["cpu_baseline_parallel"] = oracle_baseline_parallel(wl, budget_s=args.cpu_budget)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return res if rank == 0 else None


def run_retopk(args, ws, rank, local):
    """ReTopK decode (Qwen2.5-7B geometry, 64K or 1M): one layer-step is retopk_step
    for all 28 query heads -- cosine recall, candidate union, rescoring and
    re-top-K on reuse heads, the exact scan + top-K on exact heads, sparse
    softmax.V and the FIFO push.  Reports microseconds per layer-step over the
    config's 512-step stream, per path class, and the path mix."""
    import torch
    import top_retrieval_sparse_gb300 as tsa
    from workloads.gen import make_retopk
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = make_retopk(args.workload, device=dev, seed=rank)
    kv = tsa.kv_contiguous(wl.k, wl.v)
    g = tsa.ReTopK(wl.Hq, wl.Hkv, wl.d, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r, wl.lcap,
                   device=dev)
    # the FIFO starts from the last C prefill queries and their exact causal
    # top-K (one library call for all of them)
    sup, cnt = tsa.prefill_supports(wl.q_prefill.contiguous(), kv, wl.L0, wl.K, wl.scale)
    g.init(wl.q_prefill.contiguous(), sup, cnt)
    out = torch.empty((wl.Hq, wl.d), dtype=torch.float32, device=dev)
    path = torch.empty((wl.steps, wl.Hq), dtype=torch.int32, device=dev)
    mc = torch.empty((wl.steps, wl.Hq), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    steps = min(args.steps, wl.steps)
    state0, counters0 = g.state.clone(), g.counters()

    def stream_steps(record_path, ev=None):
        g.state.copy_(state0)
        g.set_counters(*counters0)
        n0 = tsa.kernel_launches()
        for t in range(steps):
            if ev is not None:
                ev[t][0].record(stream)
            g.step(wl.q_all[t], kv, wl.length(t), wl.scale, out=out,
                   path_out=path[t] if record_path else None,
                   mcand_out=mc[t] if record_path else None, stream=stream)
            if ev is not None:
                ev[t][1].record(stream)
        return tsa.kernel_launches() - n0

    for _ in range(max(1, args.warmup // 8)):
        stream_steps(False)
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device() if ws == 1 else local)
    clocks.start()
    # Launched from the host one call at a time, a reuse step's kernels are
    # shorter than the host's launch work, so the device time is measured on
    # a CUDA graph of the whole step stream (captured from the same calls);
    # the host-launched time is reported beside it.
    side = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    g.state.copy_(state0)
    g.set_counters(*counters0)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        n_launch0 = tsa.kernel_launches()
        for t in range(steps):
            g.step(wl.q_all[t], kv, wl.length(t), wl.scale, out=out, stream=side)
        launches = tsa.kernel_launches() - n_launch0
    for _ in range(2):  # warm-up replays
        g.state.copy_(state0)
        graph.replay()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    g.state.copy_(state0)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    total_ms = max_over_ranks(t0.elapsed_time(t1), ws, dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    stream_steps(False)
    e1.record(stream)
    torch.cuda.synchronize()
    eager_us = 1000.0 * e0.elapsed_time(e1) / steps
    # per-step events and the path of every head (a second pass over the same stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    stream_steps(True, ev)
    torch.cuda.synchronize()
    clk = clocks.stop()
    per = [e[0].elapsed_time(e[1]) * 1000 for e in ev]
    p_h, m_h = path[:steps].cpu(), mc[:steps].cpu()
    exact_steps = [t for t in range(steps) if int(p_h[t].sum()) > 0]
    reuse_steps = [t for t in range(steps) if int(p_h[t].sum()) == 0]
    reuse_heads = int((p_h == 0).sum())
    mean_m = float(m_h[p_h == 0].float().mean()) if reuse_heads else None
    us = 1000.0 * total_ms / steps / ws
    # bytes a step must move: exact heads scan the K cache of their KV heads and
    # gather their selected V rows; reuse heads read M_t K rows, their K V rows
    # and their cached supports (R*K indices) and queries (C*128 floats)
    L = wl.length(0)
    k_scan = wl.Hkv * L * wl.d * 2
    v_rows = wl.Hq * wl.K * wl.d * 2
    reuse_bytes = (mean_m or 0) * wl.d * 2 * wl.Hq + v_rows + wl.Hq * (wl.R * wl.K * 4 + wl.C * wl.d * 4)
    res = {
        "metric": METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / steps, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                   "context": wl.L0, "K": wl.K, "C": wl.C, "R": wl.R, "W": wl.W,
                   "tau": wl.tau, "T_r": wl.T_r, "decode_steps": steps,
                   "l2": (f"K cache {wl.Hkv * wl.lcap * wl.d * 2 >> 20} MiB on exact steps "
                          "(L2 126 MiB); the stream is run as is"),
                   "parallelism": f"replicas{ws}" if ws > 1 else "single"},
        "host_launched_us_per_step": round(eager_us, 3),
        "timing": f"CUDA graph of the {steps}-step stream captured from retopk_step calls",
        "paths": {"steps_with_exact_heads": len(exact_steps), "all_reuse_steps": len(reuse_steps),
                  "reuse_head_fraction": round(reuse_heads / (steps * wl.Hq), 4),
                  "mean_candidates_reuse": round(mean_m, 1) if mean_m else None,
                  "us_steps_with_exact": round(statistics.median([per[t] for t in exact_steps]), 2)
                  if exact_steps else None,
                  "us_all_reuse_steps": round(statistics.median([per[t] for t in reuse_steps]), 2)
                  if reuse_steps else None},
        "roofline": {"kernel": "whole reuse step (selector, key scan with no exact head, finish)", "bound": "hbm",
                     "achieved": round(reuse_bytes / (statistics.median([per[t] for t in reuse_steps])
                                                      * 1e-6) / 1e9, 1) if reuse_steps else None,
                     "peak": peaks()[0], "peak_kind": peaks()[1], "unit": "GB/s",
                     "frac": None, "traffic": None,
                     "algorithmic_bytes_per_reuse_step": int(reuse_bytes),
                     "algorithmic_bytes_per_exact_step": int(k_scan + v_rows)},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if res["roofline"]["achieved"]:
        res["roofline"]["frac"] = round(res["roofline"]["achieved"] / peaks()[0], 4)
    if not args.device_only:
        res["e2e"] = run_retopk_e2e(args, wl, kv, g, tsa, torch, dev, state0, counters0, steps,
                                    ws)
        if args.cpu_baseline and rank == 0:
            res["cpu_baseline"] = oracle_retopk_baseline(wl, budget_s=args.cpu_budget)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return res if rank == 0 else None


def run_retopk_batched(args, ws, rank, local, nseq=4):
    """Batched ReTopK (continuous batching with per-request state): nseq
    sequences of the 64K ReTopK workload (Qwen2.5-7B geometry, their own
    seeds), each with its own FIFO state, stepped together by
    retopk_step_batched; CUDA-graph timed over the step stream."""
    import torch
    import top_retrieval_sparse_gb300 as tsa
    from workloads.gen import make_retopk
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    steps = min(args.steps, 512)
    wls = [make_retopk("retopk64k", device=dev, seed=97 * rank + i, steps=steps)
           for i in range(nseq)]
    w0 = wls[0]
    k = torch.stack([w.k[0] for w in wls]).contiguous()
    v = torch.stack([w.v[0] for w in wls]).contiguous()
    for w in wls:
        w.k = w.v = None
    torch.cuda.empty_cache()
    kv = tsa.kv_contiguous(k, v)
    hs = []
    for i, w in enumerate(wls):
        kv1 = tsa.kv_contiguous(k[i:i + 1], v[i:i + 1])
        sup, cnt = tsa.prefill_supports(w.q_prefill.contiguous(), kv1, w.L0, w.K, w.scale)
        g = tsa.ReTopK(w.Hq, w.Hkv, w.d, w.K, w.C, w.R, w.W, w.tau, w.T_r, w.lcap, device=dev)
        g.init(w.q_prefill.contiguous(), sup, cnt)
        hs.append(g)
    state0 = [(g.state.clone(), g.counters()) for g in hs]
    work = torch.zeros(tsa.ReTopK.batched_workspace_size(hs[0], nseq), dtype=torch.uint8,
                       device=dev)
    q_all = torch.stack([torch.stack([w.q_all[t] for w in wls]) for t in range(steps)]).contiguous()
    out = torch.empty((nseq, w0.Hq, w0.d), dtype=torch.float32, device=dev)
    path = torch.empty((steps, nseq, w0.Hq), dtype=torch.int32, device=dev)

    def reset():
        for g, (st, cn) in zip(hs, state0):
            g.state.copy_(st)
            g.set_counters(*cn)

    def run(stream, record=False):
        for t in range(steps):
            tsa.ReTopK.step_batched(hs, q_all[t], kv, [w.length(t) for w in wls], w0.scale,
                                    out=out, path_out=path[t] if record else None,
                                    workspace=work, stream=stream)

    stream = torch.cuda.current_stream()
    reset()
    run(stream, record=True)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    reset()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        n0 = tsa.kernel_launches()
        run(side)
        launches = tsa.kernel_launches() - n0
    for _ in range(2):
        for g, (st, _) in zip(hs, state0):
            g.state.copy_(st)
        graph.replay()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    for g, (st, _) in zip(hs, state0):
        g.state.copy_(st)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    p_h = path.cpu()
    return {
        "metric": "us per batched ReTopK decode layer-step", "value": round(1000 * ms / steps, 3),
        "unit": "us/batched-layer-step", "n_gpus": 1, "steps": steps, "warmup": 2,
        "ms_per_step": round(ms / steps, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "us_per_sequence_step": round(1000 * ms / steps / nseq, 3),
        "config": {"workload": "retopk_batched", "sequences": nseq, "Hq": w0.Hq, "Hkv": w0.Hkv,
                   "context": w0.L0, "K": w0.K, "C": w0.C, "R": w0.R, "W": w0.W, "tau": w0.tau,
                   "T_r": w0.T_r, "decode_steps": steps},
        "timing": f"CUDA graph of the {steps}-step stream of retopk_step_batched calls",
        "paths": {"reuse_head_fraction": round(float((p_h == 0).float().mean()), 4)},
        "gpu_launches": launches, "clocks": clk,
    }


def run_trace(args, step, tsa, torch, dev, nsteps=3):
    """Run a few steps with the per-CTA trace on and summarise each kernel:
    span (first CTA start -> last CTA exit), gap from the previous kernel,
    CTA count and mean per-phase durations (us)."""
    cap = 1 << 16
    buf = torch.zeros(64 + 48 * cap, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    tsa.set_trace(buf)
    for i in range(nsteps):
        step(10_000 + i)
    torch.cuda.synchronize()
    tsa.set_trace(None)
    recs = tsa.read_trace(buf)
    names = {1: "scan", 4: "retopk_selector", 7: "finish",
             8: "finish_phases"}
    # records of one launch share the kernel id; a launch of a kernel starts
    # after the previous launch of that kernel has ended
    by_kernel = {}
    for r in recs:
        by_kernel.setdefault(r["kernel"], []).append(r)
    launches = []
    for k, rs in by_kernel.items():
        rs.sort(key=lambda r: r["t"][0])
        cur = None
        for r in rs:
            if cur is None or r["t"][0] > cur["end"]:
                cur = {"kernel": k, "recs": [], "end": 0}
                launches.append(cur)
            cur["recs"].append(r)
            cur["end"] = max(cur["end"], r["t"][3])
    launches.sort(key=lambda ln: min(r["t"][0] for r in ln["recs"]))
    out, prev_end = [], None
    for ln in launches:
        rs = ln["recs"]
        t0 = min(r["t"][0] for r in rs)
        t3 = max(r["t"][3] for r in rs)
        ph = []
        for a_, b_ in ((0, 1), (1, 2), (2, 3)):
            v = [(r["t"][b_] - r["t"][a_]) / 1e3 for r in rs if r["t"][a_] and r["t"][b_]]
            ph.append(round(sum(v) / len(v), 3) if v else None)
        out.append({"kernel": names.get(ln["kernel"], ln["kernel"]), "ctas": len(rs),
                     "span_us": round((t3 - t0) / 1e3, 3),
                     "gap_us": round((t0 - prev_end) / 1e3, 3) if prev_end else None,
                     "cta_us_mean": round(sum((r["t"][3] - r["t"][0]) for r in rs) / len(rs) / 1e3, 3),
                     "phase_us_mean": ph})
        if ln["kernel"] != 8:
            prev_end = t3
    return out


def _cudart():
    """The CUDA runtime the library is linked against (already loaded)."""
    import ctypes as C
    path = None
    with open("/proc/self/maps") as f:
        for line in f:
            if "libcudart.so" in line:
                path = line.split()[-1]
                break
    rt = C.CDLL(path or "libcudart.so")
    P, sz, i32 = C.c_void_p, C.c_size_t, C.c_int
    rt.cudaMemcpyAsync.argtypes = [P, P, sz, i32, P]
    rt.cudaMemcpy2DAsync.argtypes = [P, sz, P, sz, sz, sz, i32, P]
    rt.cudaStreamSynchronize.argtypes = [P]
    return rt


def run_e2e(args, wl, kv, work, tsa, torch, dev, ws=1, codes=None):
    """End to end through the C ABI with host buffers.  Per step, on one
    stream: a host -> device copy of the step's query and lengths (pinned,
    one copy), the append of the step's K and V token rows from pinned host
    memory straight into their cache rows (one strided copy per sequence and
    tensor), the sparse_attn_decode call, a device -> host copy of the output
    and lse (one copy), and a stream synchronisation.  Wall-clock per step."""
    import ctypes as C
    import numpy as np
    rt = _cudart()
    H2D, D2H = 1, 2
    B, Hq, d, Hkv = wl.B, wl.Hq, wl.d, wl.Hkv
    paged = wl.page_table is not None
    qb, lb, rowb = B * Hq * d * 2, B * 4, d * 2
    host_ql = torch.empty((wl.steps, qb + lb), dtype=torch.uint8).pin_memory()
    host_k = torch.empty((wl.steps, B, Hkv, d), dtype=torch.bfloat16).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    pt = wl.page_table.cpu() if paged else None
    kc, vc = (wl.k_pages, wl.v_pages) if paged else (wl.k, wl.v)
    dst_rows = []  # per step: [(k address, v address, pitch)] per sequence
    for t in range(wl.steps):
        host_ql[t, :qb] = wl.q_all[t].cpu().contiguous().view(torch.uint8).reshape(-1)
        host_ql[t, qb:] = torch.from_numpy(np.asarray(wl.lens(t), dtype=np.int32).view(np.uint8))
        rows = []
        for b in range(B):  # the token appended at step t sits at row L0 + t
            pos = wl.L0[b] + t
            if paged:
                page, r = int(pt[b, pos // wl.page_size]), pos % wl.page_size
                host_k[t, b] = wl.k_pages[page, :, r].cpu()
                host_v[t, b] = wl.v_pages[page, :, r].cpu()
                off = ((page * Hkv) * wl.page_size + r) * rowb
                pitch = wl.page_size * rowb
            else:
                host_k[t, b] = wl.k[b, :, pos].cpu()
                host_v[t, b] = wl.v[b, :, pos].cpu()
                off = ((b * Hkv) * kv.l_cap + pos) * rowb
                pitch = kv.l_cap * rowb
            rows.append((kc.data_ptr() + off, vc.data_ptr() + off, pitch))
        dst_rows.append(rows)
    stage = torch.empty(qb + lb, dtype=torch.uint8, device=dev)
    res = torch.empty(B * Hq * (d + 1), dtype=torch.float32, device=dev)
    res_host = torch.empty_like(res, device="cpu").pin_memory()
    stream = torch.cuda.current_stream()
    sp = C.c_void_p(stream.cuda_stream)
    lib = tsa.lib()
    # the C ABI call's arguments, fixed for the run (the quantised call codes
    # the appended key itself: n_new = 1)
    call = (C.c_void_p(stage.data_ptr()), C.byref(kv.struct), C.c_void_p(stage.data_ptr() + qb),
            B, Hq, Hkv, d, wl.K, wl.n_init, wl.n_recent, C.c_float(wl.scale),
            C.c_void_p(res.data_ptr()), C.c_void_p(res.data_ptr() + B * Hq * d * 4), None, None,
            C.c_void_p(work.data_ptr()), C.c_size_t(work.numel()), sp)
    if codes is not None:
        call = call[:2] + (C.byref(codes.struct), 1) + call[2:]
    hk, hv, hq = host_k.data_ptr(), host_v.data_ptr(), host_ql.data_ptr()
    tokb = Hkv * rowb

    def one(i):
        t = i % wl.steps
        err = rt.cudaMemcpyAsync(stage.data_ptr(), hq + t * (qb + lb), qb + lb, H2D, sp)
        for b, (kd, vd, pitch) in enumerate(dst_rows[t]):
            src = (t * B + b) * tokb
            err |= rt.cudaMemcpy2DAsync(kd, pitch, hk + src, rowb, rowb, Hkv, H2D, sp)
            err |= rt.cudaMemcpy2DAsync(vd, pitch, hv + src, rowb, rowb, Hkv, H2D, sp)
        rc = lib.sparse_attn_decode(*call) if codes is None else lib.sparse_attn_decode_q8(*call)
        if rc:
            raise tsa.TsaError(rc, lib.tsa_last_error().decode())
        err |= rt.cudaMemcpyAsync(res_host.data_ptr(), res.data_ptr(), res.numel() * 4, D2H, sp)
        err |= rt.cudaStreamSynchronize(sp)
        if err:
            raise RuntimeError(f"CUDA copy or synchronise failed ({err})")

    for i in range(args.warmup):
        one(i)
    n = args.steps
    if ws > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(n):
        one(args.warmup + i)
    dt = time.perf_counter() - t0
    # whole job: the slowest rank's wall time over every rank's layer-steps
    dt = max_over_ranks(dt, ws, dev) / ws
    return {"value": round(1e6 * dt / n, 3), "unit": UNIT,
            "h2d_bytes_per_step": qb + lb + 2 * B * Hkv * rowb,
            "d2h_bytes_per_step": res_host.numel() * 4}


def cpu_model() -> str:
    """The host CPU's model string (x86 'model name', else Arm implementer/part)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model name", "Model"):
        for line in info.splitlines():
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    impl = part = None
    for line in info.splitlines():
        if line.startswith("CPU implementer") and ":" in line:
            impl = line.split(":", 1)[1].strip()
        if line.startswith("CPU part") and ":" in line:
            part = line.split(":", 1)[1].strip()
    if impl or part:
        name = {("0x41", "0xd4f"): "Arm Neoverse V2"}.get((impl, part), "")
        return f"{name} (implementer {impl}, part {part})".strip()
    import platform
    return platform.processor() or "unknown"


def oracle_baseline_parallel(wl, budget_s=10.0):
    """The same fp64 oracle with one thread per query head (the pages' own CPU
    axis): whole query heads of decode step 0 run concurrently, a wave of as
    many heads as there are threads at a time, until the budget; the wall time
    is scaled to a layer-step.  The oracle's C code releases the interpreter
    lock, so the threads run in parallel."""
    import oracle as orc
    from concurrent.futures import ThreadPoolExecutor
    from workloads.gen import bits
    G = wl.Hq // wl.Hkv
    L = wl.lens(0)
    threads = max(1, min(wl.Hq, os.cpu_count() or 1))
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
    done, t_used = 0, 0.0
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for i in range(0, len(pairs), threads):
            wave = pairs[i:i + threads]
            kv = {}
            for b, h in wave:  # the wave's KV heads, widened outside the timed part
                if (b, h // G) not in kv:
                    kv[(b, h // G)] = (bits(wl.k[b, h // G, :L[b]]), bits(wl.v[b, h // G, :L[b]]))
            qs = {(b, h): bits(wl.q(0)[b, h]) for b, h in wave}

            def job(bh):
                b, h = bh
                kb, vb = kv[(b, h // G)]
                orc.decode_head(qs[bh], kb, vb, wl.K, wl.n_init, wl.n_recent, wl.scale)

            t0 = time.perf_counter()
            list(ex.map(job, wave))
            t_used += time.perf_counter() - t0
            done += len(wave)
            if t_used >= budget_s:
                break
    return {"value": round(1e6 * t_used / done * wl.B * wl.Hq, 1), "unit": UNIT, "cores": threads,
            "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{done} of {wl.B * wl.Hq} (sequence, query head) pairs of decode step 0 in "
                      f"waves of {threads} threads (one per query head), {t_used:.1f} s, scaled "
                      f"to a whole layer-step"}


def oracle_baseline(wl, budget_s=12.0, steps=1):
    """fp64 single-threaded oracle on a bounded sample: whole query heads of
    decode step 0, as many as fit the time budget, scaled to one layer-step."""
    import oracle as orc
    from workloads.gen import bits
    G = wl.Hq // wl.Hkv
    done, t_used = 0, 0.0
    L = wl.lens(0)
    order = [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
    kcache = {}
    for b, h in order:
        key = (b, h // G)
        if key not in kcache:
            kcache.clear()
            src_k = wl.k if wl.k is not None else None
            kcache[key] = (bits(src_k[b, h // G, :L[b]]), bits(wl.v[b, h // G, :L[b]]))
        kb, vb = kcache[key]
        qb = bits(wl.q(0)[b, h])
        t0 = time.perf_counter()
        orc.decode_head(qb, kb, vb, wl.K, wl.n_init, wl.n_recent, wl.scale)
        t_used += time.perf_counter() - t0
        done += 1
        if t_used >= budget_s:
            break
    per_head = t_used / done
    return {"value": round(1e6 * per_head * wl.B * wl.Hq, 1), "unit": UNIT, "cores": 1,
            "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{done} of {wl.B * wl.Hq} (sequence, query head) pairs of decode step 0, "
                      f"{t_used:.1f} s, scaled to a whole layer-step"}


def run_retopk_e2e(args, wl, kv, g, tsa, torch, dev, state0, counters0, steps, ws=1):
    """ReTopK end to end through the C ABI with host buffers, over the step
    stream from its start (the FIFO state is stateful).  Per step, on one
    stream: a host -> device copy of the step's query (pinned), the append of
    the step's K and V token rows (row L0 + t of each KV head) from pinned
    host memory, the retopk_step call, a device -> host copy of the output
    and lse (one copy), and a stream synchronisation.  Wall-clock per step
    over the steps after the warm-up ones."""
    import ctypes as C
    rt = _cudart()
    H2D, D2H = 1, 2
    Hq, Hkv, d = wl.Hq, wl.Hkv, wl.d
    qb, rowb = Hq * d * 2, d * 2
    host_q = torch.empty((steps, qb), dtype=torch.uint8).pin_memory()
    host_k = torch.empty((steps, Hkv, d), dtype=torch.bfloat16).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    for t in range(steps):
        host_q[t] = wl.q_all[t].cpu().contiguous().view(torch.uint8).reshape(-1)
        host_k[t] = wl.k[0, :, wl.L0 + t].cpu()
        host_v[t] = wl.v[0, :, wl.L0 + t].cpu()
    stage = torch.empty(qb, dtype=torch.uint8, device=dev)
    res = torch.empty(Hq * (d + 1), dtype=torch.float32, device=dev)
    res_host = torch.empty_like(res, device="cpu").pin_memory()
    stream = torch.cuda.current_stream()
    sp = C.c_void_p(stream.cuda_stream)
    lib = tsa.lib()
    pitch = kv.l_cap * rowb
    hq, hk, hv = host_q.data_ptr(), host_k.data_ptr(), host_v.data_ptr()
    kc, vc = wl.k.data_ptr(), wl.v.data_ptr()
    tokb = Hkv * rowb

    def one(t):
        err = rt.cudaMemcpyAsync(stage.data_ptr(), hq + t * qb, qb, H2D, sp)
        off = (wl.L0 + t) * rowb
        err |= rt.cudaMemcpy2DAsync(kc + off, pitch, hk + t * tokb, rowb, rowb, Hkv, H2D, sp)
        err |= rt.cudaMemcpy2DAsync(vc + off, pitch, hv + t * tokb, rowb, rowb, Hkv, H2D, sp)
        rc = lib.retopk_step(g.handle, stage.data_ptr(), C.byref(kv.struct), wl.length(t),
                             C.c_float(wl.scale), res.data_ptr(), None, None, None, None,
                             res.data_ptr() + Hq * d * 4, g.workspace.data_ptr(),
                             g.workspace.numel(), sp)
        if rc:
            raise tsa.TsaError(rc, lib.tsa_last_error().decode())
        err |= rt.cudaMemcpyAsync(res_host.data_ptr(), res.data_ptr(), res.numel() * 4, D2H, sp)
        err |= rt.cudaStreamSynchronize(sp)
        if err:
            raise RuntimeError(f"CUDA copy or synchronise failed ({err})")

    torch.cuda.synchronize()
    g.state.copy_(state0)
    g.set_counters(*counters0)
    torch.cuda.synchronize()
    w = min(args.warmup, steps // 4)
    for t in range(w):
        one(t)
    if ws > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for t in range(w, steps):
        one(t)
    dt = time.perf_counter() - t0
    dt = max_over_ranks(dt, ws, dev) / ws  # whole job, as for the decode leg
    return {"value": round(1e6 * dt / (steps - w), 3), "unit": UNIT,
            "h2d_bytes_per_step": qb + 2 * tokb, "d2h_bytes_per_step": res_host.numel() * 4,
            "steps_timed": steps - w}


def oracle_retopk_baseline(wl, budget_s=12.0):
    """fp64 single-threaded oracle ReTopK on a bounded sample: query head 0
    from the start of the step stream.  Its FIFO holds the oracle's own exact
    causal top-K of the last C prefill queries (built untimed); its steps are
    timed per path class (exact: step 0 is a refresh; reuse: the following
    steps, until the budget), and the layer-step estimate weighs the classes
    by the refresh period T_r (one exact step in T_r) over all query heads."""
    import oracle as orc
    from workloads.gen import bits
    h = 0
    G = wl.Hq // wl.Hkv
    o = orc.ReTopK(wl.Hq, wl.d, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r)
    kb, vb = bits(wl.k[0, h // G]), bits(wl.v[0, h // G])
    qpre, qall = bits(wl.q_prefill[:, h]), bits(wl.q_all[:, h])
    for c in range(wl.C):
        p = wl.L0 - wl.C + c
        r = orc.decode_head(qpre[c], kb[: p + 1], vb[: p + 1], wl.K, 0, 0, wl.scale)
        o.set_slot(h, c, qpre[c], r["sel"])
    times = {0: [], 1: []}
    used = 0.0
    for t in range(wl.steps):
        L = wl.length(t)
        t0 = time.perf_counter()
        r = o.step_head(h, qall[t], kb[:L], vb[:L], wl.scale)
        dt = time.perf_counter() - t0
        o.advance()
        times[int(r["path"])].append(dt)
        used += dt
        if used >= budget_s and times[0] and times[1]:
            break
    te = statistics.mean(times[1]) if times[1] else 0.0
    tr = statistics.mean(times[0]) if times[0] else te
    per_step = wl.Hq * (te / wl.T_r + tr * (1.0 - 1.0 / wl.T_r))
    return {"value": round(1e6 * per_step, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"query head 0, steps 0-{len(times[0]) + len(times[1]) - 1} of the stream "
                       f"({len(times[1])} exact at {1e3 * te:.1f} ms, {len(times[0])} reuse at "
                       f"{1e3 * tr:.2f} ms, {used:.1f} s), weighted one exact step in T_r = "
                       f"{wl.T_r} and scaled to {wl.Hq} query heads")}


def run_reference(args, ws, rank):
    """The reference arm: the fp64 oracle on the host cores, bounded sample."""
    if rank != 0:
        return None
    import torch
    from workloads.gen import make_decode, make_retopk
    if args.workload.startswith("retopk"):
        # the ReTopK stream is stateful: one pass of the oracle over its start
        # (FIFO built untimed, then timed steps per path class, bounded)
        batched = args.workload == "retopk_batched"  # 4 sequences of the 64K stream
        wl = make_retopk("retopk64k" if batched else args.workload, device="cpu")
        t0 = time.perf_counter()
        base = oracle_retopk_baseline(wl, budget_s=args.cpu_budget)
        dt = time.perf_counter() - t0
        if batched:
            base["value"] = round(4 * base["value"], 1)
            base["unit"] = "us/batched-layer-step"
            base["sample"] += "; times 4 sequences of the batch"
        v = base["value"]
        return {
            "impl": "reference", "metric": METRIC, "value": v, "unit": base["unit"],
            "n_gpus": ws, "steps": 1, "warmup": 0, "ms_per_step": round(1000 * dt, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload},
            "timing": "one bounded pass of the oracle over the start of the step stream",
            "cpu_baseline": base,
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    wl = make_decode(args.workload, device="cpu")
    # the whole run stays within a few minutes: each step is a bounded sample
    # (at least one query head) of the workload
    per_step_budget = 150.0 / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        oracle_baseline(wl, budget_s=per_step_budget * 0.25)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(oracle_baseline(wl, budget_s=per_step_budget))
    dt = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    del torch
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * dt / args.steps, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload},
        "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": vals[-1]["sample"]},
        "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_secondary(args, ws, rank, local):
    """The other workloads the metric names, timed in the same run (N = 1):
    the 1M-token decode step (the metric's second context) and the ReTopK
    reuse stream at 64K (CUDA-graph timed over its 512 steps)."""
    import torch
    out = {}
    for leg, name, over in (
            ("llama1m", "llama1m", dict(steps=20, warmup=max(16, args.warmup))),
            ("llama128k_q8", "llama128k", dict(q8=True)),
            ("llama1m_q8", "llama1m", dict(steps=20, warmup=max(16, args.warmup), q8=True)),
            ("retopk64k", "retopk64k", dict(steps=512, warmup=args.warmup))):
        torch.cuda.empty_cache()
        sub = argparse.Namespace(**{**vars(args), "workload": name, "cpu_baseline": False,
                                    "trace": False, "device_only": False, "q8": False,
                                    **over})
        r = run_retopk(sub, ws, rank, local) if name.startswith("retopk") else \
            run_ours(sub, ws, rank, local)
        keep = ("value", "unit", "ms_per_step", "steps", "warmup", "config", "stages_ms",
                "path_algorithmic_gbs", "roofline", "e2e", "gpu_launches", "clocks",
                "host_launched_us_per_step", "timing", "paths")
        out[leg] = {k: r[k] for k in keep if k in r}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="llama128k",
                    choices=["tiny", "llama128k", "llama1m", "yi_paged", "retopk64k",
                             "retopk1m", "retopk4m", "retopk_batched"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--trace", action="store_true",
                    help="also record a per-CTA kernel timeline of 3 extra steps")
    ap.add_argument("--device-only", action="store_true",
                    help="profiling mode: time only the device path (no e2e, no baseline)")
    ap.add_argument("--q8", action="store_true",
                    help="decode through the int8 key codes with exact rescoring")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false",
                    help="skip the 1M decode and 64K ReTopK legs of the default run")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
    elif args.workload == "retopk_batched":
        res = run_retopk_batched(args, ws, rank, local) if rank == 0 else None
    elif args.workload.startswith("retopk"):
        res = run_retopk(args, ws, rank, local)
    else:
        res = run_ours(args, ws, rank, local)
        if (args.secondary and ws == 1 and args.workload == "llama128k" and not args.device_only
                and not args.q8 and res is not None):
            res["secondary"] = run_secondary(args, ws, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
