"""Decode-step benchmark: paged decode-step latency and KV-read HBM bandwidth.

Default workload: bs 32, 8192 cached tokens per request, Hq 32 / Hkv 8, head_dim 128,
page_size 64, bf16 K/V (1.07 GB of KV per step, far larger than the 129 MB L2, so no
L2 flush is needed between steps).  One step = fused metadata + split-K producer +
log-sum-exp reducer, replayed from a CUDA graph with PDL.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload NAME]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an independent
replica of the step on its own GPU (the step has no cross-GPU exchange); the reported
time is the maximum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-step µs & KV-read HBM GB/s (frac of ~8 TB/s), bs1–64 ctx1K–16K"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "splitk_traffic.json")
FALLBACK_HBM_GBS = 6800.0
E2E_NOTE = ("inputs and outputs in pinned host memory, host stream sync every step; "
            "zero_copy: the kernels read q / req_pool_indices / seq_lens and write O / LSE "
            "over the host link; copy_engine: pa_decode_step_host_packed, one copy each way; "
            "eager: the C call every step; graph: that call captured once, replayed every step")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # defaults: 5000 / 50 GPU steps; the reference arm (whole oracle steps of ~0.1 s on
    # 16 host cores) defaults to 20 / 3 so that a run without flags ends in seconds
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="bs32_ctx8k")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the PDL study, e2e and CPU baseline")
    ap.add_argument("--profile", action="store_true",
                    help="eager steps only (warm-up + steps launches of each kernel), for ncu")
    ap.add_argument("--producer", default="auto", choices=["auto", "mma", "fma"],
                    help="with --profile: the split-K producer implementation")
    ap.add_argument("--window", action="store_true",
                    help="with --profile: the workload's sliding-window layer step instead")
    ap.add_argument("--all-workloads", action="store_true",
                    help="report table: every named workload, graph with / without PDL and "
                         "eager (one JSON line per workload; not the benchmark line)")
    args = ap.parse_args()
    ref = args.impl == "reference"
    if args.steps is None:
        args.steps = 20 if ref else 5000
    if args.warmup is None:
        args.warmup = 3 if ref else 50
    return args


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def kernel_source_hash():
    """Hash of the producer's sources with comments and blank space removed, so that a
    comment edit does not retire the committed ncu traffic record."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_metadata_gb300", "csrc")
    for name in ("pa_splitk_mma.cuh", "pa_common.cuh", "pa_splitk_mma_config.h",
                 "pa_splitk_mma_bf16.cu", "pa_splitk_mma_int8.cu",
                 "pa_splitk_mma_window_bf16.cu", "pa_splitk_mma_window_int8.cu"):
        with open(os.path.join(csrc, name)) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(l.strip() for l in text.splitlines() if l.strip()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per producer launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        rec = json.load(f)
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, f"t_{which}", time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), sm_max=float(parts[2]),
                                 active=parts[4], hw=parts[5], hw_thermal=parts[6],
                                 sw_thermal=parts[7], sw_power=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["sm_max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "window": "warm-up tail and timed region"}


def oracle_sample_us(wl, tokens, request):
    """Oracle wall time (us) for one request's first `tokens` cached tokens, all heads."""
    import numpy as np
    import torch

    import oracle

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    meta = oracle.build_metadata(wl.req_pool_indices.numpy(), wl.seq_lens.numpy(),
                                 wl.req_to_token.numpy(), wl.spec.seqlen_offset,
                                 wl.max_seq_pages, wl.spec.page_size)
    if wl.spec.kv_dtype == "int8":
        k, v, ks, vs = wl.k_cache.numpy(), wl.v_cache.numpy(), wl.k_scale.numpy(), wl.v_scale.numpy()
    else:
        k, v, ks, vs = bits(wl.k_cache), bits(wl.v_cache), None, None
    n = min(tokens, int(meta["cache_seqlens"][request]))
    q = bits(wl.q)[request:request + 1]
    t0 = time.perf_counter()
    oracle.paged_attention(q, k, v, meta["page_table"][request:request + 1],
                           np.array([n], np.int32), wl.sm_scale, ks, vs)
    return (time.perf_counter() - t0) * 1e6, n


def oracle_step_runner(wl):
    """A callable that runs the oracle, unchanged, over one whole decode step of the
    workload with one request (all its heads) per task on every host core (the oracle's
    C calls release the interpreter lock); returns (callable, threads).  The callable's
    ``pool`` attribute is the thread pool (a context manager)."""
    import concurrent.futures

    import numpy as np
    import torch

    import oracle

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    meta = oracle.build_metadata(wl.req_pool_indices.numpy(), wl.seq_lens.numpy(),
                                 wl.req_to_token.numpy(), wl.spec.seqlen_offset,
                                 wl.max_seq_pages, wl.spec.page_size)
    if wl.spec.kv_dtype == "int8":
        k, v, ks, vs = wl.k_cache.numpy(), wl.v_cache.numpy(), wl.k_scale.numpy(), wl.v_scale.numpy()
    else:
        k, v, ks, vs = bits(wl.k_cache), bits(wl.v_cache), None, None
    q, pt, cl = bits(wl.q), meta["page_table"], meta["cache_seqlens"]
    threads = os.cpu_count() or 1
    pool = concurrent.futures.ThreadPoolExecutor(threads)

    def one(r):
        oracle.paged_attention(q[r:r + 1], k, v, pt[r:r + 1], cl[r:r + 1], wl.sm_scale, ks, vs)

    def run_step():
        list(pool.map(one, range(wl.spec.bs)))
    run_step.pool = pool
    return run_step, threads


def cpu_baseline_all_cores(wl, budget_s=10.0):
    """Whole decode steps of the oracle on every host core (``oracle_step_runner``),
    repeated until ~budget_s of wall time (at least one, at most five).  Returns
    (us per step, threads, steps timed)."""
    run_step, threads = oracle_step_runner(wl)
    with run_step.pool:
        steps, t0 = 0, time.perf_counter()
        while steps == 0 or (time.perf_counter() - t0 < budget_s and steps < 5):
            run_step()
            steps += 1
        wall = time.perf_counter() - t0
    return wall / steps * 1e6, threads, steps


def cpu_baseline(wl, budget_s=10.0):
    """The oracle on the workload's host cores: whole steps with the requests spread over
    every core (the reported value), and, for reference, whole requests one after
    another on one core until ~budget_s of CPU time, scaled to one step."""
    all_us, threads, steps = cpu_baseline_all_cores(wl, budget_s)
    single = cpu_baseline_one_core(wl, budget_s)
    return {"value": all_us, "unit": "us/step", "cores": threads, "kind": "oracle",
            "sample": f"{steps} whole step(s): {wl.spec.bs} requests x {wl.spec.num_q_heads} "
                      f"query heads over {sum(wl.ctx)} cached tokens, one request per task on "
                      f"{threads} threads",
            "single_core": single}


def cpu_baseline_one_core(wl, budget_s=10.0):
    """The oracle on whole requests of the workload (all cached tokens, all heads), one
    request after another until ~budget_s of CPU time; scaled to one full step."""
    total_tokens = sum(wl.ctx)
    spent, sampled, used = 0.0, 0, 0
    while spent < budget_s * 1e6 and used < 4 * wl.spec.bs:
        us, n = oracle_sample_us(wl, 1 << 30, used % wl.spec.bs)
        spent += us
        sampled += n
        used += 1
    per_step_us = spent / sampled * total_tokens
    return {"value": per_step_us, "unit": "us/step", "cores": 1, "kind": "oracle",
            "sample": f"{used} whole requests ({sampled} cached tokens x "
                      f"{wl.spec.num_q_heads} query heads, {spent / 1e6:.1f} s on one core); "
                      f"scaled to the step's {total_tokens} tokens"}


def max_over_ranks(value, world, device="cpu"):
    """The largest of each rank's `value` (every rank gets it); `value` on one rank.
    Uses the default process group, so `device` must suit its backend (cuda for nccl,
    cpu for gloo)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, spec, rank, world):
    """The oracle as the reference arm: every step is one whole decode step of the
    workload (all requests, all heads, every cached token), the requests spread over
    every host core, timed as it stands.  Rank 0 alone runs it."""
    if rank != 0:
        return
    from paged_kv_decode_metadata_gb300 import synthetic

    wl = synthetic.make(spec)
    run_step, threads = oracle_step_runner(wl)
    with run_step.pool:
        for _ in range(max(1, args.warmup)):
            run_step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            run_step()
        wall = time.perf_counter() - t0
    per_step_us = wall / args.steps * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": per_step_us, "unit": "us/step",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step_us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(spec, wl),
        "cpu_baseline": {"value": per_step_us, "unit": "us/step", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{args.steps} whole step(s) after {max(1, args.warmup)} "
                                   f"warm-up: {spec.bs} requests x {spec.num_q_heads} query "
                                   f"heads over {sum(wl.ctx)} cached tokens, one request per "
                                   f"task on {threads} threads"},
        "e2e": {"value": per_step_us, "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(spec, wl):
    """The workload (the same dict on the GPU line and the reference arm's line)."""
    cfg = {"workload": spec.name, "bs": spec.bs,
           "ctx": spec.ctx if spec.ragged is None else f"U[{spec.ragged[0]},{spec.ragged[1]}]",
           "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads,
           "head_dim": spec.head_dim, "page_size": spec.page_size, "kv_dtype": spec.kv_dtype,
           "seqlen_offset": spec.seqlen_offset}
    if spec.swa_window is not None:
        cfg["swa_window"] = spec.swa_window
    kv_gb = sum(wl.ctx) * spec.num_kv_heads * 2 * spec.head_dim * (
        1 if spec.kv_dtype == "int8" else 2) / 1e9
    cfg["l2"] = "inputs larger than L2: %.2f GB of KV per step, no flush" % kv_gb
    return cfg


def time_graph(torch, graph, n, stream):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(n):
            graph.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / n * 1e3  # us


def capture(torch, fn, stream):
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn()
    torch.cuda.synchronize()
    return graph


def pdl_study(torch, synthetic, DeviceStep, stream, replays=300, steps_per_graph=16):
    """Batch-1 decode-step latency with and without PDL.  One CUDA graph holds
    `steps_per_graph` consecutive steps (48 kernels), so graph-launch overhead on the
    host is amortised and the time per step is the GPU's, including the step-to-step
    hand-off; eager: back-to-back C-ABI calls."""
    out = {}
    for name in ("bs1_ctx1k", "bs1_ctx8k"):
        wl = synthetic.make(synthetic.WORKLOADS[name])
        ds = DeviceStep(wl)
        row = {}
        for pdl in (False, True):
            def steps(pdl=pdl):
                for _ in range(steps_per_graph):
                    ds.step(use_pdl=pdl)
            g = capture(torch, steps, stream)
            for _ in range(3):
                time_graph(torch, g, 20, stream)
            row["graph_pdl_us" if pdl else "graph_us"] = statistics.median(
                time_graph(torch, g, replays, stream) for _ in range(5)) / steps_per_graph
            del g
            with torch.cuda.stream(stream):
                for _ in range(50):
                    ds.step(use_pdl=pdl)
                start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                start.record(stream)
                for _ in range(500):
                    ds.step(use_pdl=pdl)
                end.record(stream)
            end.synchronize()
            row["eager_pdl_us" if pdl else "eager_us"] = start.elapsed_time(end) / 500 * 1e3
        row["num_splits"] = ds.num_splits
        row["steps_per_graph"] = steps_per_graph
        out[name] = row
        del ds
    return out


def pdl_gap_study(torch, synthetic, DeviceStep, binding, stream, reps=300):
    """Inter-stage gaps of one decode step from the timestamp-instrumented build: each
    kernel records its earliest block entry, earliest return from griddepcontrol.wait
    and latest warp finish (%globaltimer).  One step at a time, graph replay, with and
    without PDL; medians over `reps` steps, nanoseconds."""
    import numpy as np

    lib = binding.load_instrumented()
    buf = torch.empty(9, dtype=torch.int64, device="cuda")
    init = torch.tensor([-1, -1, 0] * 3, dtype=torch.int64, device="cuda")  # UINT64_MAX / 0
    if lib.pa_set_timestamp_buffer(buf.data_ptr()) != 0:
        raise RuntimeError("pa_set_timestamp_buffer failed")
    result = {}
    try:
        for name in ("bs1_ctx1k", "bs1_ctx8k"):
            wl = synthetic.make(synthetic.WORKLOADS[name])
            ds = DeviceStep(wl)
            row = {}
            for pdl in (False, True):
                g = capture(torch, lambda: ds.step(use_pdl=pdl, lib=lib), stream)
                rec = []
                for _ in range(reps):
                    with torch.cuda.stream(stream):
                        buf.copy_(init)
                        g.replay()
                    stream.synchronize()
                    rec.append(buf.cpu().numpy().view(np.uint64).astype(np.float64))
                del g
                r = np.median(np.stack(rec), axis=0)
                e0, w0, x0, e1, w1, x1, e2, w2, x2 = r
                key = "pdl" if pdl else "no_pdl"
                row[key] = {
                    "step_ns": x2 - e0,
                    "metadata_ns": x0 - e0,
                    "producer_ns": x1 - w1,
                    "reducer_ns": x2 - w2,
                    "gap_metadata_to_producer_ns": w1 - x0,
                    "gap_producer_to_reducer_ns": w2 - x1,
                    "producer_resident_before_metadata_end_ns": x0 - e1,
                    "reducer_resident_before_producer_end_ns": x1 - e2,
                }
            result[name] = row
            del ds
    finally:
        lib.pa_set_timestamp_buffer(None)
    return result


def run_gb300(args, spec, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from paged_kv_decode_metadata_gb300 import binding, synthetic
    from paged_kv_decode_metadata_gb300 import build as pa_build
    from paged_kv_decode_metadata_gb300.runtime import DeviceStep

    if rank == 0:
        pa_build.build()
        if not args.no_extras:
            pa_build.build(instrumented=True)
    if world > 1:
        dist.barrier()
    torch.cuda.set_device(local_rank)
    binding.load()
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))

    wl = synthetic.make(spec)
    ds = DeviceStep(wl)
    stream = torch.cuda.Stream()
    binding.pa_read_error_flags(reset=True)
    # One graph holds several consecutive steps (PDL chains each step's kernels to the
    # previous step's, as consecutive layers of a model graph would), so the time per
    # step is the GPU's and not the host's graph-launch rate.  K is timed exactly:
    # the steps per graph divide K.
    per_graph = next(n for n in (8, 4, 2, 1) if args.steps % n == 0)

    def steps():
        for _ in range(per_graph):
            ds.step(use_pdl=True)
    graph = capture(torch, steps, stream)
    if binding.pa_read_error_flags(reset=True):
        raise RuntimeError("device error flags set during warm-up")

    sampler = ClockSampler(local_rank)
    if rank == 0:
        sampler.start()
        time.sleep(1.0)
    for _ in range(-(-max(3, args.warmup) // per_graph)):
        graph.replay()
    # keep the GPU busy for ~1.5 s so the clock samples see the loaded state
    t_end = time.time() + 1.5
    while time.time() < t_end:
        for _ in range(max(1, 200 // per_graph)):
            graph.replay()
        torch.cuda.synchronize()

    # ---- timed region: exactly K steps ------------------------------------------------
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark("start")
    us_step = time_graph(torch, graph, args.steps // per_graph, stream) / per_graph
    torch.cuda.synchronize()
    sampler.mark("stop")
    if world > 1:
        dist.barrier()
    us_step = max_over_ranks(us_step, world, "cuda")
    clocks = sampler.stop() if rank == 0 else None

    # ---- dominant kernel alone: the split-K producer, CUDA events on its stream -------
    n_kernel = max(20, min(args.steps, 500))
    splitk_us = producer_launch_us(torch, ds, stream, n_kernel)
    producer_alt = {}
    if spec.num_q_heads // spec.num_kv_heads <= 8:
        with binding.producer(binding.PA_PRODUCER_FMA):
            producer_alt["fma_us"] = producer_launch_us(torch, ds, stream, n_kernel)

    kv_bytes = ds.kv_bytes(wl.ctx)
    splitk_bytes = producer_bytes(ds, wl, [-(-int(n) // spec.page_size) for n in wl.ctx])
    achieved = splitk_bytes / (splitk_us * 1e-6) / 1e9
    traffic = ncu_traffic(spec.name)
    step_bytes = ds.step_bytes(wl.ctx)

    extras = {}
    if rank == 0 and not args.no_extras:
        # ---- end to end through the public C ABI with the step's inputs and outputs in
        # pinned host memory (see e2e_us)
        extras["e2e"] = e2e_record(torch, ds, stream, max(20, min(args.steps, 2000)))
        # ---- same graph without PDL, and the batch-1 PDL study -------------------------
        def steps_nopdl():
            for _ in range(per_graph):
                ds.step(use_pdl=False)
        g_nopdl = capture(torch, steps_nopdl, stream)
        extras["graph_no_pdl_us"] = time_graph(
            torch, g_nopdl, max(1, min(args.steps, 2000) // per_graph), stream) / per_graph
        del g_nopdl
        extras["pdl_bs1"] = pdl_study(torch, synthetic, DeviceStep, stream)
        extras["pdl_gaps_bs1"] = pdl_gap_study(torch, synthetic, DeviceStep, binding, stream)
        # ---- every other workload of the path: graph +/- PDL, eager, L2-rotated for the
        # small ones; the int8 batch and its sliding-window layer with their producer
        # roofline (and the int8 batch end to end)
        l2_bytes = torch.cuda.get_device_properties(local_rank).L2_cache_size
        table = []
        for name, window in all_rows(synthetic):
            if name == spec.name and not window:
                continue
            big = synthetic.WORKLOADS[name].kv_dtype == "int8"
            table.append(measure_workload(torch, name, window, stream, args.steps, hbm_peak,
                                          peak_kind, l2_bytes, with_producer=big,
                                          with_e2e=big and not window))
        extras["workloads"] = table
        extras["cpu_baseline"] = cpu_baseline(wl)

    flags = binding.pa_read_error_flags(reset=True)
    if flags:
        raise RuntimeError(f"device error flags 0x{flags:x}")
    if rank != 0:
        return
    kv_gbs = kv_bytes / (us_step * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": us_step, "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us_step / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if spec.kv_dtype == "bf16" else "int8", "data": "synthetic",
        "config": workload_config(spec, wl),
        "method": {"num_splits": ds.num_splits, "pdl": True, "cuda_graph": True,
                   "steps_per_graph": per_graph,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "kv_hbm_gbs": kv_gbs, "kv_hbm_frac": kv_gbs / hbm_peak,
        "step_hbm_gbs": step_bytes / (us_step * 1e-6) / 1e9,
        "producer_cuda_core_fma_us": producer_alt.get("fma_us"),
        "roofline": {"bound": "hbm", "kernel": "splitk_mma_kernel", "achieved": achieved,
                     "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": splitk_bytes, "launch_us": splitk_us},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    line.update({k: v for k, v in extras.items() if k not in ("cpu_baseline",)})
    line["cpu_baseline"] = extras.get("cpu_baseline")
    print(json.dumps(line), flush=True)


def producer_launch_us(torch, ds, stream, n):
    """Average duration of one split-K producer launch: n eager launches without PDL
    between CUDA events on the launching stream (the metadata stage runs first, once)."""
    with torch.cuda.stream(stream):
        ds.metadata(use_pdl=False)
        for _ in range(5):
            ds.splitk(use_pdl=False)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(n):
            ds.splitk(use_pdl=False)
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / n * 1e3


def producer_bytes(ds, wl, pages_read):
    """Algorithmic bytes of one producer launch: KV (+ int8 scales) of the attended
    tokens, Q read, partials written, page-table entries and lengths read."""
    spec = wl.spec
    rows = spec.bs * spec.num_q_heads
    return (ds.kv_bytes(wl.ctx) + rows * spec.head_dim * 2
            + rows * ds.num_splits * (spec.head_dim + 2) * 4
            + spec.bs * 4 + sum(pages_read) * 4)


def e2e_us(torch, ds, stream, n):
    """End to end with the step's inputs (q, req_pool_indices, seq_lens) and outputs (O,
    LSE) in pinned host memory, a host stream sync every step, n steps.  Four ways a
    caller drives it: the kernels reading and writing the host buffers directly over the
    host link (pa_decode_step on pinned pointers), eager and as one CUDA graph replayed
    every step; and pa_decode_step_host_packed (one copy in, the kernels, one copy
    out on the copy engines), eager and graph-replayed.  Each replay reads the host
    inputs as they are then and writes the host outputs.  Returns (dict of us per step,
    h2d bytes, d2h bytes); the bytes are those of the host tensors."""
    h_in, h_outs, (h_q, h_rpi, h_sl, h_out, h_lse) = ds.host_buffers()
    h_q.copy_(ds.q)
    h_rpi.copy_(ds.req_pool_indices)
    h_sl.copy_(ds.seq_lens)

    def per_step(fn):
        with torch.cuda.stream(stream):  # (a graph replay runs on the current stream)
            for _ in range(20):
                fn()
                stream.synchronize()
            t0 = time.perf_counter()
            for _ in range(n):
                fn()
                stream.synchronize()
            return (time.perf_counter() - t0) / n * 1e6

    out = {}
    for key, call in (
            ("zero_copy", ds.prepare_host_io_step(h_in, h_outs, use_pdl=True, stream=stream)),
            ("copy_engine", ds.prepare_packed_host_step(h_in, h_outs, use_pdl=True,
                                                        stream=stream))):
        out[key + "_eager_us"] = per_step(call)
        graph = capture(torch, call, stream)
        out[key + "_graph_us"] = per_step(graph.replay)
        del graph
    h2d = h_q.numel() * 2 + h_sl.numel() * 8 + h_rpi.numel() * 8
    d2h = h_out.numel() * 2 + h_lse.numel() * 4
    return out, h2d, d2h


def e2e_record(torch, ds, stream, n):
    """The bench line's e2e object: the value is the zero-copy step replayed from a CUDA
    graph (how a serving loop drives the step: the kernels move the host inputs and
    outputs themselves); the other three ways of e2e_us beside it."""
    ways, h2d, d2h = e2e_us(torch, ds, stream, n)
    return {"value": ways["zero_copy_graph_us"], "unit": "us/step", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "method": "zero_copy_graph", **ways, "note": E2E_NOTE}


def measure_workload(torch, name, window, stream, steps, hbm_peak, peak_kind, l2_bytes,
                     with_producer=False, with_e2e=False):
    """One workload's decode step: CUDA graphs holding 8 consecutive steps (so the time
    per step is the GPU's, not the host's graph-launch rate), with and without PDL, and
    eager C-ABI calls with PDL.  Steps whose bytes fit in 2x the 129 MB L2 are also
    timed with the inputs rotated over enough copies to exceed 2x L2 (one graph stepping
    through every copy in turn).  with_producer: the producer launch alone and its
    roofline; with_e2e: the end-to-end step with host-memory inputs and outputs (e2e_us)."""
    from paged_kv_decode_metadata_gb300 import binding, synthetic
    from paged_kv_decode_metadata_gb300.runtime import DeviceStep, WindowStep

    spec = synthetic.WORKLOADS[name]
    if window:
        wl = synthetic.make(spec, with_cache=False, with_swa_cache=True)
        make_step = lambda: WindowStep(wl)  # noqa: E731
    else:
        wl = synthetic.make(spec)
        make_step = lambda: DeviceStep(wl)  # noqa: E731
    ds = make_step()
    per_graph = 8
    label = name + (f" window {spec.swa_window}" if window else "")
    row = {"workload": label, "num_splits": ds.num_splits, "steps_per_graph": per_graph}
    reps = max(20, min(steps, 2000) // per_graph)
    for pdl in (False, True):
        def run(pdl=pdl):
            for _ in range(per_graph):
                ds.step(use_pdl=pdl)
        g = capture(torch, run, stream)
        time_graph(torch, g, 5, stream)
        row["graph_pdl_us" if pdl else "graph_us"] = statistics.median(
            time_graph(torch, g, reps, stream) for _ in range(5)) / per_graph
        del g
    n = max(200, min(steps, 2000))
    with torch.cuda.stream(stream):
        for _ in range(20):
            ds.step(use_pdl=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            ds.step(use_pdl=True)
        b.record(stream)
    b.synchronize()
    row["eager_pdl_us"] = a.elapsed_time(b) / n * 1e3
    footprint = ds.step_bytes(wl.ctx)
    if footprint < 2 * l2_bytes:
        copies = int(2 * l2_bytes // footprint) + 1
        others = [make_step() for _ in range(copies - 1)]
        everyone = [ds] + others

        def rotate():
            for d in everyone:
                d.step(use_pdl=True)
        g = capture(torch, rotate, stream)
        time_graph(torch, g, 2, stream)
        row["graph_pdl_l2_rotated_us"] = statistics.median(
            time_graph(torch, g, max(5, reps // copies), stream) for _ in range(5)) / copies
        row["l2_rotation_copies"] = copies
        del g, others, everyone
    best = row.get("graph_pdl_l2_rotated_us", row["graph_pdl_us"])
    row["kv_bytes"] = ds.kv_bytes(wl.ctx)
    row["step_bytes"] = footprint
    row["kv_gbs"] = row["kv_bytes"] / (best * 1e-6) / 1e9
    row["kv_frac"] = row["kv_gbs"] / hbm_peak
    if with_producer:
        us = producer_launch_us(torch, ds, stream, max(20, min(steps, 500)))
        P = spec.page_size
        if window:   # pages holding the window's positions n - v .. n - 1
            pages = [(n - 1) // P - (n - v) // P + 1 if v > 0 else 0
                     for n, v in zip(map(int, wl.ctx), ds.visible_tokens(wl.ctx))]
        else:
            pages = [-(-int(n) // P) for n in wl.ctx]
        nbytes = producer_bytes(ds, wl, pages)
        achieved = nbytes / (us * 1e-6) / 1e9
        row["roofline"] = {"bound": "hbm", "kernel": "splitk_mma_kernel", "achieved": achieved,
                           "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
                           "frac": achieved / hbm_peak, "traffic": ncu_traffic(label),
                           "algorithmic_bytes_per_launch": nbytes, "launch_us": us}
    if with_e2e:
        row["e2e"] = e2e_record(torch, ds, stream, max(20, min(steps, 2000)))
    if binding.pa_read_error_flags(reset=True):
        raise RuntimeError("device error flags set")
    del ds
    torch.cuda.empty_cache()
    return row


def run_table(args):
    """Per-workload latency table, one JSON line per workload (not the benchmark line)."""
    import torch

    from paged_kv_decode_metadata_gb300 import binding, synthetic
    from paged_kv_decode_metadata_gb300 import build as pa_build

    pa_build.build()
    binding.load()
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    stream = torch.cuda.Stream()
    l2_bytes = torch.cuda.get_device_properties(0).L2_cache_size
    for name, window in all_rows(synthetic):
        print(json.dumps(measure_workload(torch, name, window, stream, args.steps, hbm_peak,
                                          peak_kind, l2_bytes, with_producer=True)), flush=True)


def all_rows(synthetic):
    """Every named workload, then the sliding-window layer of those that have one."""
    rows = [(n, False) for n in synthetic.WORKLOAD_ORDER]
    rows += [(n, True) for n in synthetic.WORKLOAD_ORDER
             if synthetic.WORKLOADS[n].swa_window is not None]
    return rows


def run_profile(args, spec):
    """Plain eager decode steps with no timing, sampling or extras: the command that
    ncu captures.  Kernel launch order per step: metadata, split-K producer, reducer."""
    import torch

    from paged_kv_decode_metadata_gb300 import binding, synthetic
    from paged_kv_decode_metadata_gb300 import build as pa_build
    from paged_kv_decode_metadata_gb300.runtime import DeviceStep

    pa_build.build()
    binding.load()
    if args.window:
        from paged_kv_decode_metadata_gb300.runtime import WindowStep
        wl = synthetic.make(spec, with_cache=False, with_swa_cache=True)
        ds = WindowStep(wl)
    else:
        wl = synthetic.make(spec)
        ds = DeviceStep(wl)
    which = {"auto": binding.PA_PRODUCER_AUTO, "mma": binding.PA_PRODUCER_MMA,
             "fma": binding.PA_PRODUCER_FMA}[args.producer]
    with binding.producer(which):
        for _ in range(args.warmup + args.steps):
            ds.step(use_pdl=True)
    torch.cuda.synchronize()
    flags = binding.pa_read_error_flags(reset=True)
    if flags:
        raise RuntimeError(f"device error flags 0x{flags:x}")
    print(json.dumps({"profile": spec.name + (" window" if args.window else ""),
                      "steps": args.warmup + args.steps, "num_splits": ds.num_splits}))


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from paged_kv_decode_metadata_gb300 import synthetic

    spec = synthetic.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, spec, rank, world)
        return
    if args.profile:
        run_profile(args, spec)
        return
    if args.all_workloads:
        run_table(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_gb300(args, spec, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
