"""Benchmark of the single-token KV-cache decode step (append + decode attention, every layer).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-graph]

Prints ONE JSON line on rank 0.  A step = one decode step of the whole model: for each of the
workload's layers one fused kvc_decode_step (append the new token, attend over the history).
The metric is the decode-attention KV-read bandwidth, 2 * H_kv * D * s * sum_b L_b bytes per
layer, divided by the step time.  Inputs are synthetic (counter-based generator), resident in
HBM, and larger than L2 (every layer has its own cache).

--impl reference times the CPU oracle (the plain C, fp64 restatement of the pages) on the
host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn KV-read GB/s (% of GB300 HBM peak) and µs/step, 8B-GQA B=24"
NOMINAL_HBM_GBS = 8000.0


def _env_int(k, d):
    try:
        return int(os.environ.get(k, d))
    except ValueError:
        return d


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle arm
def oracle_sample(w, budget_s: float, threads: int, max_layers: int | None = None):
    """Times the oracle on whole layers of the workload until budget_s is used (at least one
    layer).  Returns (GB/s of algorithmic KV read, layers done, seconds, threads used)."""
    import numpy as np
    import torch

    import oracle
    from kv_cache_decode_kvc_gb300 import synth

    used = oracle.set_threads(threads)
    # the generator gives identical values on any device; the GPU makes them faster
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    lens = w.lens()
    lens_np = lens.numpy()
    done, secs, nbytes = 0, 0.0, 0
    layers = w.layers if max_layers is None else min(w.layers, max_layers)
    for layer in range(layers):
        # the post-append cache of this layer is the generator's rows [0, L_b) of each stream
        T_max = int(lens.max())
        K = synth.bf16_bits(synth.block(w.seed, layer, "K", 0, w.B, w.H_kv, 0, T_max, w.D, w.B,
                                        device=gen_dev).cpu())
        V = synth.bf16_bits(synth.block(w.seed, layer, "V", 0, w.B, w.H_kv, 0, T_max, w.D, w.B,
                                        device=gen_dev).cpu())
        q = synth.bf16_bits(synth.queries(w.seed, layer, w.B, w.H_q, w.D, device=gen_dev).cpu())
        t0 = time.perf_counter()
        oracle.decode_attn(q, K, V, lens_np)
        secs += time.perf_counter() - t0
        nbytes += w.kv_read_bytes_per_layer()
        done += 1
        if secs >= budget_s:
            break
    return nbytes / secs / 1e9, done, secs, used


def run_reference(args, w):
    rank = _env_int("RANK", 0)  # under torchrun only rank 0 runs the CPU arm
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    per_step = []
    for i in range(args.warmup + args.steps):
        gbs, layers, secs, used = oracle_sample(w, budget_s=0.0, threads=threads, max_layers=1)
        if i >= args.warmup:
            per_step.append((gbs, secs))
    gbs = statistics.median(g for g, _ in per_step)
    sample = f"layer 0 of {w.name} (all {w.B} sequences x {w.H_q} query heads) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(s for _, s in per_step), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- GPU arm
def traffic_from_profiles(kernel_src_hash: str, paged: int = 0):
    """DRAM bytes per launch of the decode kernel from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    name = f"decode_kernel_gqa8b_b24_paged{paged}.md" if paged else "decode_kernel_gqa8b_b24.md"
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path, encoding="utf-8"):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_src_hash:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def kernel_source_hash():
    """Hash of the CUDA sources with comments and whitespace removed: an edit to a comment does
    not invalidate a profile, any change to the code does."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_decode_kvc_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)  # block comments
        text = re.sub(r"//[^\n]*", " ", text)                # line comments (no '//' in strings)
        h.update(f.encode() + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    from kv_cache_decode_kvc_gb300 import kvc
    from kv_cache_decode_kvc_gb300.replicas import env_rank, max_over_ranks, replica_seed, whole_job_rate
    from kv_cache_decode_kvc_gb300.workloads import fill_layer, paged_table, step_inputs, step_inputs_multi

    rank, local, world = env_rank()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    kvc.load()  # fails loudly without the CUDA library

    def barrier():
        if world > 1:
            dist.barrier()

    seed = replica_seed(w.seed, rank)  # each replica decodes its own batch (weak scaling)
    L = w.layers
    table_d = None
    if args.paged:
        # the same sequences in a paged pool: block_size-token blocks at shuffled pool positions
        table, num_blocks, max_blocks = paged_table(w, args.paged, spare=w.B)
        cache = kvc.PagedKVCache(L, num_blocks, args.paged, w.B, max_blocks, w.H_q, w.H_kv, w.D, w.dtype)
        table_d = table.to(dev)
    elif args.int8 or args.fp8:
        # int8 or fp8 (E4M3) cache with one fp32 scale per (sequence, head, token) row; q / out /
        # new rows bf16
        cache = kvc.QuantKVCache(L, w.B, w.H_q, w.H_kv, w.D, w.T_max(), fp8=args.fp8)
    elif args.window:
        # sliding-window attention: a rolling cache of `window` slots per sequence
        cache = kvc.RollingKVCache(L, w.B, w.H_q, w.H_kv, w.D, args.window, w.dtype)
    else:
        # room for the step's new tokens (one, or --tq of them)
        cache = kvc.KVCache(L, w.B, w.H_q, w.H_kv, w.D, w.T_max() + args.tq - 1, w.dtype)
    # the launch preceding each decode launch is the previous layer's decode step, which writes
    # neither lens nor this layer's history rows: early history loads are allowed
    cache.set_launch_overlap(0 if args.no_overlap else 1)
    t_fill = time.perf_counter()
    for layer in range(L):
        fill_layer(cache, layer, w, seed=seed, table=table_d)
    if args.tq > 1:  # several new tokens per sequence and step (speculative decoding)
        ins = [step_inputs_multi(w, layer, args.tq, seed=seed) for layer in range(L)]
        outs = [torch.empty(w.B, w.H_q, args.tq, w.D, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    else:
        ins = [step_inputs(w, layer, seed=seed) for layer in range(L)]
        outs = [torch.empty(w.B, w.H_q, w.D, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    lens_d = (w.lens_pre() + args.tq).to(dev)
    torch.cuda.synchronize()
    t_fill = time.perf_counter() - t_fill
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream

    def decode(layer, q, kn, vn, out, lens):
        if args.tq > 1:
            kvc.kvc_decode_step_multi(cache.h, layer, q, kn, vn, out, lens, args.tq, sptr)
        elif table_d is None:
            kvc.kvc_decode_step(cache.h, layer, q, kn, vn, out, lens, sptr)
        else:
            kvc.kvc_paged_decode_step(cache.h, layer, q, kn, vn, out, table_d, lens, sptr)

    def step():
        for layer in range(L):
            q, kn, vn = ins[layer]
            decode(layer, q, kn, vn, outs[layer], lens_d)

    # the automatic merge path adds a combine kernel per layer when streams are few and long
    # (same rule as the library: segments per stream x group outputs above 64 KB)
    P, U = kvc.kvc_get_ctas(cache.h), w.B * w.H_kv
    nseg = (P + U - 1) // U + 1
    launches_per_step = 2 * L if nseg * w.G * w.D * 4 > 65536 else L

    graph = None
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step()
        stream.synchronize()
        if not args.no_graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                step()
            for _ in range(args.warmup):
                graph.replay()
        stream.synchronize()
    st, detail = cache.last_error(sptr)
    if st != kvc.KVC_OK:
        raise RuntimeError(f"device error during warm-up: status {st} detail {detail:#x}")

    run = graph.replay if graph is not None else step

    # ---- the same steps launched eagerly (no graph), for the eager step time beside the graph's
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        ee0, ee1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ee0.record(stream)
        for _ in range(args.steps):
            step()
        ee1.record(stream)
    torch.cuda.synchronize()
    eager_ms = ee0.elapsed_time(ee1) / args.steps

    # ---- timed region: K steps, barrier + synchronize on both sides, CUDA events on `stream`
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(vis.split(",")[local] if vis else str(local))
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed_region")
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            run()
        ev1.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier()
    clock_info = clocks.stop()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms = max_over_ranks(ms_local, world, dev)
    st, detail = cache.last_error(sptr)
    if st != kvc.KVC_OK:
        raise RuntimeError(f"device error in the timed region: status {st} detail {detail:#x}")

    quant = args.int8 or args.fp8  # 8-bit codes + a 4-byte scale per row
    kv_bytes_step = L * w.kv_read_bytes_per_layer(args.window, args.tq, quant)
    gbs = whole_job_rate(world, kv_bytes_step, ms)
    peak, peak_kind = measured_peaks()

    # ---- per-launch durations of the decode kernel (events around each launch, same stream)
    per_launch = []
    with torch.cuda.stream(stream):
        evs = []
        for _ in range(max(1, min(args.steps, 5))):
            for layer in range(L):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                q, kn, vn = ins[layer]
                decode(layer, q, kn, vn, outs[layer], lens_d)
                b.record(stream)
                evs.append((a, b))
    torch.cuda.synchronize()
    per_launch = [a.elapsed_time(b) for a, b in evs]
    launch_ms = statistics.mean(per_launch)
    B, Hq, Hkv, D, s = w.B, w.H_q, w.H_kv, w.D, w.elem_bytes
    T_q = args.tq
    alg_bytes_launch = (w.kv_read_bytes_per_layer(args.window, T_q, quant) + 2 * B * Hq * T_q * D * s
                        + 2 * B * Hkv * T_q * D * s  # k/v new read
                        + 2 * B * Hkv * T_q * (D + 4 if quant else D * s) + 4 * B)  # written, lens
    if args.paged:  # each block-table entry a sequence uses, read once
        alg_bytes_launch += 4 * sum(-(-int(x) // args.paged) for x in w.lens().tolist())
    # average decode-launch duration over the timed region (graph replay, gaps included; a layer
    # whose split streams are merged by a separate combine launch counts both launches)
    region_launch_ms = ms_local / L
    achieved = alg_bytes_launch / (region_launch_ms * 1e-3) / 1e9
    # the committed summaries are captures of the 8B-GQA workload (plain, or paged): another
    # workload, layer count or mode has no measured traffic
    profiled = (w.name == "gqa8b_b24_ragged3000_6000" and not (args.window or args.tq > 1 or quant))
    traffic = traffic_from_profiles(kernel_source_hash(), args.paged) if profiled else None
    path = kvc.kvc_get_math(cache.h)
    kernel_name = {1: f"decode_kernel<{w.dtype},{w.D},{w.G}> (CUDA cores)",
                   2: f"decode_tc_kernel<{w.D},{w.G}> (mma.sync)",
                   3: f"decode_tc5_kernel<{w.G}, {'paged' if args.paged else 'int8' if args.int8 else 'fp8' if args.fp8 else 'rolling' if args.window else 'contiguous'}> (tcgen05)"}[path]

    # ---- end to end through the C ABI with host buffers: each step copies its inputs (lens and
    # every layer's q, k_new, v_new, packed in one pinned buffer) host -> device in one copy,
    # runs the layers, and copies every layer's output device -> host in one copy
    parts = [lens_d] + [t for i in ins for t in i]
    nbytes = [t.numel() * t.element_size() for t in parts]
    offs, o = [], 0
    for nb in nbytes:
        offs.append(o)
        o += -(-nb // 256) * 256  # 256-byte aligned pieces
    h_in = torch.empty(o, dtype=torch.uint8).pin_memory()
    for t, off, nb in zip(parts, offs, nbytes):
        h_in[off: off + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
    d_in = torch.empty(o, dtype=torch.uint8, device=dev)
    views = [d_in[off: off + nb].view(t.dtype).view(t.shape) for t, off, nb in zip(parts, offs, nbytes)]
    d_lens, d_ins = views[0], [views[1 + 3 * l: 4 + 3 * l] for l in range(L)]
    d_out = torch.empty((L,) + tuple(outs[0].shape), dtype=torch.bfloat16, device=dev)
    h_out = torch.empty(d_out.shape, dtype=torch.bfloat16).pin_memory()
    h2d, d2h = o, h_out.numel() * h_out.element_size()

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        for layer in range(L):
            q, kn, vn = d_ins[layer]
            decode(layer, q, kn, vn, d_out[layer], d_lens)
        h_out.copy_(d_out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
        stream.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        stream.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_gbs = whole_job_rate(world, kv_bytes_step, e2e_ms)
    st, detail = cache.last_error(sptr)
    if st != kvc.KVC_OK:
        raise RuntimeError(f"device error in the e2e region: status {st} detail {detail:#x}")

    # ---- CPU baseline: the oracle on the host cores, rank 0 at N=1 only
    cpu = None
    plain = not (args.paged or args.window or args.tq > 1 or quant)  # the oracle arm's workload
    if rank == 0 and world == 1 and not args.no_cpu_baseline and plain:
        threads = os.cpu_count() or 1
        cgbs, layers_done, secs, used = oracle_sample(w, budget_s=args.cpu_budget, threads=threads)
        one_gbs, _, one_secs, _ = oracle_sample(w, budget_s=0.0, threads=1, max_layers=1)
        cpu = {"value": round(cgbs, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
               "sample": f"{layers_done} whole layer(s) of {w.name} ({secs:.1f} s of oracle time, "
                         f"{used} threads)",
               "single_thread": {"value": round(one_gbs, 4), "unit": "GB/s",
                                 "sample": f"layer 0 of {w.name} on 1 thread ({one_secs:.1f} s)"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "us_per_step": round(ms * 1e3, 1), "pct_of_hbm_peak": round(100 * gbs / world / peak, 2),
            "pct_of_nominal_8tbs": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
            "attn_tokens_per_s": round(world * w.B / (ms * 1e-3), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (counter-based generator, bf16)",
            "config": {"workload": w.name + (f", paged cache, {args.paged}-token blocks" if args.paged else "")
                                   + (f", rolling cache, window {args.window}" if args.window else "")
                                   + (f", {args.tq} new tokens per step" if args.tq > 1 else "")
                                   + (", int8 cache with per-row fp32 scales" if args.int8 else "")
                                   + (", fp8 (E4M3) cache with per-row fp32 scales" if args.fp8 else ""),
                       "layers": L, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv,
                       "D": w.D, "lens": (f"U{{{w.T_lo}..{w.T_hi}}}+1 seed {w.seed}" if w.T is None else f"{w.T}+1"),
                       "kv_bytes_per_step": kv_bytes_step,
                       "l2": "inputs larger than L2 (each layer has its own cache; "
                             f"{kv_bytes_step / 1e9:.1f} GB read per step)",
                       "cuda_graph": graph is not None, "launch_overlap": cache.launch_overlap(),
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                         "kernel": kernel_name, "launch_us": round(region_launch_ms * 1e3, 2),
                         "launch_us_eager_events": round(launch_ms * 1e3, 2),
                         "eager_ms_per_step": round(eager_ms, 4),
                         "alg_bytes_per_launch": alg_bytes_launch},
            "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                    "copies_per_step": {"h2d": 1, "d2h": 1}, "launch": "eager"},
            "eager_ms_per_step": round(eager_ms, 4),
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clock_info,
            "cpu_baseline": cpu,
            "setup_s": round(t_fill, 1),
        }
        print(json.dumps(line), flush=True)
    cache.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--paged", type=int, default=0, choices=[0, 16, 32, 64, 128, 256],
                    help="run the workload from a paged cache with this block size (0: contiguous)")
    ap.add_argument("--int8", action="store_true",
                    help="int8 cache with per-row fp32 scales (quantized on write)")
    ap.add_argument("--fp8", action="store_true",
                    help="fp8 (E4M3) cache with per-row fp32 scales (quantized on write)")
    ap.add_argument("--tq", type=int, default=1, choices=[1, 2, 4, 8],
                    help="new tokens per sequence and step (speculative decoding; 1: plain decode)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window attention over a rolling cache of this many slots (0: off)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch overlap off: nothing is read before the preceding launch ends")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=None,
                    help="run only this many layers of the workload (profiling of small cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.paged and args.window:
        ap.error("--paged and --window are separate cache kinds")
    if args.tq > 1 and (args.paged or args.window):
        ap.error("--tq runs on the contiguous cache")
    if (args.int8 or args.fp8) and (args.paged or args.window or args.tq > 1):
        ap.error("--int8 / --fp8 run on the contiguous cache with one new token")
    if args.int8 and args.fp8:
        ap.error("--int8 and --fp8 are separate cache kinds")
    from kv_cache_decode_kvc_gb300.workloads import HEADLINE, WORKLOADS
    w = WORKLOADS[args.workload or HEADLINE]
    if args.layers:
        import dataclasses
        w = dataclasses.replace(w, layers=min(args.layers, w.layers))
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
