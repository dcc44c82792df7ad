#!/usr/bin/env python3
"""Benchmark: attention calls/s of the write-time FP8 ring cache at 757 queries
over a 5,788-slot ring (48 heads x 128), and ms per 240-call chunk, on GB300.

One step = one four-frame chunk of the production model shape: for each of the
4 denoising passes and 60 layers, write the chunk's 757 new tokens into the
layer's ring (RoPE + per-head E4M3 quantisation) and run the attention call of
the 757 queries over all 5,788 slots; then one position reset (delta rotation of
every stored key in all 60 layers) that moves the window back by one chunk, so
positions stay in [0, 5788).  That is every step of the path once per step.
The rings (4.3 GB) and the 240 distinct (K, V, Q) inputs of a chunk (6.7 GB)
are far larger than L2, so no L2 flush is needed between steps.  Each timed
step's 481 launches are captured into a CUDA graph (the calls launch kernels
only) while the GPU runs the previous step, and the graph is launched once.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --sustained 3600    # per-head std U[0.5, 4], restart every 300 chunks: mean / p99 ms per chunk
  python bench.py --stress 100        # 60 full rings, 100 deltas ~ U_int[-200000, 0], each + write + attend
  python bench.py --copy-window       # the copy-based window (shift every chunk) against the ring
  python bench.py --profile attention|write|rotate   # small fixed cases for ncu captures

Under torchrun (N > 1) every rank runs its own session on its own GPU (the
method is batch-1 per session; replicas, weak scaling) and rank 0 prints the
aggregate.  --impl reference times the fp64 oracle on the host cores instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L, H, D, C, N_NEW, PREFILL, PASSES = 60, 48, 128, 5788, 757, 5031, 4
CALLS_PER_CHUNK = L * PASSES
METRIC = "attention calls/s at 757q×5788-slot FP8 ring cache; ms per 240-call chunk"
ATTN_FLOP = 4.0 * N_NEW * C * D * H                      # 107.68 GFLOP per call (algorithmic)
WRITE_BYTES = N_NEW * H * D * (2 + 2) + N_NEW * H * D * 2  # bf16 K,V read + E4M3 K,V codes written
ROTATE_BYTES = 2.0 * L * H * C * D                        # K codes read + written, all layers
READTIME_EXTRA_BYTES = C * H * D * (2 + 2) + C * H * D * 2  # bf16 store read + FP8 ring written
BF16_WRITE_BYTES = N_NEW * H * D * (2 + 2) * 2             # bf16 K,V read + bf16 K,V written
BF16_ROTATE_BYTES = 2.0 * L * H * C * D * 2                # bf16 K read + written, all layers

# dram bytes per launch measured by ncu, valid only for the kernel source they
# were taken on
TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one attn_kernel launch at
    # the production call, valid while rc_attention.cu has this hash
    "attention": {"bytes": 87.18e6,
                  "src_sha256": "969f5fc9f6f27c22cc9e62250c525567ba42c19f63cb6de9e4160a53f3fb1657"},
}


def src_sha(name: str) -> str:
    path = os.path.join(ROOT, "fp8_ring_kv_cache_gb300", "csrc", name)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return json.load(open(path)), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.sink = None

    def start(self):
        import tempfile
        # samples go to a file, not a pipe: a long run would fill a pipe and stall the sampler
        self.sink = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=self.sink, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.sink.seek(0)
        out = self.sink.read()
        self.sink.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- ranks

def max_over_ranks(values: list[float], device, world: int) -> list[float]:
    """Element-wise maximum of per-rank timings (every rank gets the result)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor(values, device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world: int, steps: int, elapsed_ms: float) -> float:
    """Calls per second of the whole job: every rank runs `steps` chunks of
    CALLS_PER_CHUNK calls on its own GPU; the job takes the slowest rank's time."""
    return world * CALLS_PER_CHUNK * steps / (elapsed_ms / 1e3)


def capture_graph(fn, side):
    """The launches of fn() captured into a CUDA graph on stream `side` (not
    launched).  The library's host-side bookkeeping (slots, write groups) runs
    as in a direct call, so the graph holds exactly the kernels a direct call
    would launch, with the same arguments; it is launched once, in order."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        g.capture_begin(capture_error_mode="thread_local")
        try:
            fn()
        finally:
            g.capture_end()
    return g


def graphed_ms(fn, n: int, stream, ahead: bool = False) -> float:
    """Device time of n calls of fn, each captured into its own CUDA graph and
    launched once on `stream`: the host captures call i + 1 while the GPU runs
    call i, and the first graph is captured before the clock starts (ahead:
    all n are captured first, for calls whose host side is slower than their
    kernels).  Events on `stream` bracket the n launches."""
    import torch

    side = torch.cuda.Stream()
    todo = [capture_graph(fn, side) for _ in range(n if ahead else 1)]
    done = []
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(n):
        g = todo[i] if ahead else (todo[0] if i == 0 else capture_graph(fn, side))
        with torch.cuda.stream(stream):
            g.replay()
        done.append(g)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


# ---------------------------------------------------------------- our arm

def run_ours(args, rank: int, world: int, local_rank: int) -> dict | None:
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc
    import synth_inputs as si

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    seed = 21 + 1000 * rank
    cache = rc.RingKVCache(L, H, D, C, max_write=C)
    mult = si.outlier_mask(H, D, seed)
    # the 240 distinct inputs of a chunk, resident in HBM before timing
    K = torch.empty(PASSES, L, N_NEW, H, D, dtype=torch.bfloat16, device=dev)
    V = torch.empty_like(K)
    Q = torch.empty_like(K)
    for pas in range(PASSES):
        for layer in range(L):
            k, v, q = si.chunk_tensors(seed, 0, pas, layer, dev, mult=mult)
            K[pas, layer], V[pas, layer], Q[pas, layer] = k, v, q
    out = torch.empty(N_NEW, H, D, dtype=torch.float32, device=dev)
    kp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, 7), dev, mult)
    vp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, 8), dev, mult)
    for layer in range(L):
        cache.write(layer, kp, vp, np.arange(0, PREFILL))
    chunk_pos = np.arange(PREFILL, PREFILL + N_NEW)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def chunk(rec=None):
        for pas in range(PASSES):
            for layer in range(L):
                if rec is not None:
                    i = rec["i"]
                    rec["w"][i][0].record(stream)
                cache.write(layer, K[pas, layer], V[pas, layer], chunk_pos)
                if rec is not None:
                    rec["w"][i][1].record(stream)
                    rec["a"][i][0].record(stream)
                cache.attend(layer, Q[pas, layer], out)
                if rec is not None:
                    rec["a"][i][1].record(stream)
                    rec["i"] = i + 1

    def step(rec=None):
        chunk(rec)
        if rec is not None:
            j = rec["j"]
            rec["r"][j][0].record(stream)
        cache.delta_rotate(-N_NEW)          # the window restarts: oldest stored position -> 0
        if rec is not None:
            rec["r"][j][1].record(stream)
            rec["j"] = j + 1

    for _ in range(args.warmup):
        step()
    graphed_ms(step, 1, stream)  # the capture path warmed up too
    cache.sync()

    # ---- timed region: K steps, each a CUDA graph launched once
    launches0 = cache.launch_count
    clocks = ClockSampler(local_rank)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    elapsed_ms = graphed_ms(step, args.steps, stream)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    cache.sync()
    launches = cache.launch_count - launches0

    # ---- per-kernel times.  Attention and write: the chunk's 240 calls of one
    # kind captured into a graph and launched back to back, events around the
    # graphs (an event inside a graph, or around a direct call, widens every
    # span it brackets); K graphs each, all captured before the clock starts
    # (the host side of 240 writes takes longer than their kernels).  Also an event pair around every call
    # in K more steps launched directly (the rotation's time comes from there).
    def calls(kind):
        def run():
            for pas in range(PASSES):
                for layer in range(L):
                    if kind == "attend":
                        cache.attend(layer, Q[pas, layer], out)
                    else:
                        cache.write(layer, K[pas, layer], V[pas, layer], chunk_pos)
        return run

    per_call = 1e3 / (args.steps * CALLS_PER_CHUNK)
    att_us = graphed_ms(calls("attend"), args.steps, stream, ahead=True) * per_call
    w_us = graphed_ms(calls("write"), args.steps, stream, ahead=True) * per_call
    nw = args.steps * CALLS_PER_CHUNK
    rec = {"w": [(ev(), ev()) for _ in range(nw)], "a": [(ev(), ev()) for _ in range(nw)],
           "r": [(ev(), ev()) for _ in range(args.steps)], "i": 0, "j": 0}
    torch.cuda.synchronize()
    for _ in range(args.steps):
        step(rec)
    torch.cuda.synchronize()
    cache.sync()
    w_times = [a.elapsed_time(b) * 1e3 for a, b in rec["w"]]
    a_times = [a.elapsed_time(b) * 1e3 for a, b in rec["a"]]
    r_times = [a.elapsed_time(b) * 1e3 for a, b in rec["r"]]

    # ---- chunk without a reset (ms per 240-call chunk), same inputs, graphs as above
    chunk_ms = graphed_ms(chunk, args.steps, stream) / args.steps
    cache.sync()
    del cache

    # ---- read-time ablation: same chunk, whole-cache RoPE + quantisation per call
    ab = run_ablation(args, dev, K, V, Q, kp, vp)

    # ---- the same step on a bf16 ring (the FP8-versus-bf16 cache comparison)
    peaks, peak_src = load_peaks()
    bf = run_bf16_cache(args, dev, K, V, Q, kp, vp, peaks["bf16_tflops"])

    # ---- the write fused into the K/V projection (next-3)
    fused = run_fused(args, dev, 2.0 * peaks["bf16_tflops"])

    # ---- end to end through the C ABI with host buffers
    e2e = run_e2e(args, dev, K, V, Q, kp, vp)

    # ---- max over ranks
    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e["elapsed_ms"]], dev, world)
    if rank != 0:
        return None

    # fp8 dense = 2x bf16 dense (nominal ratio).  The attention kernel is timed
    # per launch (microseconds, full SM clock), so the burst rate applies; the
    # fraction against the sustained (power-capped) rate is reported beside it.
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    fp8_peak_sustained = 2.0 * peaks["bf16_tflops_sustained"]
    hbm = peaks["hbm_gbs"]
    ms_step = elapsed_ms / args.steps
    value = job_throughput(world, args.steps, elapsed_ms)
    achieved_tflops = ATTN_FLOP / (att_us * 1e-6) / 1e12
    r_us = statistics.mean(r_times)
    tr = TRAFFIC["attention"]
    traffic = tr["bytes"] if tr["bytes"] is not None and tr["src_sha256"] == src_sha("rc_attention.cu") else None
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "calls/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic",
        "config": {
            "workload": "chunk of 240 calls: 4 passes x 60 layers x (write 757 new tokens + attention of "
                        "757 queries over 5,788 FP8 slots), 48 heads x 128, then one 60-layer delta rotation",
            "layers": L, "heads": H, "head_dim": D, "slots": C, "new_tokens": N_NEW, "prefill": PREFILL,
            "calls_per_step": CALLS_PER_CHUNK, "outliers": "1% of (head, channel) pairs x20 on K and V",
            "l2": "no flush: 4.3 GB of rings and 6.7 GB of chunk inputs per step exceed the 129 MB L2",
            "parallelism": f"replicas x{world} (one session per GPU)",
            "launch": "each step captured into a CUDA graph (the host captures step k + 1 while the GPU runs "
                      "step k) and launched once",
            "kernel_times": "attention and write: mean over the chunk's 240 calls of one kind launched back to "
                            "back in a graph, events around the graph; rotation: events around the call in "
                            "steps launched directly",
        },
        "ms_per_chunk": round(chunk_ms, 4),
        "roofline": {
            "bound": "tensor", "kernel": "attention (rc_attend)",
            "achieved": round(achieved_tflops, 2), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
            "frac": round(achieved_tflops / fp8_peak, 4), "traffic": traffic,
            "peak_source": f"{peak_src}: 2 x bf16_tflops, the burst rate (fp8/bf16 nominal ratio 2)",
            "frac_of_sustained_peak": round(achieved_tflops / fp8_peak_sustained, 4),
            "per_launch_us": round(att_us, 3), "flop_per_launch": ATTN_FLOP,
        },
        "kernels": {
            "write": {"us": round(w_us, 3), "bytes": WRITE_BYTES,
                      "gbs": round(WRITE_BYTES / (w_us * 1e-6) / 1e9, 1),
                      "frac_hbm": round(WRITE_BYTES / (w_us * 1e-6) / 1e9 / hbm, 4),
                      "us_event_span_direct": round(statistics.mean(w_times), 3)},
            "delta_rotate": {"us": round(r_us, 3), "bytes": ROTATE_BYTES,
                             "gbs": round(ROTATE_BYTES / (r_us * 1e-6) / 1e9, 1),
                             "frac_hbm": round(ROTATE_BYTES / (r_us * 1e-6) / 1e9 / hbm, 4)},
            "attention": {"us": round(att_us, 3), "tflops": round(achieved_tflops, 1),
                          "frac_fp8": round(achieved_tflops / fp8_peak, 4),
                          "frac_fp8_sustained": round(achieved_tflops / fp8_peak_sustained, 4),
                          "us_event_span_direct": round(statistics.mean(a_times), 3)},
            "readtime_ablation": ab,
            "fused_write": fused,
            "bf16_cache": dict(bf, fp8_ms_per_step=round(ms_step, 4),
                               fp8_saves_ms_per_step=round(bf["ms_per_step"] - ms_step, 4),
                               peak_source=f"{peak_src}: bf16_tflops, the burst rate"),
            "hbm_peak_gbs": hbm, "peak_source": peak_src,
        },
        "e2e": {"value": round(job_throughput(world, args.steps, e2e_ms), 2), "unit": "calls/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_ms / args.steps, 3)},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(calls=args.cpu_calls)
    return res


def run_sustained(args) -> dict:
    """Sustained workload: `--sustained N` chunks of 240 calls at the production
    shape with a per-head standard deviation drawn once per (layer, head) from
    U[0.5, 4] for Q, K and V alike (the 240 distinct inputs of a chunk are
    generated once and reused).  Each chunk writes 757 new positions (4 passes
    rewrite them) and the window restarts every 300 chunks: one delta rotation
    of every layer by -(oldest stored position).  Each chunk is captured into a
    CUDA graph while the GPU runs the previous one and launched once; per-chunk
    times come from events around the launches on the launching stream; the
    steady state leaves out the first three chunks (the ring fills during the
    first)."""
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc
    import synth_inputs as si

    dev = torch.device("cuda", 0)
    seed = 41
    std = si.head_std(L, H, seed)
    cache = rc.RingKVCache(L, H, D, C, max_write=C)
    K = torch.empty(PASSES, L, N_NEW, H, D, dtype=torch.bfloat16, device=dev)
    V = torch.empty_like(K)
    Q = torch.empty_like(K)
    for pas in range(PASSES):
        for layer in range(L):
            k, v, q = si.chunk_tensors(seed, 0, pas, layer, dev, std=std[layer])
            K[pas, layer], V[pas, layer], Q[pas, layer] = k, v, q
    out = torch.empty(N_NEW, H, D, dtype=torch.float32, device=dev)
    for layer in range(L):
        sl = std[layer].view(H, 1)
        kp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, layer, 7), dev, sl)
        vp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, layer, 8), dev, sl)
        cache.write(layer, kp, vp, np.arange(0, PREFILL))
    stream = torch.cuda.current_stream()
    newest = PREFILL - 1
    nch, every = args.sustained, 300
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nch)]
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nch // every)]
    torch.cuda.synchronize()
    clocks = ClockSampler(0, period_ms=500)
    clocks.start()
    launches0 = cache.launch_count
    side = torch.cuda.Stream()

    def chunk(pos):
        for pas in range(PASSES):
            for layer in range(L):
                cache.write(layer, K[pas, layer], V[pas, layer], pos)
                cache.attend(layer, Q[pas, layer], out)

    # the host's calls keep the device's order: chunk c's graph is launched
    # (and the reset after it made) before chunk c + 1 is captured
    t0 = time.perf_counter()
    g = capture_graph(lambda: chunk(np.arange(newest + 1, newest + 1 + N_NEW)), side)
    recent = []
    for c in range(nch):
        ev[c][0].record(stream)
        g.replay()
        ev[c][1].record(stream)
        recent = (recent + [g])[-4:]     # a graph freed in flight is released when it completes
        newest += N_NEW
        if (c + 1) % every == 0:
            oldest = newest - C + 1          # the ring is full after the first chunk
            r = rev[(c + 1) // every - 1]
            r[0].record(stream)
            cache.delta_rotate(-oldest)
            r[1].record(stream)
            newest -= oldest
        if c + 1 < nch:
            g = capture_graph(lambda: chunk(np.arange(newest + 1, newest + 1 + N_NEW)), side)
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - t0
    clk = clocks.stop()
    cache.sync()
    launches = cache.launch_count - launches0
    ms = sorted(a.elapsed_time(b) for a, b in ev[3:])
    resets = [a.elapsed_time(b) for a, b in rev]
    mean = statistics.mean(ms)
    return {
        "mode": "sustained",
        "metric": "ms per 240-call chunk, steady state (mean, p50, p99, max)",
        "chunks": nch, "steady_chunks": len(ms),
        "ms_per_chunk_mean": round(mean, 4),
        "ms_per_chunk_p50": round(ms[len(ms) // 2], 4),
        "ms_per_chunk_p99": round(ms[min(len(ms) - 1, int(0.99 * len(ms)))], 4),
        "ms_per_chunk_max": round(ms[-1], 4),
        "calls_per_s": round(CALLS_PER_CHUNK / mean * 1e3, 2),
        "resets": len(resets), "ms_per_reset_mean": round(statistics.mean(resets), 4) if resets else None,
        "wall_s": round(wall_s, 2), "gpu_launches": int(launches),
        "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": "sustained chunks: 4 passes x 60 layers x (write 757 new tokens + attention of 757 "
                               "queries over 5,788 FP8 slots), 48 heads x 128, per-head std U[0.5, 4] for Q, K, V; "
                               "window restart (delta = -oldest position) every 300 chunks",
                   "layers": L, "heads": H, "head_dim": D, "slots": C, "new_tokens": N_NEW, "prefill": PREFILL},
        "clocks": clk,
    }


def run_stress(args) -> dict:
    """Reset stress at 60 layers: every ring full at positions up to 200,000, then
    `--stress N` steps of (delta rotation of all layers by a delta drawn from
    U_int[-200000, 0], then write 757 tokens at the next positions and attend,
    in every layer).  Events time the rotation and the 60 write + attend pairs
    of each step separately."""
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc
    import synth_inputs as si

    dev = torch.device("cuda", 0)
    seed = 31
    cache = rc.RingKVCache(L, H, D, C, max_write=C)
    top = 200_000
    k0 = si.normal_bf16(C, H, D, si.subseed(seed, 1), dev)
    v0 = si.normal_bf16(C, H, D, si.subseed(seed, 2), dev)
    for layer in range(L):
        cache.write(layer, k0, v0, np.arange(top - C + 1, top + 1))
    K = torch.empty(L, N_NEW, H, D, dtype=torch.bfloat16, device=dev)
    V = torch.empty_like(K)
    Q = torch.empty_like(K)
    for layer in range(L):
        K[layer] = si.normal_bf16(N_NEW, H, D, si.subseed(seed, 10, layer, 1), dev)
        V[layer] = si.normal_bf16(N_NEW, H, D, si.subseed(seed, 10, layer, 2), dev)
        Q[layer] = si.normal_bf16(N_NEW, H, D, si.subseed(seed, 10, layer, 3), dev)
    out = torch.empty(N_NEW, H, D, dtype=torch.float32, device=dev)
    deltas = si.stress_deltas(seed, args.stress)
    stream = torch.cuda.current_stream()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))  # noqa: E731
    rot, calls = [mk() for _ in deltas], [mk() for _ in deltas]
    nxt = top + 1
    torch.cuda.synchronize()
    clocks = ClockSampler(0, period_ms=200)
    clocks.start()
    for i, d in enumerate(deltas):
        rot[i][0].record(stream)
        cache.delta_rotate(d)
        rot[i][1].record(stream)
        nxt += d
        pos = np.arange(nxt, nxt + N_NEW)
        nxt += N_NEW
        calls[i][0].record(stream)
        for layer in range(L):
            cache.write(layer, K[layer], V[layer], pos)
            cache.attend(layer, Q[layer], out)
        calls[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    cache.sync()
    r = [a.elapsed_time(b) for a, b in rot]
    c = [a.elapsed_time(b) for a, b in calls]
    return {
        "mode": "stress",
        "metric": "ms per delta rotation of 60 layers and per 60 (write + attend) calls after it",
        "steps": len(deltas), "delta_range": [min(deltas), max(deltas)],
        "ms_per_rotation_mean": round(statistics.mean(r), 4), "ms_per_rotation_max": round(max(r), 4),
        "rotation_gbs": round(ROTATE_BYTES / (statistics.mean(r) * 1e-3) / 1e9, 1),
        "ms_per_60_calls_mean": round(statistics.mean(c), 4), "ms_per_60_calls_max": round(max(c), 4),
        "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": "reset stress: full 5,788-slot rings at positions up to 200,000 in 60 layers, "
                               "then delta ~ U_int[-200000, 0] + write 757 + attend in every layer, per step",
                   "layers": L, "heads": H, "head_dim": D, "slots": C, "new_tokens": N_NEW},
        "clocks": clk,
    }


def run_copy_window(args) -> dict:
    """The copy-based window against the ring on the chunk workload.  A step is
    the chunk (240 calls) and the 60-layer delta rotation that restarts the
    window, as in the default bench; the copy-based cache also moves every
    stored token 757 slots down in every layer before the chunk
    (rc_cache_window_shift), as a cache that concatenates must.  Same inputs,
    one cache at a time; per-part times from events on the launching stream."""
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc
    import synth_inputs as si

    dev = torch.device("cuda", 0)
    seed = 21
    mult = si.outlier_mask(H, D, seed)
    K = torch.empty(PASSES, L, N_NEW, H, D, dtype=torch.bfloat16, device=dev)
    V = torch.empty_like(K)
    Q = torch.empty_like(K)
    for pas in range(PASSES):
        for layer in range(L):
            k, v, q = si.chunk_tensors(seed, 0, pas, layer, dev, mult=mult)
            K[pas, layer], V[pas, layer], Q[pas, layer] = k, v, q
    out = torch.empty(N_NEW, H, D, dtype=torch.float32, device=dev)
    kp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, 7), dev, mult)
    vp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, 8), dev, mult)
    chunk_pos = np.arange(PREFILL, PREFILL + N_NEW)
    stream = torch.cuda.current_stream()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))  # noqa: E731
    res = {}
    for variant in ("ring", "copy"):
        cache = rc.RingKVCache(L, H, D, C, max_write=C, copy_window=(variant == "copy"))
        for layer in range(L):
            cache.write(layer, kp, vp, np.arange(0, PREFILL))

        def step(ev=None):
            if ev is not None:
                ev[0][0].record(stream)
            if variant == "copy":
                cache.window_shift(N_NEW)
            if ev is not None:
                ev[0][1].record(stream)
                ev[1][0].record(stream)
            for pas in range(PASSES):
                for layer in range(L):
                    cache.write(layer, K[pas, layer], V[pas, layer], chunk_pos)
                    cache.attend(layer, Q[pas, layer], out)
            if ev is not None:
                ev[1][1].record(stream)
                ev[2][0].record(stream)
            cache.delta_rotate(-N_NEW)
            if ev is not None:
                ev[2][1].record(stream)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        evs = [[mk(), mk(), mk()] for _ in range(args.steps)]
        t0, t1 = mk()
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize()
        cache.sync()
        part = lambda j: statistics.mean(e[j][0].elapsed_time(e[j][1]) for e in evs)  # noqa: E731
        res[variant] = {"ms_per_step": round(t0.elapsed_time(t1) / args.steps, 4),
                        "ms_shift": round(part(0), 4), "ms_chunk": round(part(1), 4),
                        "ms_delta": round(part(2), 4)}
        cache.close()
        del cache
    shift_bytes = 2.0 * 2 * L * H * C * D + 2.0 * 2 * L * H * C * 4   # codes and scales, read + written
    ms = res["copy"]["ms_shift"]
    return {
        "mode": "copy_window",
        "metric": "ms per step (chunk + window restart), ring vs copy-based window",
        "steps": args.steps, "warmup": args.warmup,
        "ring": res["ring"], "copy": res["copy"],
        "copy_extra_ms_per_step": round(res["copy"]["ms_per_step"] - res["ring"]["ms_per_step"], 4),
        "shift_gbs": round(shift_bytes / (ms * 1e-3) / 1e9, 1) if ms > 0 else None,
        "shift_bytes": shift_bytes,
        "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": "chunk of 240 calls (4 passes x 60 layers x (write 757 + attention of 757 queries "
                               "over 5,788 FP8 slots), 48 heads x 128) + 60-layer delta rotation; the copy-based "
                               "cache also shifts every layer's slots by 757 before each chunk",
                   "layers": L, "heads": H, "head_dim": D, "slots": C, "new_tokens": N_NEW, "prefill": PREFILL},
    }


def run_ablation(args, dev, K, V, Q, kp, vp) -> dict:
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc

    cache = rc.RingKVCache(L, H, D, C, max_write=C, readtime_ablation=True)
    for layer in range(L):
        cache.write(layer, kp, vp, np.arange(0, PREFILL))
    out = torch.empty(N_NEW, H, D, dtype=torch.float32, device=dev)
    pos = np.arange(PREFILL, PREFILL + N_NEW)
    stream = torch.cuda.current_stream()

    def chunk(readtime: bool):
        for pas in range(PASSES):
            for layer in range(L):
                cache.write(layer, K[pas, layer], V[pas, layer], pos)
                if readtime:
                    cache.attend_readtime(layer, Q[pas, layer], out)
                else:
                    cache.attend(layer, Q[pas, layer], out)

    res = {}
    for mode in (False, True):
        chunk(mode)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(max(1, args.steps // 2)):
            chunk(mode)
        b.record(stream)
        torch.cuda.synchronize()
        res["readtime" if mode else "writetime"] = a.elapsed_time(b) / max(1, args.steps // 2)
    cache.sync()
    del cache
    extra_ms = res["readtime"] - res["writetime"]
    return {"ms_per_chunk_readtime": round(res["readtime"], 3),
            "ms_per_chunk_writetime_same_store": round(res["writetime"], 3),
            "saved_ms_per_chunk": round(extra_ms, 3),
            "extra_us_per_call": round(extra_ms * 1e3 / CALLS_PER_CHUNK, 3),
            "extra_bytes_per_call": READTIME_EXTRA_BYTES}


def run_bf16_cache(args, dev, K, V, Q, kp, vp, bf16_peak: float) -> dict:
    """The same step (chunk + 60-layer delta rotation) on a bf16 ring: the
    non-FP8 side of the FP8-versus-bf16 cache comparison.  Same inputs; steps
    timed as CUDA graphs like the FP8 step, per-kernel events from steps
    launched directly."""
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc

    cache = rc.RingKVCache(L, H, D, C, max_write=C, bf16_cache=True)
    for layer in range(L):
        cache.write(layer, kp, vp, np.arange(0, PREFILL))
    out = torch.empty(N_NEW, H, D, dtype=torch.float32, device=dev)
    pos = np.arange(PREFILL, PREFILL + N_NEW)
    stream = torch.cuda.current_stream()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))  # noqa: E731

    def step(rec=None):
        for pas in range(PASSES):
            for layer in range(L):
                if rec is not None:
                    w, a = mk(), mk()
                    rec["w"].append(w)
                    rec["a"].append(a)
                    w[0].record(stream)
                cache.write(layer, K[pas, layer], V[pas, layer], pos)
                if rec is not None:
                    w[1].record(stream)
                    a[0].record(stream)
                cache.attend(layer, Q[pas, layer], out)
                if rec is not None:
                    a[1].record(stream)
        if rec is not None:
            r = mk()
            rec["r"].append(r)
            r[0].record(stream)
        cache.delta_rotate(-N_NEW)
        if rec is not None:
            r[1].record(stream)

    for _ in range(args.warmup):
        step()
    graphed_ms(step, 1, stream)
    torch.cuda.synchronize()
    steps = max(1, args.steps // 2)
    step_ms = graphed_ms(step, steps, stream) / steps
    rec = {"w": [], "a": [], "r": []}
    for _ in range(steps):
        step(rec)
    torch.cuda.synchronize()
    cache.sync()
    cache.close()
    mean_us = lambda evs: statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3  # noqa: E731
    w_us, a_us, r_us = mean_us(rec["w"]), mean_us(rec["a"]), mean_us(rec["r"])
    tflops = ATTN_FLOP / (a_us * 1e-6) / 1e12
    return {"ms_per_step": round(step_ms, 4), "steps": steps,
            "write_us": round(w_us, 3), "write_gbs": round(BF16_WRITE_BYTES / (w_us * 1e-6) / 1e9, 1),
            "attention_us": round(a_us, 3), "attention_tflops": round(tflops, 1),
            "attention_frac_bf16": round(tflops / bf16_peak, 4),
            "delta_rotate_us": round(r_us, 3),
            "delta_rotate_gbs": round(BF16_ROTATE_BYTES / (r_us * 1e-6) / 1e9, 1),
            "ring_bytes": 2 * L * H * C * D * 2}


def run_fused(args, dev, fp8_peak: float) -> dict:
    """The write fused into the K/V projection (rc_cache_write_fused) at the
    production shape -- 757 tokens, 48 heads x 128, hidden 6,144, E4M3
    operands resident in HBM -- against what it replaces: the projection as a
    library FP8 GEMM to bf16 (cuBLASLt through torch._scaled_mm), then
    rc_cache_write.  Per-call times are CUDA events on the launching stream,
    averaged over calls that cycle over four layers."""
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc
    import synth_inputs as si

    n, hidden, F = N_NEW, si.PROD_HIDDEN, H * D
    x, xs, wk, wks, wv, wvs = si.proj_operands(23, n, hidden, F, dev)
    pos = np.arange(PREFILL, PREFILL + N_NEW)
    cache = rc.RingKVCache(4, H, D, C, max_write=C)
    stream = torch.cuda.current_stream()
    calls = max(8, 4 * args.steps)
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))  # noqa: E731

    def timed(fn):
        for i in range(4):
            fn(i)
        torch.cuda.synchronize()
        a, b = mk()
        a.record(stream)
        for i in range(calls):
            fn(i % 4)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / calls

    fused_us = timed(lambda l: cache.write_fused(l, x, xs, wk, wks, wv, wvs, pos))
    flop = 2.0 * n * 2 * F * hidden
    res = {"us": round(fused_us, 3), "tflops": round(flop / (fused_us * 1e-6) / 1e12, 1),
           "frac_fp8": round(flop / (fused_us * 1e-6) / 1e12 / fp8_peak, 4), "flop_per_call": flop,
           "shape": f"{n} tokens x hidden {hidden} -> K, V of {H} heads x {D}"}
    try:
        xf = x.view(torch.float8_e4m3fn)
        wkf, wvf = wk.view(torch.float8_e4m3fn), wv.view(torch.float8_e4m3fn)
        sx = torch.tensor(xs, device=dev)
        sk, sv = torch.tensor(wks, device=dev), torch.tensor(wvs, device=dev)

        def gemms():
            kb = torch._scaled_mm(xf, wkf.t(), scale_a=sx, scale_b=sk, out_dtype=torch.bfloat16)
            vb = torch._scaled_mm(xf, wvf.t(), scale_a=sx, scale_b=sv, out_dtype=torch.bfloat16)
            return kb.view(n, H, D), vb.view(n, H, D)

        gemm_us = timed(lambda l: gemms())
        kb, vb = gemms()
        write_us = timed(lambda l: cache.write(l, kb, vb, pos))
        both_us = timed(lambda l: cache.write(l, *gemms(), pos))
        res["unfused"] = {"gemm_us": round(gemm_us, 3), "write_us": round(write_us, 3), "us": round(both_us, 3),
                          "gemm": "torch._scaled_mm (cuBLASLt FP8 -> bf16), two GEMMs"}
        res["saves_us"] = round(both_us - fused_us, 3)
    except Exception as e:  # the library GEMM is context only
        res["unfused"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    cache.sync()
    cache.close()
    return res


def run_e2e(args, dev, K, V, Q, kp, vp) -> dict:
    """The same step as the device-timed one (a 240-call chunk, then the
    60-layer delta rotation that restarts the window) through the public API
    with pinned host inputs: every call copies its K, V, Q host->device and its
    output device->host, inside the timed region.  A call's K, V and Q sit
    next to each other in one pinned host buffer and go up in one copy (three
    separate copies took ~5 % longer a step); inputs go up on one copy stream,
    three calls ahead, and outputs come down on another (the two directions
    run at once), so the copies of neighbouring calls overlap the compute
    stream."""
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc

    cache = rc.RingKVCache(L, H, D, C, max_write=C)
    for layer in range(L):
        cache.write(layer, kp, vp, np.arange(0, PREFILL))
    nbuf, nb, ahead = 8, 6, 3
    E = N_NEW * H * D                     # elements of one [n][H][D] tensor
    host = []                             # per input set: K | V | Q, pinned
    for i in range(nbuf):
        hb = torch.empty(3 * E, dtype=torch.bfloat16).pin_memory()
        for j, t in enumerate((K, V, Q)):
            hb[j * E:(j + 1) * E].copy_(t[0, i].reshape(-1).cpu())
        host.append(hb)
    hout = [torch.empty(N_NEW, H, D, dtype=torch.float32).pin_memory() for _ in range(nb)]
    dkvq = [torch.empty(3 * E, dtype=torch.bfloat16, device=dev) for _ in range(nb)]
    dout = [torch.empty(N_NEW, H, D, dtype=torch.float32, device=dev) for _ in range(nb)]
    comp = torch.cuda.current_stream()
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    pos = np.arange(PREFILL, PREFILL + N_NEW)
    in_ready = [torch.cuda.Event() for _ in range(nb)]
    consumed = [torch.cuda.Event() for _ in range(nb)]
    out_ready = [torch.cuda.Event() for _ in range(nb)]
    drained = [torch.cuda.Event() for _ in range(nb)]
    for e in consumed + drained:
        e.record(comp)
    calls = [(pas, layer) for pas in range(PASSES) for layer in range(L)]

    def upload(i):
        b = i % nb
        with torch.cuda.stream(up):
            up.wait_event(consumed[b])
            dkvq[b].copy_(host[i % nbuf], non_blocking=True)
            in_ready[b].record(up)

    def chunk():
        for i in range(min(ahead, len(calls))):
            upload(i)
        for i, (pas, layer) in enumerate(calls):
            b = i % nb
            if i + ahead < len(calls):
                upload(i + ahead)          # later calls' inputs go up during this call
            comp.wait_event(in_ready[b])
            comp.wait_event(drained[b])
            kvq = dkvq[b]
            cache.write(layer, kvq[:E].view(N_NEW, H, D), kvq[E:2 * E].view(N_NEW, H, D), pos)
            cache.attend(layer, kvq[2 * E:].view(N_NEW, H, D), dout[b])
            consumed[b].record(comp)
            out_ready[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(out_ready[b])
                hout[b].copy_(dout[b], non_blocking=True)
                drained[b].record(down)
        cache.delta_rotate(-N_NEW)          # the window restarts, as in the device-timed step

    for _ in range(args.warmup):
        chunk()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        chunk()
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3
    cache.sync()
    del cache
    per_call_in = 3 * N_NEW * H * D * 2
    per_call_out = N_NEW * H * D * 4
    return {"elapsed_ms": ms, "h2d": CALLS_PER_CHUNK * per_call_in, "d2h": CALLS_PER_CHUNK * per_call_out}


# ---------------------------------------------------------------- the oracle

def cpu_calls(calls: int, seed: int = 11) -> tuple[float, int, str]:
    """Time the fp64 oracle on full production calls (prefill untimed; each call =
    write 757 + attention of 757 queries over 5,788 slots, all 48 heads)."""
    import numpy as np

    import oracle
    import synth_inputs as si

    oracle.build()
    t = si.production_tensors(seed, "cpu")
    oc = oracle.OracleCache(1, H, D, C)
    oc.write(0, t["k_prefill"], t["v_prefill"], np.arange(0, PREFILL))
    times = []
    for i in range(calls):
        t0 = time.perf_counter()
        oc.write(0, t["k_new"], t["v_new"], np.arange(PREFILL, C))
        oc.attend(0, t["q"])
        times.append(time.perf_counter() - t0)
    cores = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    sample = (f"{calls} full production calls (write 757 tokens + attention 757 x 5,788, 48 heads x 128) "
              "after an untimed 5,031-token prefill")
    return statistics.mean(times), cores, sample


def cpu_baseline(calls: int) -> dict:
    t, cores, sample = cpu_calls(calls)
    return {"value": round(1.0 / t, 5), "unit": "calls/s", "cores": cores, "kind": "oracle", "sample": sample,
            "s_per_call": round(t, 3)}


def run_reference(args, rank: int, world: int) -> dict | None:
    if rank != 0:
        return None
    steps, warmup = args.steps, args.warmup
    t_w, cores, sample = cpu_calls(max(1, warmup))
    t, cores, sample = cpu_calls(steps)
    value = 1.0 / t
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 5), "unit": "calls/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(t * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "one production call per step: write 757 new tokens + attention of 757 queries "
                               "over 5,788 slots, 48 heads x 128 (the fp64 oracle on the host cores)",
                   "heads": H, "head_dim": D, "slots": C, "new_tokens": N_NEW, "prefill": PREFILL},
        "cpu_baseline": {"value": round(value, 5), "unit": "calls/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "calls/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile_case(kind: str) -> None:
    """Small fixed cases for ncu captures (a few hundred MB on the device).

    attention : 2 layers of the production ring (48 x 128, 5,788 slots full);
                3 attention calls alternate between the layers.
    write     : 3 writes of 757 tokens into 3 layers.
    rotate    : 2 delta rotations of 4 full layers.
    attention_bf16 : the attention case on a bf16 ring.
    fused     : 3 fused projection writes (757 tokens, hidden 6,144) into 2 layers.
    """
    import numpy as np
    import torch

    import fp8_ring_kv_cache_gb300 as rc
    import synth_inputs as si

    if kind == "fused":
        x, xs, wk, wks, wv, wvs = si.proj_operands(23, N_NEW, si.PROD_HIDDEN, H * D, "cuda")
        cache = rc.RingKVCache(2, H, D, C, max_write=C)
        for i in range(3):
            cache.write_fused(i % 2, x, xs, wk, wks, wv, wvs, np.arange(PREFILL, C))
        cache.sync()
        print(f"profile case {kind} done, {cache.launch_count} launches")
        return
    bf16 = kind == "attention_bf16"
    kind = "attention" if bf16 else kind
    nl = {"attention": 2, "write": 3, "rotate": 4}[kind]
    cache = rc.RingKVCache(nl, H, D, C, max_write=C, bf16_cache=bf16)
    mult = si.outlier_mask(H, D, 11)
    kp = si.normal_bf16(PREFILL, H, D, 1, "cuda", mult)
    vp = si.normal_bf16(PREFILL, H, D, 2, "cuda", mult)
    kn = si.normal_bf16(N_NEW, H, D, 3, "cuda", mult)
    vn = si.normal_bf16(N_NEW, H, D, 4, "cuda", mult)
    q = si.normal_bf16(N_NEW, H, D, 5, "cuda")
    out = torch.empty(N_NEW, H, D, dtype=torch.float32, device="cuda")
    for layer in range(nl):
        cache.write(layer, kp, vp, np.arange(0, PREFILL))
        cache.write(layer, kn, vn, np.arange(PREFILL, C))
    cache.sync()
    if kind == "attention":
        for i in range(3):
            cache.attend(i % nl, q, out)
    elif kind == "write":
        for layer in range(nl):
            cache.write(layer, kn, vn, np.arange(PREFILL, C))
    else:
        for _ in range(2):
            cache.delta_rotate(-N_NEW)
    cache.sync()
    print(f"profile case {kind} done, {cache.launch_count} launches")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", choices=["attention", "write", "rotate", "attention_bf16", "fused"], default=None,
                    help="run a small fixed case for an ncu capture and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-calls", type=int, default=3, help="oracle calls timed for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustained", type=int, default=0, metavar="CHUNKS",
                    help="run the sustained workload for CHUNKS chunks (e.g. 3600) and exit")
    ap.add_argument("--stress", type=int, default=0, metavar="STEPS",
                    help="run the reset stress at 60 layers for STEPS steps (e.g. 100) and exit")
    ap.add_argument("--copy-window", action="store_true",
                    help="time the copy-based window against the ring on the chunk workload and exit")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args.profile)
        return
    if args.sustained:
        print(json.dumps(run_sustained(args)), flush=True)
        return
    if args.stress:
        print(json.dumps(run_stress(args)), flush=True)
        return
    if args.copy_window:
        print(json.dumps(run_copy_window(args)), flush=True)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        res = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
