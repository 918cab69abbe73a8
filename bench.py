#!/usr/bin/env python
"""Throughput of one Kimi-K2 MLA layer on GB300 through libmla's C ABI.

Default workload: decode, B=1, a cache built by causal prefill of 1000 tokens, one new token at
position 1000 attending to all 1001 positions.  A step is one whole decode call (projections,
norms, RoPE, cache append, absorbed split-KV attention, o_proj), captured once into a CUDA graph
and replayed.  Inputs are resident in HBM; L2 is flushed (a 256 MiB write) and the device
lengths restored between timed steps, outside the step's events.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s & cache HBM GB/s per layer; prefill TFLOP/s vs roofline"
L2_FLUSH_BYTES = 256 << 20
LAT_BYTES = 576 * 2            # one latent cache row (bf16)
WEIGHT_SHAPES = {"q_a": (1536, 7168), "q_b": (12288, 1536), "kv_a": (576, 7168),
                 "kv_b": (16384, 512), "o": (7168, 8192)}


def wbytes(name):
    r, c = WEIGHT_SHAPES[name]
    return r * c + (-(-r // 128)) * (-(-c // 128)) * 4


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (100 ms) of SM clock and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        return self

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.stop()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.proc = None

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------- GPU arm
def setup_decode(torch, mla, synth, layer, seed, lengths, build, device):
    """Caches of the given lengths (built by prefill or cache append) + the new tokens."""
    B = len(lengths)
    cap = max(lengths) + 1
    cache = torch.zeros(B, cap, 576, dtype=torch.bfloat16, device=device)
    lens = torch.zeros(B, dtype=torch.int32, device=device)
    to_dev = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).to(device)
    for b in range(B):
        done = 0
        while done < lengths[b]:
            n = min(16384, lengths[b] - done)
            x = to_dev(synth.hidden_states(seed, b, done, n))[None]
            if build == "prefill" and done == 0 and n == lengths[b]:
                layer.prefill(x, cache[b:b + 1], lens[b:b + 1], [0])
            else:
                layer.cache_append(x, cache[b:b + 1], lens[b:b + 1], [done])
            done += n
    xb = np.stack([synth.hidden_states(seed, b, lengths[b], 1)[0] for b in range(B)])
    torch.cuda.synchronize()
    return cache, lens, xb, to_dev(xb)


def algorithmic_bytes(kernel, B, lengths):
    """Bytes the method must move for one launch of `kernel` in a decode step."""
    S = sum(n + 1 for n in lengths)
    return {
        "gemm_q_a_kv_a": wbytes("q_a") + wbytes("kv_a") + B * 7168 * 2 + B * 2112 * 4,
        "norm_rope_cache": B * (2112 * 4 + 1536 * 2 + LAT_BYTES),
        "gemm_q_b": wbytes("q_b") + B * 1536 * 2 + B * 12288 * 2,
        "absorb_q": 64 * 128 * 512 + 64 * 4 * 4 + B * 12288 * 2 + B * 64 * 576 * 2,
        "decode_attention": S * LAT_BYTES + B * 64 * 576 * 2,
        "decode_combine": B * 64 * 512 * 2,
        "absorb_out": 64 * 128 * 512 + 64 * 4 * 4 + B * 64 * 512 * 2 + B * 8192 * 2,
        "gemm_o": wbytes("o") + B * 8192 * 2 + B * 7168 * 2,
        # few sequences: q_b_proj with the q-latent norm and the cache-row append fused in
        "gemm_q_b_norm": wbytes("q_b") + B * 2112 * 4 + B * 12288 * 2 + B * LAT_BYTES,
        # few sequences: the split combine fused with the W_UV absorption
        "combine_absorb_out": 64 * 128 * 512 + 64 * 4 * 4 + B * 64 * 512 * 2 + B * 8192 * 2,
        "advance_lens": B * 8,
    }.get(kernel, 0)


def traffic_record(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(f"{kernel}@{workload}")
    if not rec:
        return None
    src = os.path.join(ROOT, "head_latent_attention_mla_gb300", "csrc", rec["source"])
    if not os.path.exists(src):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != rec["sha256_16"]:
        return None
    return rec["dram_bytes_per_launch"]


def time_graph(torch, g, stream, lens, lens0, flush, steps):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(stream):
        for k in range(steps):
            lens.copy_(lens0)
            flush.zero_()
            ev[k][0].record(stream)
            g.replay()
            ev[k][1].record(stream)
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def steps_for(torch, g, stream, lens, lens0, flush, steps, min_ms):
    """At least `steps` steps, and enough for `min_ms` of timed device work (estimated from a
    short trial), so that short workloads are timed over many steps."""
    trial = time_graph(torch, g, stream, lens, lens0, flush, 5)
    per = max(1e-3, sum(trial) / len(trial))
    return max(steps, int(min_ms / per) + 1)


def soak(torch, g, stream, lens, lens0, flush, seconds):
    """Untimed replays for `seconds` of wall time: the clocks settle under load and the clock
    sampler sees the workload before the timed steps."""
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        time_graph(torch, g, stream, lens, lens0, flush, 50)


def profile_kernels(torch, mla, layer, stream, call, lens, lens0, flush, steps):
    """Average device ms of each kernel of one call, from CUDA events the library records on
    the launching stream around every launch.  A bounded spin kernel (torch.cuda._sleep)
    holds the stream while the call is enqueued, so the events bracket device work only."""
    per = {}
    mla.mla_set_profiling(layer.ctx, True)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            lens.copy_(lens0)
            flush.zero_()
            torch.cuda._sleep(2_000_000)
            call()
            stream.synchronize()
            for kname, kms in mla.mla_last_launches(layer.ctx):
                per.setdefault(kname, []).append(kms)
    mla.mla_set_profiling(layer.ctx, False)
    return {k: sum(v) / len(v) for k, v in per.items()}


def run_decode_workload(torch, mla, synth, layer, name, lengths, build, steps, warmup, device,
                        flush, prof_steps=50, e2e=True, soak_s=0.0, min_ms=0.0):
    B = len(lengths)
    cache, lens, xb, x = setup_decode(torch, mla, synth, layer, 0, lengths, build, device)
    lens0 = lens.clone()
    out = torch.empty_like(x)
    stream = torch.cuda.Stream(device=device)
    ws = layer.workspace(B, 1)
    host_lens = list(lengths)

    def call(st=None):
        mla.mla_decode(layer.ctx, x, cache, lens, host_lens, out, ws, stream=st)

    with torch.cuda.stream(stream):
        for _ in range(3):
            lens.copy_(lens0)
            call(stream)
    stream.synchronize()
    graphs = {}
    g = torch.cuda.CUDAGraph()
    lens.copy_(lens0)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        call()
    graphs[False] = g
    launches = mla.load().mla_last_launches(layer.ctx, 0, None, None)

    time_graph(torch, graphs[False], stream, lens, lens0, flush, warmup)
    soak(torch, graphs[False], stream, lens, lens0, flush, soak_s)
    if min_ms > 0:
        steps = steps_for(torch, graphs[False], stream, lens, lens0, flush, steps, min_ms)
    t0 = time.perf_counter()
    times = time_graph(torch, graphs[False], stream, lens, lens0, flush, steps)
    wall = time.perf_counter() - t0
    ms = sum(times) / len(times)

    per_ms = profile_kernels(torch, mla, layer, stream, lambda: call(stream), lens, lens0,
                             flush, prof_steps)

    e2e_res = None
    if e2e:
        # One C-ABI call per step with the input and output in pinned host memory: the call
        # enqueues the host-to-device copy, the step and the device-to-host copy.
        xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        xh.copy_(x.cpu())
        yh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        wsh = torch.empty(mla.mla_decode_host_workspace_bytes(layer.ctx, B), dtype=torch.uint8,
                          device=device)
        evs = []
        with torch.cuda.stream(stream):
            for k in range(warmup + max(20, steps // 10)):
                lens.copy_(lens0)
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                mla.mla_decode_host(layer.ctx, xh, cache, lens, host_lens, yh, wsh, stream=stream)
                e1.record(stream)
                stream.synchronize()
                if k >= warmup:
                    evs.append(e0.elapsed_time(e1))
        e2e_ms = sum(evs) / len(evs)
        e2e_res = {"value": B * 1000.0 / e2e_ms, "unit": "tokens/s",
                   "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": out.numel() * 2,
                   "ms_per_step": e2e_ms,
                   "path": "mla_decode_host via ctypes, pinned host buffers, copies in the call"}
    del cache
    return {"name": name, "B": B, "lengths": lengths, "ms": ms, "times": times, "wall": wall,
            "steps": steps,
            "per_kernel_ms": per_ms, "launches_per_step": launches, "e2e": e2e_res,
            "xb": xb}


def run_prefill_workload(torch, mla, synth, layer, T, steps, warmup, device, flush, min_ms=0.0):
    xb = synth.hidden_states(0, 0, 0, T)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(device)[None]
    cache = torch.zeros(1, T, 576, dtype=torch.bfloat16, device=device)
    lens = torch.zeros(1, dtype=torch.int32, device=device)
    lens0 = lens.clone()
    out = torch.empty_like(x)
    ws = layer.workspace(1, T)
    stream = torch.cuda.Stream(device=device)
    with torch.cuda.stream(stream):
        mla.mla_prefill(layer.ctx, x, cache, lens, [0], out, ws, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    lens.copy_(lens0)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        mla.mla_prefill(layer.ctx, x, cache, lens, [0], out, ws)
    time_graph(torch, g, stream, lens, lens0, flush, warmup)
    if min_ms > 0:
        steps = steps_for(torch, g, stream, lens, lens0, flush, steps, min_ms)
    times = time_graph(torch, g, stream, lens, lens0, flush, steps)
    per = profile_kernels(torch, mla, layer, stream,
                          lambda: mla.mla_prefill(layer.ctx, x, cache, lens, [0], out, ws,
                                                  stream=stream),
                          lens, lens0, flush, max(2, steps // 2))
    return {"T": T, "ms": sum(times) / len(times), "per_kernel_ms": per, "steps": steps}


def run_chunk_workload(torch, mla, synth, layer, L, T, steps, warmup, device, flush, min_ms=0.0):
    """Chunked prefill: T new tokens after L cached positions (B=1).  The cache is built by a
    prefill of the first L tokens outside the timed region; every step restores the length
    to L, so each step recomputes the same chunk."""
    xb = synth.hidden_states(0, 0, 0, L + T)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(device)[None]
    cache = torch.zeros(1, L + T, 576, dtype=torch.bfloat16, device=device)
    lens = torch.zeros(1, dtype=torch.int32, device=device)
    layer.prefill(x[:, :L].contiguous(), cache, lens, [0])
    torch.cuda.synchronize()
    lens0 = lens.clone()
    xc = x[:, L:].contiguous()
    out = torch.empty_like(xc)
    ws = layer.workspace(1, T, L + T)
    stream = torch.cuda.Stream(device=device)
    with torch.cuda.stream(stream):
        mla.mla_prefill(layer.ctx, xc, cache, lens, [L], out, ws, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    lens.copy_(lens0)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        mla.mla_prefill(layer.ctx, xc, cache, lens, [L], out, ws)
    time_graph(torch, g, stream, lens, lens0, flush, warmup)
    if min_ms > 0:
        steps = steps_for(torch, g, stream, lens, lens0, flush, steps, min_ms)
    times = time_graph(torch, g, stream, lens, lens0, flush, steps)
    per = profile_kernels(torch, mla, layer, stream,
                          lambda: mla.mla_prefill(layer.ctx, xc, cache, lens, [L], out, ws,
                                                  stream=stream),
                          lens, lens0, flush, max(2, steps // 2))
    return {"ms": sum(times) / len(times), "per_kernel_ms": per, "steps": steps}


def chunk_flops(L, T):
    """Algorithmic FLOPs of a T-token chunk after L cached positions: the projections of the T
    new tokens, kv_b_proj over all L + T latent rows (the explicit form rebuilds the cached
    keys and values), and the attention of query t over keys 0..L+t."""
    gemm = 2 * T * (7168 * 2112 + 1536 * 12288 + 8192 * 7168) + 2 * (L + T) * 512 * 16384
    pairs = T * L + T * (T + 1) // 2
    return gemm, 2 * 64 * pairs * (192 + 128)


def prefill_flops(T):
    """Algorithmic FLOPs of one causal prefill of T tokens (GEMMs + causal QK^T and PV)."""
    gemm = 2 * T * (7168 * 2112 + 1536 * 12288 + 512 * 16384 + 8192 * 7168)
    pairs = T * (T + 1) // 2
    attn = 2 * 64 * pairs * (192 + 128)
    return gemm, attn


def init_replicas(dist, backend):
    """Rank, world size and local rank from the launcher's environment; joins the process group
    when there is more than one rank.  Each rank is an independent replica of the whole step:
    the only traffic between ranks is the barrier around the timed region and the reduction of
    its result."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group(backend)
    return world, rank, local


def aggregate_replicas(torch, dist, ms, units, device="cpu"):
    """Whole-job figure over all replicas: the slowest rank's step time (ms), the units every
    rank processed per step, and units per second over that time.  `dist` is None on one rank."""
    if dist is None:
        return ms, units, units * 1000.0 / ms
    t_ms = torch.tensor([ms], dtype=torch.float64, device=device)
    t_units = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t_ms, op=dist.ReduceOp.MAX)
    dist.all_reduce(t_units, op=dist.ReduceOp.SUM)
    ms_max, total = float(t_ms.item()), int(round(t_units.item()))
    return ms_max, total, total * 1000.0 / ms_max


def gpu_arm(args):
    import torch
    import torch.distributed as dist
    from head_latent_attention_mla_gb300 import mla, synth

    world, rank, local = init_replicas(dist, "nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    mla.load()
    wq, gains = synth.make_weights(0), synth.make_gains(0)
    layer = mla.MlaLayer(wq, gains, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    pk = peaks()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # --- headline: decode B=1 at position 1000 -------------------------------------------
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_idx = int(vis.split(",")[local]) if vis and vis.split(",")[local].isdigit() else local
    barrier()
    # The clock sampler runs from the start of the warm-up (which replays the step for a
    # third of a second, so it holds samples under load) to the end of the timed steps.
    with ClockSampler(gpu_idx) as clk:
        clk.start()
        res = run_decode_workload(torch, mla, synth, layer, "decode_b1_p1000", [1000], "prefill",
                                  args.steps, args.warmup, device, flush, soak_s=0.35)
    barrier()
    B = res["B"]
    ms, _, value = aggregate_replicas(torch, dist if world > 1 else None, res["ms"], B, device)
    per = res["per_kernel_ms"]
    dom = max(per, key=per.get)
    abytes = algorithmic_bytes(dom, B, res["lengths"])
    achieved = abytes / (per[dom] * 1e-3) / 1e9
    cache_bytes = sum(n + 1 for n in res["lengths"]) * LAT_BYTES
    att_ms = per.get("decode_attention")

    extra = {}
    if not args.headline_only and rank == 0:
        with ClockSampler(gpu_idx) as clk2:
            clk2.start()
            extra = secondary(torch, mla, synth, layer, device, flush, pk, args, wq, gains)
        extra["clocks"] = clk2.summary()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    cpu = cpu_baseline_decode(res["xb"], args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 states; N(0,0.02) weights as e4m3 with 128x128 "
                "block scales amax/448; gains 1+U(-0.1,0.1))",
        "config": {"workload": "decode B=1, cache of 1000 positions built by causal prefill, "
                               "new token at position 1000 attending to 1001 positions",
                   "batch": B, "cached_positions": res["lengths"], "layer": "Kimi-K2 MLA (7168/1536/512/64 heads/128+64/128)",
                   "weights": "e4m3, 128x128 fp32 block scales", "activations": "bf16",
                   "l2": "flushed (256 MiB write) between timed steps", "graph": "CUDA graph of one mla_decode call",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                     "traffic": traffic_record(dom, "decode_b1_p1000"),
                     "algorithmic_bytes_per_launch": abytes, "launch_ms": per[dom],
                     "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
        "per_kernel_ms": per,
        "decode_attention_cache_gbs": (cache_bytes / (att_ms * 1e-3) / 1e9) if att_ms else None,
        "cpu_baseline": cpu,
        "e2e": res["e2e"],
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": clk.summary(),
        "timed_wall_s": res["wall"],
    }
    if extra:
        line["secondary"] = extra
    if world > 1:
        dist.destroy_process_group()
    return line


def secondary(torch, mla, synth, layer, device, flush, pk, args, wq, gains):
    """The other workloads' headline figures (not the bench value)."""
    out = {}
    steps, min_ms = 5, 200.0    # each workload is timed over at least 200 ms of steps
    for name, lengths, build in (("decode_long_b8_131072", [131072] * 8, "append"),
                                 ("decode_ragged_b64", synth.ragged_lengths(0, 64, 512, 8192).tolist(), "append")):
        r = run_decode_workload(torch, mla, synth, layer, name, lengths, build, steps, 3, device,
                                flush, prof_steps=20, e2e=False, min_ms=min_ms)
        att = r["per_kernel_ms"].get("decode_attention")
        cb = sum(n + 1 for n in lengths) * LAT_BYTES
        gbs = cb / (att * 1e-3) / 1e9 if att else None
        out[name] = {"tokens_per_s": len(lengths) * 1000.0 / r["ms"], "ms_per_step": r["ms"],
                     "decode_attention_ms": att, "attention_cache_gbs": gbs,
                     "attention_hbm_frac": gbs / pk["hbm_gbs"] if gbs else None,
                     "timed_steps": r["steps"], "per_kernel_ms": r["per_kernel_ms"]}
        torch.cuda.empty_cache()
    for T in (4096, 16):
        r = run_prefill_workload(torch, mla, synth, layer, T, steps, 3, device, flush, min_ms)
        gemm, attn = prefill_flops(T)
        out[f"prefill_t{T}"] = {"tokens_per_s": T * 1000.0 / r["ms"], "ms_per_step": r["ms"],
                                "timed_steps": r["steps"],
                                "tflops": (gemm + attn) / (r["ms"] * 1e-3) / 1e12,
                                "tensor_frac": (gemm + attn) / (r["ms"] * 1e-3) / 1e12 / pk["bf16_tflops"],
                                "per_kernel_ms": r["per_kernel_ms"]}
    # The FP8-activation option (one e4m3 activation term, one MMA per k step): its prefill
    # against the FP8 tensor peak (the measured bf16 peak times the nominal 2x ratio).
    layer8 = mla.MlaLayer(wq, gains, device=device, fp8_activations=1)
    r = run_prefill_workload(torch, mla, synth, layer8, 4096, steps, 3, device, flush, min_ms)
    layer8.close()
    gemm, attn = prefill_flops(4096)
    tf = (gemm + attn) / (r["ms"] * 1e-3) / 1e12
    out["prefill_t4096_fp8_activations"] = {
        "tokens_per_s": 4096 * 1000.0 / r["ms"], "ms_per_step": r["ms"], "timed_steps": r["steps"],
        "tflops": tf, "tensor_frac_of_fp8_peak": tf / (2.0 * pk["bf16_tflops"]),
        "fp8_peak_tflops": 2.0 * pk["bf16_tflops"], "fp8_peak_source": "measured bf16 x 2 (nominal 4.5/2.25)",
        "per_kernel_ms": r["per_kernel_ms"]}
    torch.cuda.empty_cache()
    L, T = 4096, 1024
    r = run_chunk_workload(torch, mla, synth, layer, L, T, steps, 3, device, flush, min_ms)
    gemm, attn = chunk_flops(L, T)
    out[f"prefill_chunk_l{L}_t{T}"] = {
        "tokens_per_s": T * 1000.0 / r["ms"], "ms_per_step": r["ms"], "timed_steps": r["steps"],
        "tflops": (gemm + attn) / (r["ms"] * 1e-3) / 1e12,
        "tensor_frac": (gemm + attn) / (r["ms"] * 1e-3) / 1e12 / pk["bf16_tflops"],
        "per_kernel_ms": r["per_kernel_ms"]}
    return out


# ------------------------------------------------------------------------------- CPU oracle
def cpu_baseline_decode(xb, seconds):
    """The fp64 oracle's decode step (explicit form) on the host cores, B=1 at p=1000."""
    from head_latent_attention_mla_gb300 import synth
    from oracle import mla_oracle as O
    wq, g = synth.make_weights(0), synth.make_gains(0)
    W = O.weights_from_quantised(wq, g)
    xf = O.bf16_to_f64(synth.hidden_states(0, 0, 0, 1000))
    cache = O.cache_rows(xf, np.arange(1000), W)
    xn = O.bf16_to_f64(xb[0])
    O.decode(xn, cache, W)
    reps, t0 = 0, time.perf_counter()
    while True:
        O.decode(xn, cache, W)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 200:
            break
    return {"value": reps / el, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} full decode steps (B=1, p=1000, explicit fp64 form) in {el:.1f} s; "
                      "numpy BLAS with its default thread count"}


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from head_latent_attention_mla_gb300 import synth
    xb = synth.hidden_states(0, 0, 1000, 1)
    cpu = cpu_baseline_decode(xb, args.cpu_seconds)
    v = cpu["value"]
    return {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "decode B=1, cache of 1000 positions built by causal prefill, "
                                   "new token at position 1000 attending to 1001 positions",
                       "batch": 1, "cached_positions": [1000]},
            "cpu_baseline": cpu,
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def case_arm(args):
    """One workload, small enough to profile: `decode:B:L` (B sequences with L cached positions
    each, cache built by append), `prefill:T` (one sequence of T tokens) or `chunk:L:T` (T new
    tokens after L cached positions).  Prints a short JSON line with the step time and
    per-kernel device times."""
    import torch
    from head_latent_attention_mla_gb300 import mla, synth
    torch.cuda.set_device(0)
    device = "cuda:0"
    layer = mla.MlaLayer(synth.make_weights(0), synth.make_gains(0), device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    kind, *dims = args.case.split(":")
    if kind == "decode":
        B, L = int(dims[0]), int(dims[1])
        r = run_decode_workload(torch, mla, synth, layer, args.case, [L] * B, "append",
                                args.steps, args.warmup, device, flush, prof_steps=3, e2e=False)
    elif kind == "chunk":
        r = run_chunk_workload(torch, mla, synth, layer, int(dims[0]), int(dims[1]), args.steps,
                               args.warmup, device, flush)
    else:
        r = run_prefill_workload(torch, mla, synth, layer, int(dims[0]), args.steps,
                                 args.warmup, device, flush)
    return {"case": args.case, "ms_per_step": r["ms"], "per_kernel_ms": r["per_kernel_ms"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--case", default=None,
                    help="profiling case instead of the benchmark line: decode:B:L, prefill:T "
                         "or chunk:L:T")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        line = case_arm(args)
    else:
        line = reference_arm(args) if args.impl == "reference" else gpu_arm(args)
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
