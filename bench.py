#!/usr/bin/env python
"""Decode throughput of the NOSA attention path on GB300.

A step is one decode step of the whole attention stack: for every layer,
append the new token (host store + cache slot, eviction score, compressed
key), score and select blocks, gather the newly selected blocks from pinned
host memory, and attend over the selection -- all in libnosa.so kernels.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl native|reference]

N > 1 runs under torchrun with one process per GPU; every rank serves its own
batch (independent sequences, no collective on the data path: weak scaling).
Inputs are synthetic (seeded), shaped like the workload; the full K/V context
lives in pinned host memory before timing starts.

Rank 0 prints one JSON line.  Beside the contract's keys (value = tok/s of the
whole stack from CUDA events around K graph-replayed steps, max over ranks):
  roofline            the dominant kernel's algorithmic bytes / its mean launch
                      time (isolated launches of the per-kernel leg) against
                      MEASURED_PEAKS' HBM copy bandwidth; in_step = the score,
                      select and attend bytes of every layer / ms_per_step;
                      traffic = stored ncu DRAM bytes per launch while the
                      kernel's sources still hash to the capture's
  fetch_roofline      the gather kernel on the step's fetch list against the
                      best pinned 1 GiB host-to-device copy of the same run;
                      in_attend = the new blocks' bytes / the attention launch
                      that copies them; in_step = fetched bytes / ms_per_step
  hbm_frac_score_select_attend, stages_us_per_layer (per-kernel leg), gamma,
  fetch_blocks_per_step, short_selections, clocks (nvidia-smi samples taken
  during the timed region), gpu_launches (this library's kernels in the timed
  region), plan (the kernels nosa_step runs)
  e2e                 the same metric through the public API on pinned host
                      buffers, copies inside the timed region (device, host wall
                      and host busy time per step reported)
  cpu_baseline        the oracle on a bounded sample on the host cores (rank 0)
--impl reference times the oracle alone (this path has no other reference
implementation); --quick keeps only the timed leg (profiling runs); --forecast
runs the SparDA-style pipeline (every leg above, on its kernels); the sizing
flags set nosa_config's kernel sizing fields.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s (attn path, 1 GB300) + % HBM roofline and % PCIe H2D BW for fetch"
BLOCK_BYTES = 32768


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="nosa8b_32k_b32",
                    help="default: the 8B-shaped stack (32 layers, 32/8 heads, 32K context, batch 32), the "
                         "largest workload that fits one GPU and its host")
    ap.add_argument("--sigma", type=float, default=None)
    ap.add_argument("--k-q", type=int, default=None)
    ap.add_argument("--gather-ctas", type=int, default=0)
    ap.add_argument("--layers", type=int, default=None, help="fewer layers (only for host-memory limits)")
    ap.add_argument("--batch", type=int, default=None,
                    help="fewer sequences than the workload's batch (--prefill only: small cases for profiling)")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--dma-bias", action="store_true", help="attention adds each token's eviction score (DMA bias)")
    ap.add_argument("--dense", action="store_true",
                    help="full-attention comparator: dense decode attention over a device-resident KV cache")
    ap.add_argument("--forecast", action="store_true",
                    help="SparDA-style selection one layer ahead from forecast vectors, the next layer's "
                         "selection and prefetch overlapping the current layer (timed leg only)")
    ap.add_argument("--quick", action="store_true", help="timed graph leg only (profiling runs)")
    # kernel sizing overrides (nosa_config fields; 0 = the library's rule)
    for f in ("score-ctas", "attend-blocks-per-cta", "attend-merge", "decode-cluster", "decode-teams",
              "decode-stages", "forecast-streams", "cache-slots"):
        ap.add_argument(f"--{f}", type=int, default=0)
    ap.add_argument("--unfused", action="store_true", help="three-kernel step even where the fused kernel fits")
    ap.add_argument("--prefill", action="store_true",
                    help="NOSA_S sparse prefill of the workload's context length as one prompt, every layer, "
                         "from empty layers (nosa_prefill); prints a prefill tok/s line")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


# ---------------------------------------------------------------------------- helpers
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
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
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# the sources each measured kernel is compiled from
KERNEL_SOURCES = {
    "decode_kernel": ["decode.cu", "append_core.cuh", "select_core.cuh", "attend_core.cuh", "ptx.cuh",
                      "nosa_internal.cuh"],
    "attend_kernel": ["attend.cu", "attend_core.cuh", "ptx.cuh", "nosa_internal.cuh"],
    "score_select_kernel": ["select.cu", "select_core.cuh", "append_core.cuh", "ptx.cuh", "nosa_internal.cuh"],
}


def kernel_source_hash(kernel):
    """sha256 over a kernel's sources, to tell whether stored ncu counters still describe it."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, []):
        h.update(f.encode())
        with open(os.path.join(ROOT, "offloadable_block_sparse_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def captured_traffic(kernel, key):
    """DRAM bytes per launch of `kernel` on workload `key` from a stored ncu capture, or (None, why)."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None, "no capture"
    e = data.get("entries", {}).get(f"{kernel}|{key}")
    if not e:
        return None, "no capture of this kernel and workload"
    if e.get("source_hash") != kernel_source_hash(kernel):
        return None, "kernel changed since the capture"
    return e["dram_bytes_per_launch"], e["capture"]


def h2d_peak(torch, nbytes=1 << 30, reps=6):
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        d.copy_(h, non_blocking=True)
        e.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (s.elapsed_time(e) * 1e-3) / 1e9)
    del h, d
    return best


def oracle_baseline(wl, seconds, total_units):
    """Time the CPU oracle on a bounded sample of the workload (a few units' decode steps)."""
    from oracle import nosa_oracle as O
    from synth import inputs as syn
    samples = []
    lbg = [(0, 0, 0), (wl.layers - 1, wl.batch - 1, wl.kv_heads - 1), (wl.layers // 2, wl.batch // 2, 0),
           (1 % wl.layers, wl.batch - 1, 0)]
    for (l, b, g) in lbg:
        x = wl.unit_inputs(l, b, g)
        o = O.UnitOracle(head_dim=wl.head_dim, k_q=wl.k_q, k_e=wl.k_e, sink_blocks=wl.sink_blocks,
                         window_tokens=wl.window_tokens, max_context=wl.max_context, W1=x["W1"], W2=x["W2"])
        o.append(x["K"][:wl.context], x["V"][:wl.context])
        samples.append((o, x))
    n = 0
    t0 = time.perf_counter()
    t = 0
    while time.perf_counter() - t0 < seconds and t < wl.steps:
        for o, x in samples:
            p = wl.context + t
            o.step(x["Q"][t], x["K"][p:p + 1], x["V"][p:p + 1])
            n += 1
        t += 1
    dt = time.perf_counter() - t0
    per_unit = dt / max(n, 1)
    value = wl.batch / (per_unit * total_units)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} unit-steps ({len(samples)} units x {t} decode steps) of {total_units} units/step, "
                      f"{dt:.1f} s; numpy float64 with its default BLAS threading"}


def sizing_overrides(args):
    """nosa_config sizing fields set on the command line (0 = the library's rule)."""
    return {k: getattr(args, k) for k in ("score_ctas", "attend_blocks_per_cta", "attend_merge", "decode_cluster",
                                          "decode_teams", "decode_stages", "forecast_streams", "cache_slots")}


def workload_config(wl, args, layers, world):
    """The `config` object of the JSON line: the workload, as both arms print it."""
    cfg = {"workload": wl.name, "layers": layers, "batch_per_gpu": wl.batch, "q_heads": wl.q_heads,
           "kv_heads": wl.kv_heads, "head_dim": wl.head_dim, "context": wl.context, "k_q": wl.k_q, "k_e": wl.k_e,
           "sink_blocks": wl.sink_blocks, "window_tokens": wl.window_tokens, "sigma": wl.sigma,
           "parallelism": f"replicas x{world} (independent sequences per GPU)",
           "dma_bias": bool(args.dma_bias),
           "selection": "forecast one layer ahead, overlapped prefetch" if args.forecast else "query (per step)",
           "l2": "no flush: one step reads > 1 GB of distinct K/V, compressed keys and cache (L2 is 129 MB)"}
    over = {k: v for k, v in sizing_overrides(args).items() if v}
    if over:
        cfg["sizing"] = over
    return cfg


def slowest_rank_ms(ms: float, world: int, device: str = "cpu") -> float:
    """Per-step time of the slowest rank (max over ranks; every rank must call it)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(batch_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job decode tokens/s: every rank serves its own batch (weak scaling)."""
    return world * batch_per_rank / (ms_per_step * 1e-3)


# ---------------------------------------------------------------------------- native arm
def run_native(args, rank, world, local_rank):
    import torch
    from offloadable_block_sparse_gb300 import nosa as N
    from synth import inputs as syn
    torch.cuda.set_device(local_rank)
    dev = "cuda"
    over = {}
    if args.sigma is not None:
        over["sigma"] = args.sigma
    if args.k_q is not None:
        over["k_q"], over["k_e"] = args.k_q, 64 - args.k_q
    wl = syn.workload(args.workload, **over)
    L = args.layers or wl.layers
    B, Hq, Hkv, d = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim
    U = B * Hkv
    K, W = args.steps, args.warmup
    n_time_leg = 0 if args.quick else 3 * min(K, 6)
    n_e2e = 0 if args.quick else min(K, 64)
    n_e2e_warm = 6 if n_e2e else 0  # two untimed replays of each e2e graph (the first uploads it)
    total_steps = 1 + W + K + n_time_leg + n_e2e_warm + n_e2e
    flags = (N.NOSA_F_DMA_BIAS if args.dma_bias else 0) | (N.NOSA_F_UNFUSED_STEP if args.unfused else 0)
    cfg = N.make_config(num_layers=L, batch=B, num_q_heads=Hq, num_kv_heads=Hkv, k_q=wl.k_q, k_e=wl.k_e,
                        window_tokens=wl.window_tokens, max_context=wl.context + total_steps,
                        sink_blocks=wl.sink_blocks, evict_hidden=wl.evict_hidden, gather_ctas=args.gather_ctas,
                        flags=flags, **sizing_overrides(args))
    stream = torch.cuda.current_stream()
    ctx = N.nosa_create(cfg, stream.cuda_stream)
    sizes = N.nosa_query_sizes(cfg)
    step_kernels, decode_cluster = N.nosa_step_plan(ctx)
    gen = torch.Generator(device=dev).manual_seed(1000 * rank + 7)
    cgen = torch.Generator().manual_seed(1000 * rank + 11)
    for l in range(L):
        W1 = (torch.randn((Hkv, d, wl.evict_hidden), generator=cgen) / math.sqrt(d)).float().contiguous()
        W2 = (torch.randn((Hkv, wl.evict_hidden), generator=cgen) / math.sqrt(wl.evict_hidden)).float().contiguous()
        N.nosa_set_eviction_head(ctx, l, W1.numpy(), W2.numpy())
        Kc = torch.randn((B, Hkv, wl.context, d), generator=gen, device=dev).to(torch.bfloat16)
        Vc = torch.randn((B, Hkv, wl.context, d), generator=gen, device=dev).to(torch.bfloat16)
        N.nosa_append_kv(ctx, l, Kc.view(torch.int16), Vc.view(torch.int16), wl.context)
        del Kc, Vc
    torch.cuda.synchronize()
    # per-step inputs: random-walk queries (normalised, sqrt(d) norm), fresh N(0,1) keys/values
    qs = torch.randn((L, B, Hq, d), generator=gen, device=dev)
    qs = qs / qs.norm(dim=-1, keepdim=True) * math.sqrt(d)
    Qall = torch.empty((total_steps, L, B, Hq, d), dtype=torch.bfloat16, device=dev)
    for t in range(total_steps):
        qs = qs + wl.sigma * torch.randn(qs.shape, generator=gen, device=dev)
        qs = qs / qs.norm(dim=-1, keepdim=True) * math.sqrt(d)
        Qall[t] = qs.to(torch.bfloat16)
    KVall = torch.randn((total_steps, 2, L, B, Hkv, d), generator=gen, device=dev).to(torch.bfloat16)
    fc = args.forecast
    if fc:  # forecast vectors: one random walk per (layer, sequence, kv head), like the queries
        fs = torch.randn((L, B, Hkv, d), generator=gen, device=dev)
        fs = fs / fs.norm(dim=-1, keepdim=True) * math.sqrt(d)
        Fall = torch.empty((total_steps + 1, L, B, Hkv, d), dtype=torch.bfloat16, device=dev)
        for t in range(total_steps + 1):
            fs = fs + wl.sigma * torch.randn(fs.shape, generator=gen, device=dev)
            fs = fs / fs.norm(dim=-1, keepdim=True) * math.sqrt(d)
            Fall[t] = fs.to(torch.bfloat16)
        cur_f = torch.empty((L, B, Hkv, d), dtype=torch.bfloat16, device=dev)
        cur_f0n = torch.empty((B, Hkv, d), dtype=torch.bfloat16, device=dev)  # layer 0, next step
    out = torch.empty((L, B, Hq, d), dtype=torch.bfloat16, device=dev)
    cur_q = torch.empty((L, B, Hq, d), dtype=torch.bfloat16, device=dev)
    cur_kv = torch.empty((2, L, B, Hkv, d), dtype=torch.bfloat16, device=dev)
    i16 = torch.int16
    step_i = [0]

    def forecast_calls(q, kv, f, f0n):
        # layer l's call starts layer l+1's forecast and prefetch; the last layer forecasts layer 0
        # of the next step; the step ends joined to the prefetch stream
        for l in range(L):
            fn, nxt = (f[l + 1], l + 1) if l + 1 < L else (f0n, 0)
            N.nosa_step_forecast(ctx, l, q[l].view(i16), kv[0, l].view(i16), kv[1, l].view(i16), out[l].view(i16),
                                 fn.view(i16), nxt)
        N.nosa_forecast_join(ctx)

    def eager_step(t):
        if fc:
            forecast_calls(Qall[t], KVall[t], Fall[t], Fall[t + 1, 0])
            return
        for l in range(L):
            N.nosa_step(ctx, l, Qall[t, l].view(i16), KVall[t, 0, l].view(i16), KVall[t, 1, l].view(i16),
                        out[l].view(i16))

    # step 1 (cold fetch of every selected block) is not timed
    if fc:
        N.nosa_forecast_select(ctx, 0, Fall[0, 0].view(i16))
    eager_step(0)
    step_i[0] = 1
    use_graph = not args.no_graph
    graph = None
    if use_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        N.nosa_set_stream(ctx, side.cuda_stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            if fc:
                forecast_calls(cur_q, cur_kv, cur_f, cur_f0n)
            else:
                for l in range(L):
                    N.nosa_step(ctx, l, cur_q[l].view(i16), cur_kv[0, l].view(i16), cur_kv[1, l].view(i16),
                                out[l].view(i16))
        N.nosa_set_stream(ctx, stream.cuda_stream)
        assert N.nosa_sync(ctx) == N.NOSA_OK

    def run_step(t):
        if use_graph:
            cur_q.copy_(Qall[t], non_blocking=True)
            cur_kv.copy_(KVall[t], non_blocking=True)
            if fc:
                cur_f.copy_(Fall[t], non_blocking=True)
                cur_f0n.copy_(Fall[t + 1, 0], non_blocking=True)
            graph.replay()
        else:
            eager_step(t)

    for _ in range(W):
        run_step(step_i[0])
        step_i[0] += 1
    N.nosa_reset_stats(ctx)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading before the timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        run_step(step_i[0])
        step_i[0] += 1
    e1.record()
    torch.cuda.synchronize()
    ck = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1) / K
    st = N.nosa_sync(ctx)
    if st != N.NOSA_OK:
        raise RuntimeError(f"device error {N.STATUS_NAMES[st]}")
    stats = N.nosa_get_stats(ctx)
    ms = slowest_rank_ms(ms, world, dev)
    value = job_throughput(B, world, ms)
    fetched_per_step = stats.blocks_fetched / K

    result = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
              "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "dtype": "bf16", "data": "synthetic",
              "config": workload_config(wl, args, L, world),
              "plan": {"cuda_graph": use_graph, "gather_ctas": args.gather_ctas or (16 if B < 32 else 32),
                       "step_kernels_per_layer": step_kernels, "decode_cluster": decode_cluster,
                       "cache_slots": sizes.cache_slots, "select_slots": sizes.select_slots},
              # forecast: forecast select and gather (prefetch stream), append, attention, merge
              "gpu_launches": (5 if fc else step_kernels) * L * K,
              "clocks": ck,
              "gamma": {"mean": stats.gamma_mean, "min": stats.gamma_min, "bound": wl.k_e / (wl.k_q + wl.k_e)},
              "fetch_blocks_per_step": fetched_per_step,
              "short_selections": stats.short_selections}
    if args.quick or rank != 0:
        N.nosa_destroy(ctx)
        return result

    # ---------------- per-kernel leg: one event pair around each launch, on the launching stream.
    # Plain mode cycles three kinds of step: (0) nosa_step per layer (the fused decode kernel, or
    # the chain); (1) the separate calls append, select and attend, the attention copying the new
    # blocks from host memory itself, as in the timed step ("attend_fetch"); (2) append, select,
    # the standalone gather (nosa_fetch) on that fresh fetch list, then the attention over blocks
    # that are all resident ("attend": HBM only).  Forecast mode: every step times the forecast
    # path's kernels as separate calls on the step stream: forecast selection, the gather of its
    # new blocks, append, attention.
    ev = {k: [] for k in ("decode", "append", "select", "attend_fetch", "attend", "gather", "fselect")}
    fetched = {"fetch": 0, "gather": 0}
    steps_of = {"fetch": 0, "gather": 0}
    for it in range(n_time_leg):
        t = step_i[0]
        step_i[0] += 1
        kind = "gather" if fc else ("decode", "fetch", "gather")[it % 3]
        if kind != "decode":
            s0 = N.nosa_get_stats(ctx).blocks_fetched
            steps_of[kind] += 1
        for l in range(L):
            pairs = []
            # hold the stream while the launches and their events are queued, so that the
            # events time the kernels back to back rather than the host's launch latency
            torch.cuda._sleep(400000)
            if fc:
                # after the timed graphs layer 0 of this step already has its forecast selection
                calls = [] if (it == 0 and l == 0) else [
                    ("fselect", lambda: N.nosa_forecast_select(ctx, l, Fall[t, l].view(i16)))]
                calls += [("gather", lambda: N.nosa_fetch(ctx, l)),
                          ("append", lambda: N.nosa_append_kv(ctx, l, KVall[t, 0, l].view(i16),
                                                              KVall[t, 1, l].view(i16), 1)),
                          ("attend", lambda: N.nosa_attend(ctx, l, Qall[t, l].view(i16), out[l].view(i16)))]
            elif kind == "decode":
                calls = [("decode", lambda: N.nosa_step(ctx, l, Qall[t, l].view(i16), KVall[t, 0, l].view(i16),
                                                        KVall[t, 1, l].view(i16), out[l].view(i16)))]
            else:
                calls = [("append", lambda: N.nosa_append_kv(ctx, l, KVall[t, 0, l].view(i16),
                                                             KVall[t, 1, l].view(i16), 1)),
                         ("select", lambda: N.nosa_select(ctx, l, Qall[t, l].view(i16)))]
                if kind == "gather":
                    calls += [("gather", lambda: N.nosa_fetch(ctx, l)),
                              ("attend", lambda: N.nosa_attend(ctx, l, Qall[t, l].view(i16), out[l].view(i16)))]
                else:
                    calls += [("attend_fetch", lambda: N.nosa_attend(ctx, l, Qall[t, l].view(i16),
                                                                     out[l].view(i16)))]
            for name, fn in calls:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                pairs.append((name, a, b))
            torch.cuda.synchronize()
            for name, a, b in pairs:
                ev[name].append(a.elapsed_time(b) * 1e3)
        if kind != "decode":
            fetched[kind] += N.nosa_get_stats(ctx).blocks_fetched - s0
    us = {k: statistics.mean(v) for k, v in ev.items() if v}
    G = Hq // Hkv
    T_now = N.nosa_context_length(ctx, 0)
    valid_tail = T_now - 64 * ((T_now + 63) // 64 - 1)
    nc = (T_now - 32) // 16 + 1
    nb = (T_now + 63) // 64
    attend_layers = []
    for l in range(L):  # every layer's selection sizes: algorithmic K+V bytes of its attention
        n_sel = np.zeros(U, np.int32)
        N.nosa_export_state(ctx, l, n_sel=n_sel)
        attend_layers.append(float(np.sum((n_sel.astype(np.int64) * 64 - (64 - valid_tail)) * d * 2 * 2))
                             + 2 * U * G * d * 2)
    attend_bytes = statistics.mean(attend_layers)
    select_bytes = U * (nc * d * 2 + nb * 4 + G * d * 2)
    fetch_bytes_launch = fetched["gather"] / max(steps_of["gather"] * L, 1) * BLOCK_BYTES
    fetch_bytes_attend = fetched["fetch"] / max(steps_of["fetch"] * L, 1) * BLOCK_BYTES
    hbm, src = measured_peaks()
    peak_src = f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured" else "fallback"
    if step_kernels == 1 and not fc:
        dominant, dom_bytes = "decode", attend_bytes + select_bytes
        note = ("fused decode kernel (append + score + select + fetch + attend); bytes = compressed keys, "
                "pooled scores and q read by the scorer plus K+V of every selected token read by the attention "
                "and its output; the newly selected blocks among them arrive over the host link inside the kernel")
    else:
        # the attention as the timed step runs it: with its own host copies in plain mode, over
        # prefetched blocks in forecast mode
        att = "attend" if fc else "attend_fetch"
        hbm_kernels = {att: attend_bytes, "fselect" if fc else "select": select_bytes}
        dominant = max(hbm_kernels, key=lambda k: us[k])
        dom_bytes = hbm_kernels[dominant]
        note = ("attend bytes = K+V of every selected token and the output; in plain mode the newly selected "
                "blocks among them arrive over the host link inside the same kernel, in forecast mode the "
                "gather copied them before")
    ach = dom_bytes / (us[dominant] * 1e-6) / 1e9
    kname = ("score_select_kernel" if dominant in ("select", "fselect") else
             "attend_kernel" if dominant.startswith("attend") else f"{dominant}_kernel")
    traffic, traffic_src = captured_traffic(kname, f"{wl.name}|sigma{wl.sigma}|kq{wl.k_q}|dma{int(args.dma_bias)}")
    step_bytes = float(sum(attend_layers)) + L * select_bytes
    in_step = step_bytes / (ms * 1e-3) / 1e9
    result["roofline"] = {"kernel": kname, "bound": "hbm", "achieved": ach, "peak": hbm,
                          "peak_source": peak_src, "unit": "GB/s", "frac": ach / hbm, "traffic": traffic,
                          "traffic_source": traffic_src, "algorithmic_bytes_per_launch": dom_bytes,
                          "avg_launch_us": us[dominant],
                          "how": "events around each launch of the per-kernel leg (isolated launches)",
                          "in_step": {"achieved": in_step, "frac": in_step / hbm, "unit": "GB/s",
                                      "algorithmic_bytes_per_step": step_bytes,
                                      "how": "score + select + attend bytes of every layer / ms_per_step of the "
                                             "timed graph leg"},
                          "note": note}
    if "attend" in us:  # the same attention over blocks already resident: its HBM rate alone
        a_hbm = attend_bytes / (us["attend"] * 1e-6) / 1e9
        result["roofline"]["attend_resident"] = {
            "achieved": a_hbm, "frac": a_hbm / hbm, "avg_launch_us": us["attend"],
            "how": "attend_kernel after nosa_fetch copied the step's new blocks: every block read from HBM"}
    result["stages_us_per_layer"] = us
    att_us = us["decode"] if (step_kernels == 1 and not fc) else us["attend" if fc else "attend_fetch"]
    sel_att_us = att_us if (step_kernels == 1 and not fc) else att_us + us.get("select", us.get("fselect", 0))
    result["hbm_frac_score_select_attend"] = (attend_bytes + select_bytes) / (sel_att_us * 1e-6) / 1e9 / hbm

    # ---------------- e2e through the public API, copies inside the timed region.  Plain mode:
    # nosa_step_host_all (one host-to-device copy of every layer's q, k, v, the layers' steps, one
    # device-to-host copy of the outputs).  Forecast mode: host-to-device copies of q, k, v and the
    # forecast vectors from pinned memory, the nosa_step_forecast calls, the device-to-host copy of
    # the outputs.  Three CUDA graphs, each capturing one step on its own set of pinned host
    # buffers, take turns: while one replays, the host reads the outputs of the set that finished
    # and writes the next step's inputs into it, up to two steps ahead of the device.
    e2e_graph = use_graph
    n_sets = 3
    sets = [dict(q=torch.empty((L, B, Hq, d), dtype=torch.bfloat16).pin_memory(),
                 kv=torch.empty((2, L, B, Hkv, d), dtype=torch.bfloat16).pin_memory(),
                 out=torch.empty((L, B, Hq, d), dtype=torch.bfloat16).pin_memory()) for _ in range(n_sets)]
    if fc:
        for bs in sets:
            bs["f"] = torch.empty((L + 1, B, Hkv, d), dtype=torch.bfloat16).pin_memory()  # layers, then next layer 0
    q_src = Qall[step_i[0]:step_i[0] + n_e2e_warm + n_e2e].cpu()
    kv_src = KVall[step_i[0]:step_i[0] + n_e2e_warm + n_e2e].cpu()
    if fc:
        f_src = torch.cat([Fall[step_i[0]:step_i[0] + n_e2e_warm + n_e2e],
                           Fall[step_i[0] + 1:step_i[0] + n_e2e_warm + n_e2e + 1, :1]], dim=1).cpu()
    outs_host = torch.zeros((n_e2e, L, B, Hq, d), dtype=torch.bfloat16)  # pages touched before the timing

    def host_step(bs):
        if not fc:
            N.nosa_step_host_all(ctx, bs["q"].view(i16), bs["kv"][0].view(i16), bs["kv"][1].view(i16),
                                 bs["out"].view(i16))
            return
        cur_q.copy_(bs["q"], non_blocking=True)
        cur_kv.copy_(bs["kv"], non_blocking=True)
        cur_f.copy_(bs["f"][:L], non_blocking=True)
        cur_f0n.copy_(bs["f"][L], non_blocking=True)
        forecast_calls(cur_q, cur_kv, cur_f, cur_f0n)
        bs["out"].copy_(out, non_blocking=True)

    def fill(bs, j):
        bs["q"].copy_(q_src[j])
        bs["kv"].copy_(kv_src[j])
        if fc:
            bs["f"].copy_(f_src[j])

    if fc:  # the pipeline expects layer 0's forecast for the next token to exist
        N.nosa_forecast_select(ctx, 0, Fall[step_i[0], 0].view(i16))
    graphs_e2e = []
    if e2e_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        N.nosa_set_stream(ctx, side.cuda_stream)
        for bs in sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                host_step(bs)
            graphs_e2e.append(g)
        N.nosa_set_stream(ctx, stream.cuda_stream)
        assert N.nosa_sync(ctx) == N.NOSA_OK
    # untimed: two replays of each graph (its first launch uploads it), on real steps of the sequence
    for j in range(n_e2e_warm):
        bs = sets[j % n_sets]
        fill(bs, j)
        if e2e_graph:
            graphs_e2e[j % n_sets].replay()
        else:
            host_step(bs)
    torch.cuda.synchronize()
    q_src, kv_src = q_src[n_e2e_warm:], kv_src[n_e2e_warm:]
    if fc:
        f_src = f_src[n_e2e_warm:]
    step_i[0] += n_e2e_warm
    done = [None] * n_sets
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    a.record(stream)
    busy = 0.0  # host time outside the waits: copies and graph launches
    for j in range(n_e2e):
        k = j % n_sets
        bs = sets[k]
        if done[k] is not None:
            done[k].synchronize()                   # that set's previous step has finished
        tb = time.perf_counter()
        if done[k] is not None:
            outs_host[j - n_sets].copy_(bs["out"])  # read its result back on the host
        fill(bs, j)
        if e2e_graph:
            graphs_e2e[k].replay()
        else:
            host_step(bs)
        done[k] = torch.cuda.Event()
        done[k].record(stream)
        busy += time.perf_counter() - tb
    b.record(stream)
    torch.cuda.synchronize()
    for j in range(max(0, n_e2e - n_sets), n_e2e):
        outs_host[j].copy_(sets[j % n_sets]["out"])
    wall = time.perf_counter() - t0
    step_i[0] += n_e2e
    dev_ms, wall_ms = a.elapsed_time(b) / n_e2e, wall * 1e3 / n_e2e
    e2e_ms = max(dev_ms, wall_ms)
    h2d_step = L * (B * Hq * d * 2 + 2 * U * d * 2) + ((L + 1) * U * d * 2 if fc else 0)
    how = ("nosa_step_host_all on pinned host q/k/v/out (one host-to-device copy of every layer's inputs, the "
           "layers' steps, one device-to-host copy of the outputs)" if not fc else
           "host-to-device copies of q, k, v and the forecast vectors from pinned memory, nosa_step_forecast for "
           "every layer, the device-to-host copy of the outputs")
    result["e2e"] = {"value": B / (e2e_ms * 1e-3), "unit": "tok/s", "ms_per_step": e2e_ms,
                     "device_ms_per_step": dev_ms, "host_wall_ms_per_step": wall_ms,
                     "host_busy_ms_per_step": busy * 1e3 / n_e2e, "steps": n_e2e,
                     "h2d_bytes_per_step": h2d_step, "d2h_bytes_per_step": L * B * Hq * d * 2,
                     "how": how + ", outputs then copied out of the pinned buffers on the host; " +
                            ("three CUDA graphs of those calls taking turns" if e2e_graph else "eager calls") +
                            "; max of device-event and host wall time"}
    assert N.nosa_sync(ctx) == N.NOSA_OK
    # the link's peak: a 1 GiB pinned copy, after the e2e leg (whose pinned buffers it would share)
    h2d = h2d_peak(torch)
    fach = fetch_bytes_launch / (us["gather"] * 1e-6) / 1e9
    fetch_step = fetched_per_step * BLOCK_BYTES
    fr = {"kernel": "gather_kernel", "bound": "host-to-device link", "achieved": fach, "peak": h2d, "unit": "GB/s",
          "frac": fach / h2d, "peak_source": "best pinned 1 GiB cudaMemcpyAsync H2D measured in this run",
          "bytes_per_launch": fetch_bytes_launch, "avg_launch_us": us["gather"],
          "in_step": {"achieved": fetch_step / (ms * 1e-3) / 1e9, "frac": fetch_step / (ms * 1e-3) / 1e9 / h2d,
                      "bytes_per_step": fetch_step,
                      "how": "blocks the timed steps fetched x 32 KiB / ms_per_step: the link's use over the whole "
                             "step (selections included)"}}
    if fc:
        fr["note"] = "the forecast path's gather (nosa_fetch after nosa_forecast_select), the kernel the timed step runs"
    else:
        attend_link = fetch_bytes_attend / (us["attend_fetch"] * 1e-6) / 1e9
        fr["note"] = ("standalone nosa_fetch on a fresh fetch list (blocks not read since they were evicted); in "
                      "the timed step the attention kernel copies the new blocks itself")
        fr["in_attend"] = {"achieved": attend_link, "frac": attend_link / h2d,
                           "bytes_per_launch": fetch_bytes_attend, "avg_launch_us": us["attend_fetch"],
                           "how": "new blocks' bytes / the attention launch that copies them (a lower bound on "
                                  "the link's rate during that launch, which also reads the cached blocks)"}
    result["fetch_roofline"] = fr
    N.nosa_destroy(ctx)
    del Qall, KVall
    torch.cuda.empty_cache()
    if world == 1:
        result["cpu_baseline"] = oracle_baseline(syn.workload(args.workload, **over), args.cpu_seconds, L * U)
    result["host_store_gb"] = sizes.host_store_bytes / 1e9
    return result


def run_dense(args, rank, world, local_rank):
    """Full-attention comparator (the pages' FullAttn rows): every layer's attention reads the whole
    context from a device-resident KV cache; no selection, no host memory.  Same workload shapes."""
    import torch
    from offloadable_block_sparse_gb300 import nosa as N
    from synth import inputs as syn
    torch.cuda.set_device(local_rank)
    dev = "cuda"
    over = {"sigma": args.sigma} if args.sigma is not None else {}
    wl = syn.workload(args.workload, **over)
    L = args.layers or wl.layers
    B, Hq, Hkv, d = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim
    U, G, T = B * Hkv, Hq // Hkv, wl.context
    nb = -(-T // 64)
    K, W = args.steps, args.warmup
    gen = torch.Generator(device=dev).manual_seed(1000 * rank + 17)
    kv = torch.empty((L, U, nb, 2, 64, d), dtype=torch.bfloat16, device=dev)
    for l in range(L):
        for u0 in range(0, U, 16):
            u1 = min(U, u0 + 16)
            kv[l, u0:u1] = torch.randn((u1 - u0, nb, 2, 64, d), generator=gen, device=dev).to(torch.bfloat16)
    qs = torch.randn((K + W + 1, L, U, G, d), generator=gen, device=dev)
    Qall = (qs / qs.norm(dim=-1, keepdim=True) * math.sqrt(d)).to(torch.bfloat16)
    del qs
    out = torch.empty((L, U, G, d), dtype=torch.bfloat16, device=dev)
    cur_q = torch.empty((L, U, G, d), dtype=torch.bfloat16, device=dev)
    nbytes = N.nosa_dense_scratch_bytes(U, T)
    scratch = torch.zeros(nbytes // 4 + 64, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    i16 = torch.int16

    def calls(q, st):
        for l in range(L):
            N.nosa_dense_attend(q[l].view(i16), kv[l].view(i16), U, G, nb, T, out[l].view(i16), scratch, nbytes,
                                stream=st)

    calls(Qall[0], stream.cuda_stream)  # first call sets the kernel attributes outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        calls(cur_q, side.cuda_stream)
    for t in range(W):
        cur_q.copy_(Qall[1 + t], non_blocking=True)
        graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(K):
        cur_q.copy_(Qall[1 + W + t], non_blocking=True)
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ck = clocks.stop()
    assert int(scratch[0].item()) == 0, "device-side error in the dense attention"
    ms = slowest_rank_ms(e0.elapsed_time(e1) / K, world, dev)
    # per-launch time of one layer's dense attention (kernel + merge), stream held while queueing
    per = []
    for _ in range(5):
        torch.cuda._sleep(400000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        N.nosa_dense_attend(Qall[0, 0].view(i16), kv[0].view(i16), U, G, nb, T, out[0].view(i16), scratch, nbytes,
                            stream=stream.cuda_stream)
        b.record(stream)
        torch.cuda.synchronize()
        per.append(a.elapsed_time(b) * 1e3)
    us = statistics.median(per)
    bytes_launch = U * T * 2 * d * 2 + 2 * U * G * d * 2
    hbm, src = measured_peaks()
    return {"metric": METRIC, "value": job_throughput(B, world, ms), "unit": "tok/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "layers": L, "batch_per_gpu": B, "q_heads": Hq, "kv_heads": Hkv,
                       "head_dim": d, "context": T, "selection": "dense (full-attention comparator, KV in HBM)",
                       "parallelism": f"replicas x{world}", "cuda_graph": True},
            "gpu_launches": 2 * L * K, "clocks": ck,
            "roofline": {"kernel": "dense_attend_kernel + merge", "bound": "hbm",
                         "achieved": bytes_launch / (us * 1e-6) / 1e9, "peak": hbm,
                         "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)", "unit": "GB/s",
                         "frac": bytes_launch / (us * 1e-6) / 1e9 / hbm, "traffic": None,
                         "algorithmic_bytes_per_launch": bytes_launch, "avg_launch_us": us},
            "kv_resident_gb": kv.numel() * 2 / 1e9}


def prompt_queries(B, Hq, n, d, sigma, gen, device):
    """bf16 [B][Hq][n][d] prompt queries, correlated along the positions as the decode steps'
    random walk q_t = normalize(q_{t-1} + sigma N(0, I)) sqrt(d) is (neighbours at cosine
    1 / sqrt(1 + sigma^2)): a stationary Gaussian sequence p_t = rho p_{t-1} + sqrt(1 - rho^2) e_t,
    rho = 1 / sqrt(1 + sigma^2), each p_t scaled to norm sqrt(d); stepped in closed form 256
    positions at a time (one matrix product per chunk, no launch per position)."""
    import torch
    rho = 1.0 / math.sqrt(1.0 + sigma ** 2)
    c = 256
    i_ = torch.arange(c, device=device, dtype=torch.float32)
    lag = i_[:, None] - i_[None, :]
    A = torch.where(lag >= 0, math.sqrt(1.0 - rho * rho) * torch.pow(rho, lag.clamp(min=0)), torch.zeros_like(lag))
    r = torch.pow(rho, i_ + 1)
    q = torch.empty((B, Hq, n, d), dtype=torch.bfloat16, device=device)
    pt = torch.randn((B * Hq * d,), generator=gen, device=device)
    for t0 in range(0, n, c):
        m = min(c, n - t0)
        E = torch.randn((m, B * Hq * d), generator=gen, device=device)
        P = A[:m, :m] @ E + r[:m, None] * pt[None, :]
        pt = P[m - 1].clone()
        Qc = P.view(m, B, Hq, d)
        Qc = Qc / Qc.norm(dim=-1, keepdim=True) * math.sqrt(d)
        q[:, :, t0:t0 + m] = Qc.permute(1, 2, 0, 3).to(torch.bfloat16)
    return q


def run_prefill(args, rank, world, local_rank):
    """NOSA_S sparse prefill: a prompt of the workload's context length through every layer (nosa_prefill),
    each timed repetition on a fresh context (a prefill starts from empty layers)."""
    import torch
    from offloadable_block_sparse_gb300 import nosa as N
    from synth import inputs as syn
    torch.cuda.set_device(local_rank)
    over = {"sigma": args.sigma} if args.sigma is not None else {}
    if args.batch:
        over["batch"] = args.batch
    wl = syn.workload(args.workload, **over)
    L = args.layers or wl.layers
    B, Hq, Hkv, d, n = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim, wl.context
    U = B * Hkv
    gen = torch.Generator(device="cuda").manual_seed(1000 * rank + 23)
    q = prompt_queries(B, Hq, n, d, wl.sigma, gen, "cuda")
    k = torch.randn((B, Hkv, n, d), generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, Hkv, n, d), generator=gen, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    cgen = torch.Generator().manual_seed(1000 * rank + 29)
    heads = [((torch.randn((Hkv, d, wl.evict_hidden), generator=cgen) / math.sqrt(d)).float().numpy(),
              (torch.randn((Hkv, wl.evict_hidden), generator=cgen) / math.sqrt(wl.evict_hidden)).float().numpy())
             for _ in range(L)]
    flags = N.NOSA_F_DMA_BIAS if args.dma_bias else 0
    cfg = N.make_config(num_layers=L, batch=B, num_q_heads=Hq, num_kv_heads=Hkv, k_q=wl.k_q, k_e=wl.k_e,
                        window_tokens=wl.window_tokens, max_context=n + 1, sink_blocks=wl.sink_blocks,
                        evict_hidden=wl.evict_hidden, flags=flags, **sizing_overrides(args))
    stream = torch.cuda.current_stream()
    times = []
    K, W = max(args.steps, 1), max(args.warmup, 1)
    scratch, nbytes = None, 0
    clocks = ClockSampler(local_rank)
    i16 = torch.int16
    for rep in range(W + K):
        ctx = N.nosa_create(cfg, stream.cuda_stream)
        for l in range(L):
            N.nosa_set_eviction_head(ctx, l, *heads[l])
        if scratch is None:
            nbytes = N.nosa_prefill_scratch_bytes(ctx, n)
            scratch = torch.empty(nbytes // 2 + 64, dtype=torch.int16, device="cuda")
        torch.cuda.synchronize()
        if rep == W:
            clocks.start()
            time.sleep(0.3)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for l in range(L):
            N.nosa_prefill(ctx, l, q.view(i16), k.view(i16), v.view(i16), n, out.view(i16), scratch, nbytes)
        b.record(stream)
        torch.cuda.synchronize()
        if N.nosa_sync(ctx) != N.NOSA_OK:
            raise RuntimeError("device error in the prefill")
        if rep >= W:
            times.append(a.elapsed_time(b))
        stats = N.nosa_get_stats(ctx)
        N.nosa_destroy(ctx)
    ck = clocks.stop()
    ms = slowest_rank_ms(statistics.mean(times), world, "cuda")
    return {"metric": "sparse prefill tok/s (NOSA_S, attn path, 1 GB300)", "value": job_throughput(B * n, world, ms),
            "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(wl, args, L, world), prompt_tokens=n,
                           selection="NOSA_S: every prompt position selected as the decode step would, in order",
                           prompt_queries=f"correlated along the positions as the decode walk with sigma {wl.sigma}"),
            "gpu_launches": 6 * L * K, "clocks": ck,
            "step": "one prompt of context tokens per sequence through every layer (nosa_prefill per layer)",
            "gamma": {"mean": stats.gamma_mean, "min": stats.gamma_min},
            "blocks_selected_fetched": stats.blocks_fetched}


def run_reference(args):
    """The oracle, as it stands, on host cores: each step is a bounded sample of the workload."""
    from synth import inputs as syn
    over = {}
    if args.sigma is not None:
        over["sigma"] = args.sigma
    if args.k_q is not None:
        over["k_q"], over["k_e"] = args.k_q, 64 - args.k_q
    wl = syn.workload(args.workload, **over)
    U = wl.layers * wl.batch * wl.kv_heads
    per_step = max(2.0, min(8.0, 150.0 / max(args.steps + args.warmup, 1)))
    base = oracle_baseline(wl, per_step * (args.steps + args.warmup), U)
    return {"impl": "reference", "metric": METRIC, "value": base["value"], "unit": "tok/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wl.batch / base["value"],
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, args, args.layers or wl.layers, 1),
            "cpu_baseline": base,
            "e2e": {"value": base["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.batch and not args.prefill:
        raise SystemExit("--batch applies to --prefill only")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    if args.dense:
        res = run_dense(args, rank, world, local_rank)
    elif args.prefill:
        res = run_prefill(args, rank, world, local_rank)
    else:
        res = run_native(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
