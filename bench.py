"""Benchmark of the SWA(w, s) hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of the long-prefill
workload with the widest window of the sweep (B=2, L=32768, Hq=32, Hkv=8,
d=128, SWA(w=512, s=4), bf16, q/k/v ~ N(0,1) with the four sink keys scaled
x4; the inputs, 1.34 GB, exceed the 126 MB L2):
    swa_prefill  ->  swa_cache_append (prompt survivors)
                 ->  swa_append_decode (append one new token, decode at pos = L)
Metric: in-band TFLOP/s = 4 * B * Hq * d * (sum over the step's query rows of
|K(t)|) / step time.

Besides the K timed steps, each measured kernel is timed over its own fixed
loop of at least one second of device time (CUDA graph replays on the
launching stream), so its per-launch figure does not depend on K:
  roofline     the prefill kernel of the step (tensor-bound at this window)
  llama_layer  the Llama-3.1-8B shaped layer prefill (B=1, L=4096, SWA(128,4);
               HBM-bound; rotating input sets larger than L2)
  decode       batch-64 decode, SWA(64,4), 68-slot ring cache (HBM-bound;
               rotating caches larger than 4x L2)
Under torchrun each rank runs an independent replica on its own GPU (no
data-path collective); the time is the max over ranks.

--impl reference times the fp64 CPU oracle (the reference arm of this build)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import swa_inputs  # noqa: E402

WORKLOAD = dict(name="long prefill SWA(512,4) B=2 L=32768 + append + decode", B=2, L=32768,
                Hq=32, Hkv=8, d=128, w=512, s=4, sink_rows=4, seed=1004)
LLAMA = dict(name="llama3.1-8b-layer prefill SWA(128,4)", B=1, L=4096, Hq=32, Hkv=8,
             d=128, w=128, s=4, sink_rows=4, seed=1002)
DECODE = dict(name="decode SWA(64,4) batch 64, 68-slot ring cache", B=64, Hq=32, Hkv=8, d=128,
              w=64, s=4, pos=262143)
L2_BYTES = 126 * 1024 * 1024
KERNEL_SOURCES = ("prefill.cuh", "swa_index.cuh", "sm100_ptx.cuh")
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "swa_prefill_b2_L32768_w512_s4.md")


PREFILL_KERNELS = {"auto": 0, "single": 1, "pair": 2}
# the step's prefill (SWA(512,4): the sink box rides in each block's last band tile)
KERNEL_NAMES = {"auto": "swa_prefill_kernel<128, true>", "single": "swa_prefill_kernel<128, true>",
                "pair": "swa_prefill_pair_kernel<128>"}


def step_config(args) -> dict:
    """The step workload, with the prompt length --L when given (a profiling
    aid: the default is the benchmark's L)."""
    cfg = dict(WORKLOAD)
    if getattr(args, "L", None):
        cfg["L"] = int(args.L)
        cfg["name"] = (f"long prefill SWA({cfg['w']},{cfg['s']}) B={cfg['B']} L={cfg['L']}"
                       " + append + decode")
    return cfg


def select_prefill_kernel(swa, args):
    swa.swa_prefill_select(PREFILL_KERNELS[getattr(args, "prefill_kernel", "auto")])


def pairs_per_head(L: int, w: int, s: int) -> int:
    """sum over t < L of |K(t)| = min(t+1, w) + min(s, max(0, t-w+1))."""
    t = np.arange(L, dtype=np.int64)
    return int(np.sum(np.minimum(t + 1, w) + np.minimum(s, np.maximum(0, t - w + 1))))


def keys_of_row(t: int, w: int, s: int) -> int:
    return min(t + 1, w) + min(s, max(0, t - w + 1))


def prefill_flops(cfg) -> float:
    return 4.0 * cfg["B"] * cfg["Hq"] * cfg["d"] * pairs_per_head(cfg["L"], cfg["w"], cfg["s"])


def step_flops(cfg) -> float:
    rows = pairs_per_head(cfg["L"], cfg["w"], cfg["s"]) + keys_of_row(cfg["L"], cfg["w"], cfg["s"])
    return 4.0 * cfg["B"] * cfg["Hq"] * cfg["d"] * rows


def prefill_bytes(cfg) -> int:
    """Algorithmic bytes of one prefill launch: Q, K, V read once, O written once."""
    return cfg["B"] * cfg["L"] * (2 * cfg["Hq"] + 2 * cfg["Hkv"]) * cfg["d"] * 2


def kernel_source_digest() -> str:
    """sha256 (first 16 hex digits) of the prefill kernel's source files."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sliding_window_attention_05_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the step's prefill kernel from the committed ncu
    summary, or None when the kernel's sources changed since that capture."""
    if not os.path.exists(TRAFFIC_PROFILE):
        return None, "no capture"
    with open(TRAFFIC_PROFILE) as f:
        text = f.read()
    m = re.search(r"traffic_record: dram_bytes_per_launch=(\d+) source_sha=([0-9a-f]+)", text)
    if not m:
        return None, "no traffic record"
    if m.group(2) != kernel_source_digest():
        return None, f"kernel changed since the capture (sources {kernel_source_digest()}, " \
                     f"capture {m.group(2)})"
    return int(m.group(1)), os.path.relpath(TRAFFIC_PROFILE, ROOT)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm_gbs=j["hbm_gbs"], bf16_tflops=j["bf16_tflops"],
                    bf16_tflops_sustained=j.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str | None = None):
        self.gpu_index = gpu_index
        self.path = path
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
            if self.path:
                with open(self.path, "w") as f:
                    f.write(self.FIELDS + "\n" + "\n".join(self.lines) + "\n")
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        loaded = [x for x in sm if x > 0.5 * (mx or max(sm))] or sm
        return {"sm_mhz": float(np.median(loaded)), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm

def make_step_inputs(cfg, n_sets, device, seed_offset=0):
    sets = []
    for i in range(n_sets):
        q, k, v = swa_inputs.prefill_inputs(cfg["B"], cfg["L"], cfg["Hq"], cfg["Hkv"], cfg["d"],
                                            cfg["seed"] + seed_offset + 97 * i,
                                            sink_rows=cfg["sink_rows"])
        g = torch.Generator("cpu").manual_seed(cfg["seed"] + 7 + 97 * i)
        qn = torch.randn(cfg["B"], cfg["Hq"], cfg["d"], generator=g).to(torch.bfloat16)
        kn = torch.randn(cfg["B"], 1, cfg["Hkv"], cfg["d"], generator=g).to(torch.bfloat16)
        vn = torch.randn(cfg["B"], 1, cfg["Hkv"], cfg["d"], generator=g).to(torch.bfloat16)
        sets.append(dict(q=q, k=k, v=v, qn=qn, kn=kn, vn=vn))
    return sets


class GpuStep:
    """Device-resident buffers of one input set and the hot-path calls."""

    def __init__(self, swa, cfg, host, device):
        self.swa, self.cfg = swa, cfg
        B, L, Hq, Hkv, d, w, s = (cfg[x] for x in ("B", "L", "Hq", "Hkv", "d", "w", "s"))
        self.dev = {k: t.to(device) for k, t in host.items()}
        self.out = torch.empty(B, L, Hq, d, dtype=torch.bfloat16, device=device)
        self.kc = torch.zeros(B, Hkv, s + w, d, dtype=torch.bfloat16, device=device)
        self.vc = torch.zeros_like(self.kc)
        self.pos0 = torch.zeros(B, dtype=torch.int32, device=device)
        self.posL = torch.full((B,), L, dtype=torch.int32, device=device)
        self.dec = torch.empty(B, Hq, d, dtype=torch.bfloat16, device=device)
        need = swa.swa_decode_workspace_size(B, Hq, Hkv, d, w, s)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device) if need else None
        self.graph_prefill = None
        self.graph_rest = None

    def prefill(self):
        c = self.cfg
        self.swa.swa_prefill(self.dev["q"], self.dev["k"], self.dev["v"], c["w"], c["s"],
                             out=self.out)

    def rest(self):
        c = self.cfg
        self.swa.swa_cache_append(self.dev["k"], self.dev["v"], self.kc, self.vc, self.pos0,
                                  c["w"], c["s"])
        self.swa.swa_append_decode(self.dev["qn"], self.dev["kn"][:, 0], self.dev["vn"][:, 0],
                                   self.kc, self.vc, self.posL, c["w"], c["s"], out=self.dec,
                                   workspace=self.ws)

    def capture(self, stream):
        self.graph_prefill = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_prefill, stream=stream):
            self.prefill()
        self.graph_rest = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_rest, stream=stream):
            self.rest()


def launches_per_step(swa, cfg) -> int:
    """prefill + append(prompt) + append_decode (+ the split-KV combine)."""
    splits_ws = swa.swa_decode_workspace_size(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["w"],
                                              cfg["s"])
    return 1 + 1 + (2 if splits_ws else 1)


def replay_for(graph, stream, min_seconds: float, launches_per_replay: int):
    """Replay `graph` on `stream` for at least min_seconds of device time (the
    replay count is fixed from a short calibration first); returns
    (ms per launch, replays)."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
        e0.record(stream)
        for _ in range(5):
            graph.replay()
        e1.record(stream)
        e1.synchronize()
        per = e0.elapsed_time(e1) / 5
        n = max(5, int(math.ceil(min_seconds * 1e3 / max(per, 1e-3))))
        e0.record(stream)
        for _ in range(n):
            graph.replay()
        e1.record(stream)
        e1.synchronize()
    return e0.elapsed_time(e1) / (n * launches_per_replay), n


def bench_decode(swa, device, stream, min_seconds=1.0, pos=None):
    """Kernel-only decode at batch 64 over a rotating pool of distinct caches
    (> 4x L2), captured as one CUDA graph of `ncache` decode launches and
    replayed for at least min_seconds."""
    c = dict(DECODE)
    if pos is not None:
        c["pos"] = pos
    B, Hq, Hkv, d, w, s = (c[x] for x in ("B", "Hq", "Hkv", "d", "w", "s"))
    kv_bytes = B * Hkv * (s + w) * d * 2 * 2
    ncache = max(8, int(math.ceil(4 * L2_BYTES / kv_bytes)))
    g = torch.Generator(device=device).manual_seed(1003)
    caches = [(torch.randn(B, Hkv, s + w, d, generator=g, device=device).to(torch.bfloat16),
               torch.randn(B, Hkv, s + w, d, generator=g, device=device).to(torch.bfloat16))
              for _ in range(ncache)]
    q = torch.randn(B, Hq, d, generator=g, device=device).to(torch.bfloat16)
    pos = torch.full((B,), c["pos"], dtype=torch.int32, device=device)
    out = torch.empty_like(q)
    with torch.cuda.stream(stream):
        for kc, vc in caches[:2]:
            swa.swa_decode(q, kc, vc, pos, w, s, out=out)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for kc, vc in caches:
                swa.swa_decode(q, kc, vc, pos, w, s, out=out)
    ms_per_launch, reps = replay_for(graph, stream, min_seconds, ncache)
    kv_bytes = B * Hkv * min(c["pos"] + 1, s + w) * d * 2 * 2  # slots actually read
    gbs = kv_bytes / (ms_per_launch * 1e-3) / 1e9
    return dict(kv_bytes_per_launch=kv_bytes, us_per_launch=ms_per_launch * 1e3, gbs=gbs,
                caches=ncache, pool_bytes=ncache * kv_bytes, launches=reps * ncache)


def bench_llama_layer(swa, device, stream, peaks, min_seconds=1.0):
    """The Llama-3.1-8B shaped layer prefill (B=1, L=4096, SWA(128, 4)) over
    rotating input sets larger than L2: one CUDA graph that runs the prefill
    once on each set, replayed for at least min_seconds."""
    cfg = LLAMA
    n_sets = max(2, int(math.ceil(2.5 * L2_BYTES / prefill_bytes(cfg))))
    sets = make_step_inputs(cfg, n_sets, device)
    steps = [GpuStep(swa, cfg, h, device) for h in sets]
    with torch.cuda.stream(stream):
        for st in steps:
            st.prefill()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for st in steps:
                st.prefill()
    ms, reps = replay_for(graph, stream, min_seconds, n_sets)
    by = prefill_bytes(cfg)
    gbs = by / (ms * 1e-3) / 1e9
    return {"workload": cfg["name"], "B": cfg["B"], "L": cfg["L"], "w": cfg["w"], "s": cfg["s"],
            "kernel": "swa_prefill_kernel<128, false>", "bound": "hbm",
            "us_per_launch": round(ms * 1e3, 2), "achieved": round(gbs, 1), "unit": "GB/s",
            "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4),
            "algorithmic_bytes": by,
            "tflops": round(prefill_flops(cfg) / (ms * 1e-3) / 1e12, 2),
            "launches": reps * n_sets,
            "l2": f"rotating {n_sets} input sets of {by / 1e6:.1f} MB (> 126 MB L2)"}


def run_gpu(args):
    import sliding_window_attention_05_b300 as swa

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.Stream(device)
    cfg = step_config(args)
    select_prefill_kernel(swa, args)
    peaks = load_peaks()
    default_run = cfg["L"] == WORKLOAD["L"] and args.prefill_kernel != "pair"

    # one input set: 1.34 GB of q, k, v (at the default L), far larger than the 126 MB L2
    host = make_step_inputs(cfg, 1, device, seed_offset=1000 * rank)[0]
    st = GpuStep(swa, cfg, host, device)
    with torch.cuda.stream(stream):
        st.prefill()               # eager warm-up (first-call setup happens here)
        st.rest()
        stream.synchronize()
        st.capture(stream)
        for _ in range(args.warmup):
            st.graph_prefill.replay()
            st.graph_rest.replay()
        stream.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(local, args.clocks_csv) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(K):
                ev[i][0].record(stream)
                st.graph_prefill.replay()
                ev[i][1].record(stream)
                st.graph_rest.replay()
            end.record(stream)
        torch.cuda.synchronize(device)
    barrier(world)
    total_ms = start.elapsed_time(end)
    prefill_ms_steps = sum(a.elapsed_time(b) for a, b in ev) / K
    total_ms = max_over_ranks(total_ms, world, device)
    ms_per_step = total_ms / K
    value = step_flops(cfg) * world / (ms_per_step * 1e-3) / 1e12

    # the same step through the public API with host buffers (every rank)
    e2e = None if args.skip_e2e else run_e2e(swa, cfg, host, device, stream,
                                             max(3, min(K, 10)), world)
    result = None
    if rank == 0:
        # the prefill kernel alone, over a fixed loop of >= min_seconds
        with ClockSampler(local) as clk_loop:
            pre_ms, pre_reps = replay_for(st.graph_prefill, stream, args.loop_seconds, 1)
        tf = prefill_flops(cfg) / (pre_ms * 1e-3) / 1e12
        traffic, traffic_src = recorded_traffic() if default_run else (
            None, "the recorded capture is of the default L and kernel")
        roofline = dict(
            bound="tensor", achieved=round(tf, 1), peak=peaks["bf16_tflops"], unit="TFLOP/s",
            frac=round(tf / peaks["bf16_tflops"], 4), traffic=traffic,
            kernel=KERNEL_NAMES[args.prefill_kernel], us_per_launch=round(pre_ms * 1e3, 2),
            launches_timed=pre_reps, peak_source=peaks["source"] + " (burst)",
            peak_sustained=peaks["bf16_tflops_sustained"],
            frac_sustained=(round(tf / peaks["bf16_tflops_sustained"], 4)
                            if peaks["bf16_tflops_sustained"] else None),
            inband_flop_per_launch=prefill_flops(cfg),
            algorithmic_bytes=prefill_bytes(cfg),
            hbm_gbs=round(prefill_bytes(cfg) / (pre_ms * 1e-3) / 1e9, 1),
            traffic_source=traffic_src, kernel_sources_sha=kernel_source_digest(),
            us_per_launch_in_steps=round(prefill_ms_steps * 1e3, 2),
            clocks=clk_loop.summary())
        llama = None if args.skip_llama else bench_llama_layer(swa, device, stream, peaks,
                                                               args.loop_seconds)
        dec = None if args.skip_decode else bench_decode(swa, device, stream, args.loop_seconds)
        result = {
            "metric": "SWA(w,s) prefill in-band TFLOP/s & decode KV GB/s, % of B300 roofline",
            "value": round(value, 3),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) q/k/v, sink keys x4)",
            "config": {"workload": cfg["name"], "B": cfg["B"], "L": cfg["L"], "Hq": cfg["Hq"],
                       "Hkv": cfg["Hkv"], "d": cfg["d"], "w": cfg["w"], "s": cfg["s"],
                       "global_batch": cfg["B"] * world, "seq_len": cfg["L"],
                       "parallelism": f"replicas x{world}",
                       "step": "prefill + append(prompt) + append_decode(pos=L)",
                       "prefill_kernel": args.prefill_kernel,
                       "l2": f"inputs larger than L2 ({prefill_bytes(cfg) / 1e9:.2f} GB of "
                             f"q, k, v, out per step); CUDA graph per step half"},
            "roofline": roofline,
            "llama_layer": llama,
            "decode": None if dec is None else dict(
                workload=DECODE["name"], value=round(dec["gbs"], 1), unit="GB/s",
                bound="hbm", peak=peaks["hbm_gbs"], frac=round(dec["gbs"] / peaks["hbm_gbs"], 4),
                us_per_launch=round(dec["us_per_launch"], 3),
                kv_bytes_per_launch=dec["kv_bytes_per_launch"], launches_timed=dec["launches"],
                l2=f"{dec['caches']} distinct caches, {dec['pool_bytes'] / 1e6:.0f} MB"),
            "e2e": e2e,
            "gpu_launches": launches_per_step(swa, cfg) * K,
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(cfg, host, budget_s=args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


# ------------------------------------------------------------------ other workloads
# Supplementary measurements of the other configurations (one JSON line each);
# the default workload above is the benchmark's step.

def _time_events(fn, stream, iters, warmup=3):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        e1.synchronize()
    return e0.elapsed_time(e1) / iters


def bench_window_sweep(swa, device, stream, peaks, iters=10):
    """Long prefill window sweep: B=2, L=32768, Hq=32, Hkv=8, d=128, s=4,
    w in {64, 256, 512}; inputs (1.3 GB) far exceed L2."""
    B, L, Hq, Hkv, d, s = 2, 32768, 32, 8, 128, 4
    q, k, v = (t.to(device) for t in swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, 1004,
                                                                 sink_rows=4))
    out = torch.empty_like(q)
    lines = []
    for w in (64, 256, 512):
        ms = _time_events(lambda: swa.swa_prefill(q, k, v, w, s, out=out), stream, iters)
        fl = 4.0 * B * Hq * d * pairs_per_head(L, w, s)
        by = B * L * (2 * Hq + 2 * Hkv) * d * 2
        tf = fl / (ms * 1e-3) / 1e12
        gbs = by / (ms * 1e-3) / 1e9
        lines.append({"workload": f"prefill SWA({w},{s}) B={B} L={L} Hq={Hq} Hkv={Hkv} d={d}",
                      "us_per_launch": round(ms * 1e3, 2), "tflops": round(tf, 1),
                      "tensor_frac": round(tf / peaks["bf16_tflops"], 4),
                      "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                      "inband_flop": fl, "algorithmic_bytes": by, "iters": iters})
    return lines


def bench_hybrid(swa, device, stream, peaks, n_layers=8, L=16384, steps=256):
    """The hybrid stack: 8 layers alternating SWA(2048, 100) and full causal,
    B=1, L=16384, Hq=32, Hkv=8, d=128: prefill of every layer, then `steps`
    decode steps through all layers (one step captured as a CUDA graph)."""
    B, Hq, Hkv, d = 1, 32, 8, 128
    windows = swa.hybrid_layer_windows(n_layers, L, steps)
    g = torch.Generator(device=device).manual_seed(1005)
    qkv = [tuple(torch.randn(B, L, h, d, generator=g, device=device).to(torch.bfloat16)
                 for h in (Hq, Hkv, Hkv)) for _ in range(n_layers)]
    toks = [tuple(torch.randn(B, h, d, generator=g, device=device).to(torch.bfloat16)
                  for h in (Hq, Hkv, Hkv)) for _ in range(n_layers)]
    outs = [torch.empty(B, L, Hq, d, dtype=torch.bfloat16, device=device) for _ in range(n_layers)]

    def prefill_all():
        for (q, k, v), (w, s), o in zip(qkv, windows, outs):
            swa.swa_prefill(q, k, v, w, s, out=o)

    pre_ms = _time_events(prefill_all, stream, iters=3)
    fl = sum(4.0 * B * Hq * d * pairs_per_head(L, w, s) for w, s in windows)
    with torch.cuda.stream(stream):
        stack = swa.HybridStack(B, Hq, Hkv, d, windows, device=device)
        stack.prefill(qkv)
        dec_out = stack.step(toks)            # first step: allocates workspaces
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            stack.step(toks, outs=dec_out)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps - 1):
            graph.replay()
        e1.record(stream)
        e1.synchronize()
    step_ms = e0.elapsed_time(e1) / (steps - 1)
    # KV bytes one step reads: every slot each layer holds at the last position
    kv = sum(B * Hkv * min(L + steps, s + w) * d * 2 * 2 for w, s in windows)
    return [{"workload": f"hybrid stack {n_layers} layers (SWA(2048,100) / full causal) B={B} "
                         f"L={L} Hq={Hq} Hkv={Hkv} d={d}",
             "prefill_ms_all_layers": round(pre_ms, 3),
             "prefill_tflops": round(fl / (pre_ms * 1e-3) / 1e12, 1),
             "prefill_tensor_frac": round(fl / (pre_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
             "decode_us_per_step_all_layers": round(step_ms * 1e3, 2),
             "decode_tokens_per_s": round(1e3 / step_ms, 1),
             "decode_kv_gbs": round(kv / (step_ms * 1e-3) / 1e9, 1),
             "decode_steps": steps}]


def bench_decode_positions(swa, device, stream, peaks):
    """Batch-64 decode at positions 128, 1K, 16K and 256K: the 68-slot cache
    is full at each, so the bytes read (and the time) stay flat."""
    lines = []
    for pos in (128, 1024, 16384, 262143):
        dec = bench_decode(swa, device, stream, pos=pos)
        lines.append({"workload": f"{DECODE['name']}, pos={pos}",
                      "us_per_launch": round(dec["us_per_launch"], 3),
                      "kv_gbs": round(dec["gbs"], 1), "hbm_frac": round(dec["gbs"] / peaks["hbm_gbs"], 4),
                      "kv_bytes_per_launch": dec["kv_bytes_per_launch"],
                      "l2": f"{dec['caches']} distinct caches, {dec['pool_bytes'] / 1e6:.0f} MB"})
    return lines


def bench_chunked(swa, device, stream, peaks, iters=5):
    """Chunked prefill into the ring cache: the SWA(2048, 100) layer of the
    hybrid stack (B=1, L=16384, Hq=32, Hkv=8, d=128) prefilled in chunks of
    4096 and 1024, against the same prompt in one call."""
    B, L, Hq, Hkv, d, w, s = 1, 16384, 32, 8, 128, 2048, 100
    g = torch.Generator(device=device).manual_seed(1006)
    q, k, v = (torch.randn(B, L, h, d, generator=g, device=device).to(torch.bfloat16)
               for h in (Hq, Hkv, Hkv))
    fl = 4.0 * B * Hq * d * pairs_per_head(L, w, s)
    out = torch.empty_like(q)
    lines = []
    one = _time_events(lambda: swa.swa_prefill(q, k, v, w, s, out=out), stream, iters)
    lines.append({"workload": f"prefill SWA({w},{s}) B={B} L={L} Hq={Hq} Hkv={Hkv} d={d}, one call",
                  "ms": round(one, 4), "tflops": round(fl / (one * 1e-3) / 1e12, 1),
                  "tensor_frac": round(fl / (one * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)})
    for T in (4096, 1024):
        with torch.cuda.stream(stream):
            cache = swa.RingCache(B, Hkv, d, w, s, device=device)
            chunks = [(q[:, p:p + T].contiguous(), k[:, p:p + T].contiguous(),
                       v[:, p:p + T].contiguous(), out[:, p:p + T].contiguous())
                      for p in range(0, L, T)]

        def run():
            cache.next_pos.zero_()
            cache.length = 0
            for qc, kc, vc, oc in chunks:
                cache.prefill_chunk(qc, kc, vc, out=oc)

        ms = _time_events(run, stream, iters)
        lines.append({"workload": f"chunked prefill SWA({w},{s}) B={B} L={L} in chunks of {T}",
                      "ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                      "tensor_frac": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                      "vs_one_call": round(one / ms, 3)})
    # the same prompt into the paged layout (pages of 64 positions); the
    # host-side page reservation and table copy of every chunk are timed too
    T, P = 1024, 64
    with torch.cuda.stream(stream):
        pool = swa.PagePool(B * (L // P + 2), Hkv, d, page_size=P, device=device)
        pcache = swa.PagedKVCache(pool, B, w, s, max_len=L)
        chunks = [(q[:, p:p + T].contiguous(), k[:, p:p + T].contiguous(),
                   v[:, p:p + T].contiguous(), out[:, p:p + T].contiguous())
                  for p in range(0, L, T)]

    def run_paged():
        pcache.release()
        for qc, kc, vc, oc in chunks:
            pcache.prefill_chunk(qc, kc, vc, out=oc, stream=stream)

    ms = _time_events(run_paged, stream, iters)
    lines.append({"workload": f"paged chunked prefill SWA({w},{s}) B={B} L={L} in chunks of {T},"
                              f" pages of {P}",
                  "ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                  "tensor_frac": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                  "vs_one_call": round(one / ms, 3)})
    return lines


def bench_paged_decode(swa, device, stream, peaks, iters=64, page_size=64):
    """Batch-64 decode, SWA(64, 4), through the paged layout (pages of 64
    positions: the sink page and the two window pages at position 262143),
    over a rotating set of caches drawn from one pool (> 4x L2)."""
    c = DECODE
    B, Hq, Hkv, d, w, s, pos = (c[x] for x in ("B", "Hq", "Hkv", "d", "w", "s", "pos"))
    kv_bytes = B * Hkv * (s + w) * d * 2 * 2
    ncache = max(8, int(math.ceil(4 * L2_BYTES / kv_bytes)))
    pages_per_seq = 3
    pool = swa.PagePool(ncache * B * pages_per_seq, Hkv, d, page_size=page_size, device=device)
    g = torch.Generator(device=device).manual_seed(1007)
    pool.k.copy_(torch.randn(pool.k.shape, generator=g, device=device).to(torch.bfloat16))
    pool.v.copy_(torch.randn(pool.v.shape, generator=g, device=device).to(torch.bfloat16))
    caches = []
    for _ in range(ncache):
        pc = swa.PagedKVCache(pool, B, w, s, max_len=pos + 1)
        pc._reserve(pos)
        pc.length = pos + 1
        caches.append(pc)
    q = torch.randn(B, Hq, d, generator=g, device=device).to(torch.bfloat16)
    out = torch.empty_like(q)
    with torch.cuda.stream(stream):
        for pc in caches:            # sets every cache's position outside the graph
            pc.decode(q, out=out)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for pc in caches:
                pc.decode(q, out=out)
        for _ in range(8):
            graph.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            graph.replay()
        e1.record(stream)
        e1.synchronize()
    us = e0.elapsed_time(e1) / (iters * ncache) * 1e3
    gbs = kv_bytes / (us * 1e-6) / 1e9
    ring = bench_decode(swa, device, stream)
    return [{"workload": f"paged decode SWA({w},{s}) batch {B}, pages of {page_size}, pos={pos}",
             "us_per_launch": round(us, 3), "kv_gbs": round(gbs, 1),
             "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "kv_bytes_per_launch": kv_bytes,
             "ring_us_per_launch": round(ring["us_per_launch"], 3),
             "l2": f"{ncache} caches in one pool of {pool.n_pages} pages"}]


def bench_backward(swa, device, stream, peaks, iters=5):
    """Backward of the prefill (dq, dk, dv from dout) on the Llama-shaped layer
    (B=1, L=4096, SWA(128, 4)) and the long-window case (B=2, L=32768,
    SWA(512, 4)). In-band FLOPs of the backward: 10 d per admitted (row, key)
    pair and query head (S, dP, dV, dK and dQ products; the kernels recompute
    S and dP once more, which is not counted)."""
    lines = []
    for (B, L, w, s, seed) in ((1, 4096, 128, 4, 1002), (2, 32768, 512, 4, 1004)):
        Hq, Hkv, d = 32, 8, 128
        q, k, v = (t.to(device) for t in swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, seed,
                                                                    sink_rows=4))
        g = torch.Generator(device=device).manual_seed(seed + 1)
        dout = torch.randn(B, L, Hq, d, generator=g, device=device).to(torch.bfloat16)
        lse = torch.empty(B, Hq, L, dtype=torch.float32, device=device)
        out = torch.empty_like(q)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(swa.swa_prefill_backward_workspace_size(B, L, Hq, Hkv, d, s),
                         dtype=torch.uint8, device=device)
        fwd_ms = _time_events(lambda: swa.swa_prefill(q, k, v, w, s, out=out, lse=lse), stream,
                              iters)
        bwd_ms = _time_events(lambda: swa.swa_prefill_backward(q, k, v, out, dout, lse, w, s,
                                                               dq=dq, dk=dk, dv=dv, workspace=ws),
                              stream, iters)
        pairs = pairs_per_head(L, w, s)
        fl = 10.0 * B * Hq * d * pairs
        lines.append({"workload": f"prefill backward SWA({w},{s}) B={B} L={L} Hq={Hq} Hkv={Hkv} "
                                  f"d={d}",
                      "forward_with_lse_us": round(fwd_ms * 1e3, 1),
                      "backward_us": round(bwd_ms * 1e3, 1),
                      "backward_tflops": round(fl / (bwd_ms * 1e-3) / 1e12, 1),
                      "backward_tensor_frac": round(fl / (bwd_ms * 1e-3) / 1e12 /
                                                    peaks["bf16_tflops"], 4),
                      "inband_flop": fl, "iters": iters})
    return lines


def run_other(args):
    import sliding_window_attention_05_b300 as swa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()
    select_prefill_kernel(swa, args)
    fn = {"window-sweep": bench_window_sweep, "hybrid": bench_hybrid,
          "decode-positions": bench_decode_positions, "chunked": bench_chunked,
          "paged-decode": bench_paged_decode, "backward": bench_backward}[args.workload]
    for line in fn(swa, device, stream, peaks):
        line["peak_source"] = peaks["source"]
        print(json.dumps(line), flush=True)


def run_e2e(swa, cfg, host, device, stream, K, world):
    """The same step through the public API with host buffers: every step copies
    the inputs from pinned host memory and reads the outputs back."""
    pinned = {k: t.pin_memory() for k, t in host.items()}
    out_h = torch.empty(cfg["B"], cfg["L"], cfg["Hq"], cfg["d"], dtype=torch.bfloat16).pin_memory()
    dec_h = torch.empty(cfg["B"], cfg["Hq"], cfg["d"], dtype=torch.bfloat16).pin_memory()
    st = GpuStep(swa, cfg, host, device)
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = out_h.numel() * 2 + dec_h.numel() * 2

    def one():
        for k, t in pinned.items():
            st.dev[k].copy_(t, non_blocking=True)
        st.prefill()
        st.rest()
        out_h.copy_(st.out, non_blocking=True)
        dec_h.copy_(st.dec, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            one()
        stream.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        barrier(world)
        a.record(stream)
        for _ in range(K):
            one()
        b.record(stream)
        b.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / K, world, device)
    return {"value": round(step_flops(cfg) * world / (ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": K}


# ------------------------------------------------------------------ CPU oracle arm

def _oracle_rows_timed(oracle, cfg, host, rows, nthreads):
    sc = 1.0 / math.sqrt(cfg["d"])
    t0 = time.perf_counter()
    oracle.prefill(host["q"], host["k"], host["v"], cfg["w"], cfg["s"], sc, rows=rows,
                   nthreads=nthreads)
    dt = time.perf_counter() - t0
    fl = 4.0 * cfg["B"] * cfg["Hq"] * cfg["d"] * sum(keys_of_row(int(t), cfg["w"], cfg["s"])
                                                     for t in rows)
    return dt, fl


def cpu_baseline(cfg, host, budget_s: float = 15.0):
    """The fp64 oracle as it stands, on this host's cores (all threads, OpenMP
    over rows): evenly spaced query rows of the step's prefill (every head and
    batch), as many as fit in about budget_s seconds, after a short calibration;
    plus a one-thread figure over a tenth of the budget. In-band TFLOP/s."""
    import oracle
    cores = os.cpu_count() or 1
    L = cfg["L"]
    probe = np.linspace(0, L - 1, 64).astype(np.int64)
    dt, _ = _oracle_rows_timed(oracle, cfg, host, probe, cores)
    n = int(min(L, max(64, 64 * budget_s / max(dt, 1e-3))))
    rows = np.unique(np.linspace(0, L - 1, n).astype(np.int64))
    dt, fl = _oracle_rows_timed(oracle, cfg, host, rows, cores)
    n1 = int(min(L, max(8, len(rows) * (budget_s / 10) / max(dt * cores, 1e-3))))
    rows1 = np.unique(np.linspace(0, L - 1, n1).astype(np.int64))
    dt1, fl1 = _oracle_rows_timed(oracle, cfg, host, rows1, 1)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{len(rows)} evenly spaced query rows of {L} x {cfg['Hq']} heads x "
                      f"{cfg['B']} sequences of the prefill (fp64, OpenMP over rows)",
            "single_thread": {"value": round(fl1 / dt1 / 1e12, 6), "unit": "TFLOP/s",
                              "sample": f"{len(rows1)} evenly spaced query rows x "
                                        f"{cfg['Hq']} heads x {cfg['B']} sequences",
                              "seconds": round(dt1, 2)}}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    cfg = step_config(args)
    host = make_step_inputs(cfg, 1, None)[0]
    import oracle
    cores = os.cpu_count() or 1
    L = cfg["L"]
    rows_per_step = max(8, int(args.ref_rows))
    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        r = np.sort(rng.choice(L, size=min(L, 8), replace=False)).astype(np.int64)
        _oracle_rows_timed(oracle, cfg, host, r, cores)
    total_t, total_flops = 0.0, 0.0
    for _ in range(args.steps):
        r = np.sort(rng.choice(L, size=min(L, rows_per_step), replace=False)).astype(np.int64)
        dt, fl = _oracle_rows_timed(oracle, cfg, host, r, cores)
        total_t += dt
        total_flops += fl
    value = total_flops / total_t / 1e12
    sample = (f"{rows_per_step} random query rows x {cfg['Hq']} heads x {cfg['B']} sequences "
              f"per step (fp64 oracle)")
    return {
        "impl": "reference",
        "metric": "SWA(w,s) prefill in-band TFLOP/s & decode KV GB/s, % of B300 roofline",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * total_t / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/k/v, sink keys x4)",
        "config": {"workload": cfg["name"], "B": cfg["B"], "L": cfg["L"], "Hq": cfg["Hq"],
                   "Hkv": cfg["Hkv"], "d": cfg["d"], "w": cfg["w"], "s": cfg["s"],
                   "global_batch": cfg["B"] * world, "seq_len": cfg["L"],
                   "parallelism": f"replicas x{world}",
                   "step": "prefill rows of the step (sampled)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--loop-seconds", type=float, default=1.0,
                    help="device time of each kernel's own timing loop")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--clocks-csv", default=None,
                    help="also write the raw nvidia-smi clock samples of the timed region here")
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--prefill-kernel", choices=tuple(PREFILL_KERNELS), default="auto",
                    help="prefill kernel: the library's choice (auto), one query block per "
                    "work item (single) or two (pair)")
    ap.add_argument("--L", type=int, default=None,
                    help="prompt length of the step workload (default 32768; shorter prompts "
                    "are for profiling small cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-decode", action="store_true", help="omit the batch-64 decode measurement")
    ap.add_argument("--skip-llama", action="store_true", help="omit the Llama-shaped layer loop")
    ap.add_argument("--skip-e2e", action="store_true", help="omit the host-buffer measurement")
    ap.add_argument("--workload", choices=("step", "window-sweep", "hybrid", "decode-positions",
                                           "chunked", "paged-decode", "backward"),
                    default="step", help="step (default): the benchmark line; the others print "
                    "supplementary lines for the other configurations (1 GPU)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload != "step" and args.impl == "ours":
        run_other(args)
        return
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
