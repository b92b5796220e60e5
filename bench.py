"""Benchmark of the K-quant x Q8_K path on GB300.

Headline workload: the Qwen3-4B-shaped decode layer at M = 1 (hidden 2560;
Q4_K Wq 2560->4096, Wk/Wv 2560->1024, Wo 4096->2560, gate/up 2560->9728;
Q6_K down 9728->2560).  One step = one pass of the hot path over one layer:
Q8_K quantization of the layer's four GEMV inputs, then the seven GEMVs.
Steps rotate over L distinct copies of the layer's weights (8 by default,
505 MB, about 4x the 126 MB L2) so that every step streams its weights from
HBM, as consecutive layers of a model do.  `value` = weight bytes streamed
per second (GB/s), timed on the device with CUDA events around regions of
exactly K steps replayed from CUDA graphs, repeated until the regions cover
at least 100 ms; the median region gives the value.

Also reported: the same metric end to end (activations copied in from pinned
host memory and outputs copied back every step), the roofline of the GEMV
kernels, the M = 512 GEMM throughput (TOPS, 2*M*N*K ops) on the 27B-shaped
FFN and the Qwen3-4B prefill layers and the MoE grouped GEMM, and the CPU
oracle's throughput on the same workload.

`--impl reference` times the CPU oracle instead (the only reference this
method has), with the same metric, on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_gemv_gemm_gb300 import synth  # noqa: E402

METRIC = "kq GEMV weight GB/s at M=1 and GEMM int8 TOPS at M=512, % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    p = dict(FALLBACK_PEAKS)
    p["source"] = "fallback"
    return p


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------
# DRAM traffic recorded by ncu, valid only while the kernel sources are the
# ones it was captured on (profiles/<name>.traffic.txt: "sources_sha256 = ",
# "dram_bytes_per_step = ").

KERNEL_SOURCES = ["quantized_gemv_gemm_gb300/csrc/kq_gemv.cu", "quantized_gemv_gemm_gb300/csrc/kq_device.cuh"]


def kernel_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(name):
    path = os.path.join(ROOT, "profiles", f"{name}.traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
    if kv.get("sources_sha256") != kernel_sources_sha256():
        return None
    try:
        return float(kv["dram_bytes_per_step"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------
# clocks sampled during the timed region

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------
# the decode-layer workload on the GPU

LAYER_INPUTS = [("x_attn", 2560), ("x_o", 4096), ("x_ffn", 2560), ("x_down", 9728)]
# rotations of the layer copies captured in one CUDA graph (4 x 8 = 32 layer
# steps, about one decode pass of a 36-layer model)
GRAPH_ROTATIONS = 4
# largest graph of headline steps (a region of K steps replays it K // G
# times, then a graph of the remainder)
GRAPH_MAX_STEPS = 256
DEFAULT_LAYER_COPIES = 8


def headline_config(world: int, layer_copies: int = DEFAULT_LAYER_COPIES):
    """The headline workload, shared by both arms' JSON lines."""
    mats = synth.configs()[1].matrices
    wb = sum(m.weight_bytes for m in mats)
    return {"workload": "Qwen3-4B-shaped decode layer, M=1 (Q4_K q/k/v/o/gate/up, Q6_K down)",
            "M": 1, "hidden": 2560,
            "matrices": [f"{m.name} {synth.FORMAT_NAMES[m.fmt]} {m.N}x{m.K}" for m in mats],
            "weight_bytes_per_step": wb, "layer_copies": layer_copies,
            "l2": f"inputs larger than L2: step i reads layer copy i % {layer_copies}, "
                  f"{wb * layer_copies / 1e6:.1f} MB of weights in all",
            "parallelism": f"replicas x{world}"}
# matrix -> index of its input
LAYER_USES = {"wq": 0, "wk": 0, "wv": 0, "wo": 1, "gate": 2, "up": 2, "down": 3}


class DecodeLayers:
    """L copies of the Qwen3-4B-shaped layer, packed on the device."""

    def __init__(self, kq, torch, n_copies: int, seed_cfg: int = 1):
        cfg = synth.configs()[1]
        self.kq, self.torch = kq, torch
        self.mats = cfg.matrices
        self.copies = []
        for l in range(n_copies):
            packed = []
            for i, m in enumerate(self.mats):
                disk = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(seed_cfg, 1000 * l + i))
                dd = torch.from_numpy(disk.reshape(-1)).cuda()
                packed.append(kq.kq_repack(m.fmt, dd, m.N, m.K))
                del dd
            xs = [torch.from_numpy(synth.activations(1, k, synth.rng_for(seed_cfg, 1000 * l + 100 + j))).cuda()
                  for j, (_, k) in enumerate(LAYER_INPUTS)]
            self.copies.append({"packed": packed, "x": xs})
        torch.cuda.synchronize()
        self.q8 = [kq.q8k_empty(1, k) for _, k in LAYER_INPUTS]
        self.y_total = sum(m.N for m in self.mats)
        self.y = torch.empty(self.y_total, dtype=torch.float32, device="cuda")
        offs = np.cumsum([0] + [m.N for m in self.mats])
        self.y_views = [self.y[offs[i]:offs[i + 1]] for i in range(len(self.mats))]
        self.weight_bytes = sum(m.weight_bytes for m in self.mats)
        self.x_total = sum(k for _, k in LAYER_INPUTS)

    # fused path: one launch per group of matrices sharing an input
    GROUPS = [["wq", "wk", "wv"], ["wo"], ["gate", "up"], ["down"]]

    def step(self, l, events=None, x_override=None, fused=True, y_override=None):
        """One layer: fused -> 4 launches of kq_gemv_fused (q/k/v, o, gate/up,
        down); separate -> 4 kq_quantize_q8k + 7 kq_gemv launches."""
        kq = self.kq
        c = self.copies[l]
        xs = c["x"] if x_override is None else x_override
        yv = self.y_views if y_override is None else y_override
        idx = {m.name: i for i, m in enumerate(self.mats)}
        for j, names in enumerate(self.GROUPS):
            ii = [idx[n] for n in names]
            m0 = self.mats[ii[0]]
            if fused:
                if events is not None:
                    events[j][0].record()
                kq.kq_gemv_fused(m0.fmt, [c["packed"][i] for i in ii], [self.mats[i].N for i in ii], m0.K,
                                 xs[j], [yv[i] for i in ii])
                if events is not None:
                    events[j][1].record()
            else:
                kq.kq_quantize_q8k(xs[j], out=self.q8[j])
                for i in ii:
                    kq.kq_gemv(self.mats[i].fmt, c["packed"][i], self.mats[i].N, self.mats[i].K, self.q8[j],
                               y=yv[i])

    def launches_per_step(self, fused=True):
        return len(self.GROUPS) if fused else len(LAYER_INPUTS) + len(self.mats)

    def algorithmic_launch_bytes(self):
        """Per fused launch: packed weight bytes of its matrices + the fp32
        input row (4 B per element, read once) + 4 B per output."""
        idx = {m.name: i for i, m in enumerate(self.mats)}
        out = []
        for j, names in enumerate(self.GROUPS):
            ms = [self.mats[idx[n]] for n in names]
            out.append(sum(m.weight_bytes + 4 * m.N for m in ms) + 4 * ms[0].K)
        return out


def max_over_ranks(torch, v: float, world: int, device="cuda") -> float:
    """The largest of the ranks' values (a region's time: the whole job ends
    with its slowest rank); the value itself with one rank."""
    if world == 1:
        return v
    tt = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput of N replicas: every rank's units over the
    slowest rank's time (units per second)."""
    return units_per_rank * world / (ms_max * 1e-3)


# timed regions: each holds exactly the work asked for (K steps for the
# headline); a region is repeated until the regions together cover at least
# MIN_TIMED_MS, and the median region is reported
MIN_TIMED_MS = 100.0
MIN_REGIONS = 5
MAX_REGIONS = 5000
SPIN_CYCLES = 100_000   # ~50 us spin before each start event


def time_regions(torch, run, barrier=None, min_ms=MIN_TIMED_MS, min_regions=MIN_REGIONS):
    """ms of each of R regions of `run()` (R >= min_regions, together >=
    min_ms).  Per region: barrier, synchronize, a short spin kernel (so the
    start event is recorded while the GPU is still busy and the submission of
    the region's work is not inside it), events around run(), synchronize,
    barrier.  Returns the list of region times."""
    times = []
    while True:
        if barrier is not None:
            barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(SPIN_CYCLES)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        if barrier is not None:
            barrier()
        times.append(a.elapsed_time(b))
        if len(times) >= MAX_REGIONS or (len(times) >= min_regions and sum(times) >= min_ms):
            return times


def region_summary(times):
    return {"regions": len(times), "median_ms": round(float(statistics.median(times)), 5),
            "min_ms": round(float(min(times)), 5), "max_ms": round(float(max(times)), 5),
            "total_ms": round(float(sum(times)), 3)}


def graph_of(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the path outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def run_ours(args, world, rank, local):
    import torch
    torch.cuda.set_device(local)
    from quantized_gemv_gemm_gb300 import build as kq_build
    if rank == 0 or world == 1:
        kq_build.build()
    if world > 1:
        torch.distributed.barrier()
        kq_build.build()
    from quantized_gemv_gemm_gb300 import kq

    peaks = load_peaks()
    if not args.no_pdl:
        kq.kq_set_launch_flags(kq.KQ_LAUNCH_PDL)
    L = args.layers
    layers = DecodeLayers(kq, torch, L)
    NG = len(layers.GROUPS)
    # a timed region holds exactly K = args.steps layer steps (step i reads
    # layer copy i % L), replayed from CUDA graphs of at most GRAPH_MAX_STEPS
    # steps plus one graph of the remainder
    K = args.steps
    G = min(K, GRAPH_MAX_STEPS)
    n_full, rem = divmod(K, G)

    def region_graphs(step_fn):
        gs = [graph_of(torch, lambda: [step_fn(l % L) for l in range(G)])]
        if rem:
            gs.append(graph_of(torch, lambda: [step_fn((n_full * G + l) % L) for l in range(rem)]))
        return gs

    def replay_region(gs):
        for _ in range(n_full):
            gs[0].replay()
        if rem:
            gs[1].replay()

    g_plain = region_graphs(lambda l: layers.step(l))
    g_sep = region_graphs(lambda l: layers.step(l, fused=False))

    # events around every launch of every step of one rotation
    def timing_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:  # torch without graph event-record nodes
            return None

    ev = [[[timing_event(), timing_event()] for _ in range(NG)] for _ in range(L)]
    graph_events = ev[0][0][0] is not None
    if graph_events:
        g_timed = graph_of(torch, lambda: [layers.step(l, events=ev[l]) for l in range(L)])
    else:
        ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
               for _ in range(NG)] for _ in range(L)]

    # W untimed warm-up steps (after the graphs' own set-up passes)
    for l in range(args.warmup):
        layers.step(l % L)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    with ClockSampler(local) as clk:
        regions = time_regions(torch, lambda: replay_region(g_plain), barrier)
        regions_sep = time_regions(torch, lambda: replay_region(g_sep), barrier, min_ms=MIN_TIMED_MS / 2)
        ms = float(statistics.median(regions))
        ms_sep = float(statistics.median(regions_sep))
        # kernel-timing pass: event nodes around each launch; the times of the
        # last rotation are read after each of a few replays
        kt = {j: [] for j in range(NG)}
        for _ in range(10):
            if graph_events:
                g_timed.replay()
            else:
                for l in range(L):
                    layers.step(l, events=ev[l])
            torch.cuda.synchronize()
            for l in range(L):
                for j in range(NG):
                    kt[j].append(ev[l][j][0].elapsed_time(ev[l][j][1]))
    clocks = clk.summary()

    ms_max = max_over_ranks(torch, ms, world)
    ms_sep = max_over_ranks(torch, ms_sep, world)
    steps = K
    bytes_per_step = layers.weight_bytes
    value = job_rate(bytes_per_step * steps, world, ms_max) / 1e9
    value_sep = job_rate(bytes_per_step * steps, world, ms_sep) / 1e9

    # roofline of the GEMV kernel: the timed region holds nothing but its
    # launches (4 per step), so its average launch duration is the region's
    # time / launches and achieved = algorithmic bytes of a step / step time
    alg = layers.algorithmic_launch_bytes()
    achieved = job_rate(sum(alg) * steps, world, ms_max) / 1e9
    hbm = float(peaks["hbm_gbs"])
    mean_ms = [float(np.mean(kt[j])) for j in range(NG)]
    per_launch = [{"matrices": "+".join(names), "event_us": round(t * 1e3, 3), "bytes": b}
                  for names, t, b in zip(layers.GROUPS, mean_ms, alg)]
    traffic = recorded_traffic("gemv_decode_layer")

    # end to end through the public API: every step copies its four input
    # rows in from pinned host memory (kq_copy_in: a kernel of the launch
    # chain that reads the host rows before its dependency wait) and the four
    # GEMV launches store all seven outputs straight into pinned host memory.
    # Two rotating input/output buffers, so a step's host outputs are never
    # overwritten while an earlier step may still be writing them; replayed
    # from a graph.  (Copy-engine copies on side streams with event waits
    # measured 2.31 TB/s: each cross-stream wait breaks the early launch.)
    x_host = torch.from_numpy(np.concatenate(
        [synth.activations(1, k, synth.rng_for(1, 7000 + j))[0] for j, (_, k) in enumerate(LAYER_INPUTS)])).pin_memory()
    NBUF = 2
    y_host = [torch.empty(layers.y_total, dtype=torch.float32).pin_memory() for _ in range(NBUF)]
    x_dev = [torch.empty(layers.x_total, dtype=torch.float32, device="cuda") for _ in range(NBUF)]
    xo = np.cumsum([0] + [k for _, k in LAYER_INPUTS])
    yo = np.cumsum([0] + [m.N for m in layers.mats])
    x_views = [[xd[xo[j]:xo[j + 1]].view(1, -1) for j in range(len(LAYER_INPUTS))] for xd in x_dev]
    y_views = [[yh[yo[i]:yo[i + 1]] for i in range(len(layers.mats))] for yh in y_host]

    def e2e_step(i):
        b = i % NBUF
        kq.kq_copy_in(x_host, x_dev[b])
        layers.step(i % L, x_override=x_views[b], y_override=y_views[b])

    g_e2e = region_graphs(e2e_step)
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e_regions = time_regions(torch, lambda: replay_region(g_e2e), barrier, min_ms=MIN_TIMED_MS / 2)
    e_ms = max_over_ranks(torch, float(statistics.median(e_regions)), world)
    e2e_value = job_rate(bytes_per_step * steps, world, e_ms) / 1e9
    y_check = np.concatenate([yh.numpy() for yh in y_host])
    assert np.isfinite(y_check).all()

    small_batch = bench_small_batch(kq, torch, layers, peaks, args)
    gemv_27b = bench_gemv_27b(kq, torch, peaks, args)
    q8_0_line = bench_q8_0(kq, torch, peaks, args)
    moe_decode = bench_moe_decode(kq, torch, peaks, args)
    gemm = None if args.no_gemm else bench_gemm(kq, torch, peaks, args)

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_max / steps, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic (seeded random K-quant superblocks and N(0,1) activations)",
            "config": headline_config(world, L),
            "timing": {"how": f"each timed region is exactly K = {steps} layer steps, replayed from CUDA graphs "
                              f"(of at most {GRAPH_MAX_STEPS} steps) with programmatic dependent launch "
                              f"{'on' if not args.no_pdl else 'off'}; CUDA events on the launching stream, a "
                              f"short spin kernel before each start event; regions repeated until they cover "
                              f">= {MIN_TIMED_MS:.0f} ms; value and ms_per_step from the median region",
                       **region_summary(regions)},
            "roofline": {"bound": "hbm", "kernel": "kq gemv_kernel (fused quantize + GEMV, 4 launches per step)",
                         "timing": "the headline's median region of K steps (only gemv_kernel launches in it)",
                         "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4),
                         "peak_source": f"{peaks['source']} hbm_gbs (STREAM-style copy)",
                         "alg_bytes_per_step": sum(alg),
                         "traffic": traffic,
                         "traffic_unit": "DRAM bytes per step (4 launches), ncu, profiles/gemv_decode_layer.traffic.txt",
                         "per_launch_diag": {"how": "event nodes between launches in a graph replay (they break "
                                                    "the launch overlap, so these durations read long)",
                                             "launches": per_launch}},
            "separate_path": {"value": round(value_sep, 2), "unit": "GB/s",
                              "how": "4 kq_quantize_q8k + 7 kq_gemv launches per step"},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": 4 * layers.x_total, "d2h_bytes_per_step": 4 * layers.y_total,
                    "how": "graph replay of, every step: kq_copy_in of the 4 fp32 input rows from pinned host "
                           "memory (a kernel in the launch chain, reading the host rows before its dependency "
                           "wait), 4 kq_gemv_fused launches storing all 7 outputs straight into pinned host "
                           f"memory; {NBUF} rotating input/output buffers; regions of exactly K steps as for "
                           f"the headline, median of {len(e_regions)}"},
            "gpu_launches": layers.launches_per_step() * steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "small_batch": small_batch,
            "gemv_27b": gemv_27b,
            "q8_0_gemv": q8_0_line,
            "moe_decode": moe_decode,
            "gemm": gemm,
        }
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# small batches on the decode layer (secondary line)

def bench_small_batch(kq, torch, layers, peaks, args):
    """The Qwen3-4B-shaped decode layer for a batch of M = 2, 4, 8 tokens:
    per step, four kq_gemv_fused_batch launches (q/k/v, o, gate/up, down),
    each quantizing its [M, K] input inside the kernel and reading every
    weight item once for all M tokens, over the same rotating layer copies,
    replayed from CUDA graphs of 32 steps."""
    out = []
    idx = {m.name: i for i, m in enumerate(layers.mats)}
    hbm = float(peaks["hbm_gbs"])
    for M in (2, 4, 8):
        xs = [torch.from_numpy(synth.activations(M, k, synth.rng_for(1, 9000 + 10 * M + j))).cuda()
              for j, (_, k) in enumerate(LAYER_INPUTS)]
        ys = [torch.empty((M, m.N), dtype=torch.float32, device="cuda") for m in layers.mats]

        def step(l):
            c = layers.copies[l]
            for j, names in enumerate(layers.GROUPS):
                ii = [idx[nm] for nm in names]
                m0 = layers.mats[ii[0]]
                kq.kq_gemv_fused_batch(m0.fmt, [c["packed"][i] for i in ii], [layers.mats[i].N for i in ii],
                                       m0.K, xs[j], [ys[i] for i in ii])

        L = len(layers.copies)
        G = GRAPH_ROTATIONS * L
        g = graph_of(torch, lambda: [step(l % L) for l in range(G)])
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        us = statistics.median(time_regions(torch, g.replay, min_ms=50)) * 1e3 / G
        gbs = layers.weight_bytes / (us * 1e-6) / 1e9
        out.append({"M": M, "us_per_step": round(us, 3), "weight_gbs": round(gbs, 1),
                    "frac_of_hbm": round(gbs / hbm, 4), "tokens_per_s": round(M / (us * 1e-6), 1),
                    "launches_per_step": 4})
        del g
    return {"workload": "Qwen3-4B-shaped decode layer, batch of M tokens (4 kq_gemv_fused_batch launches per step)",
            "lines": out}


# --------------------------------------------------------------------------
# 27B-shaped FFN at M = 1 (secondary GEMV line)

def bench_moe_decode(kq, torch, peaks, args):
    """MoE decode on the 30B-A3B shapes: one token routed to 8 of 128 experts.
    Per step two kq_gemv_grouped_fused launches: gate and up (Q4_K 768x2048 per
    expert) over the token's 8 routed fp32 rows, quantized in the kernel, then
    down (Q6_K 2048x768) over the 8 down inputs.  Each of the 32 steps of a
    graph routes to 8 fresh experts (uniform, distinct), so the 392 MB of
    experts stream from HBM; value = expert bytes read per second."""
    cfg = synth.configs()[4]
    E, topk = cfg.experts, cfg.topk
    mats = cfg.matrices
    packed, per = [], []
    for i, m in enumerate(mats):
        b = kq.kq_repack_bytes(m.fmt, m.N, m.K)
        buf = torch.empty(b * E, dtype=torch.uint8, device="cuda")
        for e in range(E):
            disk = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(4, 10 + 1000 * i + e))
            kq.kq_repack(m.fmt, torch.from_numpy(disk.reshape(-1)).cuda(), m.N, m.K, packed=buf[e * b:(e + 1) * b])
        packed.append(buf)
        per.append(b)
    S = 32
    rng = synth.rng_for(4, 7000)
    offs = []
    for _ in range(S):
        chosen = np.sort(rng.choice(E, topk, replace=False))
        cnt = np.zeros(E, np.int64)
        cnt[chosen] = 1
        offs.append(torch.from_numpy(np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)).cuda())
    x = torch.from_numpy(np.repeat(synth.activations(1, mats[0].K, synth.rng_for(4, 7001)), topk, axis=0)).cuda()
    h = torch.from_numpy(synth.activations(topk, mats[2].K, synth.rng_for(4, 7002))).cuda()
    ys = [torch.empty((topk, m.N), dtype=torch.float32, device="cuda") for m in mats]

    def steps():
        for r in range(S):
            kq.kq_gemv_grouped_fused(mats[0].fmt, packed[:2], [mats[0].N, mats[1].N], mats[0].K, E, offs[r], x,
                                     ys[:2])
            kq.kq_gemv_grouped_fused(mats[2].fmt, packed[2:], [mats[2].N], mats[2].K, E, offs[r], h, ys[2:])

    g = graph_of(torch, steps)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    times = time_regions(torch, g.replay, min_ms=50)
    us = statistics.median(times) * 1e3 / S
    step_bytes = topk * sum(per)
    gbs = step_bytes / (us * 1e-6) / 1e9
    hbm = float(peaks["hbm_gbs"])
    del packed, g
    torch.cuda.empty_cache()
    return {"workload": "30B-A3B-shaped MoE decode: 1 token, top-8 of 128 experts, gate/up Q4_K 768x2048 + "
                        "down Q6_K 2048x768 (2 kq_gemv_grouped_fused launches per step)",
            "us_per_step": round(us, 3), "value": round(gbs, 1), "unit": "GB/s", "frac_of_hbm": round(gbs / hbm, 4),
            "expert_bytes_per_step": step_bytes,
            "timing": f"median of {len(times)} timed graph replays of {S} steps, each step routed to 8 fresh experts "
                      f"(experts {E * sum(per) / 1e6:.0f} MB)"}


def bench_q8_0(kq, torch, peaks, args):
    """The Q8_0 rail on the 27B-shaped FFN at M = 1: per step gate, up
    (17408x5120) and down (5120x17408) by kq_gemv_q8_0_fused (the row quantized
    inside each GEMV), over rotating copies of the 284 MB of Q8_0 weights,
    replayed from a CUDA graph with programmatic dependent launch.  The same
    step with the quantize as its own launch (2 kq_quantize_q8_0 + 3
    kq_gemv_q8_0) is timed beside it."""
    shapes = [(17408, 5120), (17408, 5120), (5120, 17408)]
    step_bytes = sum(N * K * 34 // 32 for N, K in shapes)
    C = max(2, -(-600_000_000 // step_bytes))
    base = []
    for i, (N, K) in enumerate(shapes):
        disk = torch.from_numpy(synth.disk_weights_q8_0(N, K, synth.rng_for(3, 50 + i)).reshape(-1)).cuda()
        base.append(kq.kq_repack(synth.Q8_0, disk, N, K))
        del disk
    copies = [base] + [[b.clone() for b in base] for _ in range(C - 1)]
    x = torch.from_numpy(synth.activations(1, 5120, synth.rng_for(3, 150), outliers=True)[0]).cuda()
    h = torch.from_numpy(synth.activations(1, 17408, synth.rng_for(3, 151))[0]).cuda()
    dx, qx = kq.kq_quantize_q8_0(x)
    dh, qh = kq.kq_quantize_q8_0(h)
    ys = [torch.empty(N, dtype=torch.float32, device="cuda") for N, _ in shapes]

    def rot_fused():
        for c in copies:
            kq.kq_gemv_q8_0_fused(c[0], 17408, 5120, x, y=ys[0])
            kq.kq_gemv_q8_0_fused(c[1], 17408, 5120, x, y=ys[1])
            kq.kq_gemv_q8_0_fused(c[2], 5120, 17408, h, y=ys[2])

    def rot_split():
        for c in copies:
            kq.kq_quantize_q8_0(x, d=dx, qs=qx)
            kq.kq_gemv_q8_0(c[0], 17408, 5120, dx, qx, y=ys[0])
            kq.kq_gemv_q8_0(c[1], 17408, 5120, dx, qx, y=ys[1])
            kq.kq_quantize_q8_0(h, d=dh, qs=qh)
            kq.kq_gemv_q8_0(c[2], 5120, 17408, dh, qh, y=ys[2])

    def timed(rot):
        g = graph_of(torch, rot)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        times = time_regions(torch, g.replay, min_ms=50)
        del g
        return statistics.median(times) * 1e3 / C

    us = timed(rot_fused)
    us_split = timed(rot_split)
    gbs = step_bytes / (us * 1e-6) / 1e9
    hbm = float(peaks["hbm_gbs"])
    del copies, base
    torch.cuda.empty_cache()
    return {"workload": "27B-shaped dense FFN in Q8_0 at M=1 (gate/up 17408x5120, down 5120x17408), "
                        "3 kq_gemv_q8_0_fused launches",
            "us_per_step": round(us, 3), "value": round(gbs, 1), "unit": "GB/s", "frac_of_hbm": round(gbs / hbm, 4),
            "split_quantize_us_per_step": round(us_split, 3),
            "weight_bytes_per_step": step_bytes, "copies": C,
            "timing": f"median of >= {MIN_REGIONS} timed graph replays of {C} steps covering >= 50 ms "
                      f"(weights {C * step_bytes / 1e6:.0f} MB)"}


def bench_gemv_27b(kq, torch, peaks, args):
    """The 27B-shaped dense FFN decoded at M = 1: gate+up in one fused launch
    (x of 5120), down in another (x of 17408), over rotating copies of the
    150 MB of weights (larger than L2), replayed from a CUDA graph."""
    cfg = synth.configs()[3]
    mats = cfg.matrices
    step_bytes = sum(m.weight_bytes for m in mats)
    C = max(2, -(-600_000_000 // step_bytes))
    base = []
    for i, m in enumerate(mats):
        disk = torch.from_numpy(synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(3, 2 * i)).reshape(-1)).cuda()
        base.append(kq.kq_repack(m.fmt, disk, m.N, m.K))
        del disk
    copies = [base] + [[b.clone() for b in base] for _ in range(C - 1)]
    xs = [torch.from_numpy(synth.activations(1, m.K, synth.rng_for(3, 100 + i), outliers=True)[0]).cuda()
          for i, m in enumerate(mats)]
    ys = [torch.empty(m.N, dtype=torch.float32, device="cuda") for m in mats]
    gate, up, down = mats

    def rot():
        for c in copies:
            kq.kq_gemv_fused(gate.fmt, c[:2], [gate.N, up.N], gate.K, xs[0], ys[:2])
            kq.kq_gemv_fused(down.fmt, c[2:], [down.N], down.K, xs[2], ys[2:])

    g = graph_of(torch, rot)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    times = time_regions(torch, g.replay, min_ms=50)
    us = statistics.median(times) * 1e3 / C
    gbs = step_bytes / (us * 1e-6) / 1e9
    hbm = float(peaks["hbm_gbs"])
    del copies, base, g
    torch.cuda.empty_cache()
    return {"workload": "27B-shaped dense FFN at M=1 (Q4_K gate/up 17408x5120, down 5120x17408), 2 launches",
            "us_per_step": round(us, 3), "value": round(gbs, 1), "unit": "GB/s", "frac_of_hbm": round(gbs / hbm, 4),
            "weight_bytes_per_step": step_bytes, "copies": C,
            "timing": f"median of {len(times)} timed graph replays of {C} steps "
                      f"(weights {C * step_bytes / 1e6:.0f} MB)"}


# --------------------------------------------------------------------------
# M = 512 GEMMs (secondary metric)

def int8_mma_sync_peak(kq, torch):
    """int8 rate of the warp-level MMA (mma.sync m16n8k32 s8, the only integer
    tensor-core MMA on sm_103a): kq_measure_mma_s8 over 4 blocks of 8 warps
    per SM, best of 5 launches of ~10 ms; TOPS counting multiply and add."""
    try:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        blocks, iters = 4 * sms, 2000
        out = kq.kq_measure_mma_s8(blocks, 10)
        torch.cuda.synchronize()
        best = None
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            kq.kq_measure_mma_s8(blocks, iters, out=out)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        if not bool((out == 1024 * iters).all()):
            raise RuntimeError("mma.sync rate kernel checksum mismatch")
        return blocks * 8 * iters * 8 * 8192 / (best * 1e-3) / 1e12
    except Exception as ex:
        print(f"mma.sync int8 rate unavailable: {ex}", file=sys.stderr)
        return None


def int8_tensor_peak(torch):
    """Dense int8 GEMM throughput of the vendor library on this GPU
    (torch._int_mm -> cuBLASLt), best of 10 on 8192^3."""
    try:
        n = 8192
        a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda")
        b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda")
        for _ in range(3):
            torch._int_mm(a, b)
        torch.cuda.synchronize()
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._int_mm(a, b)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception as ex:  # no int8 GEMM on this torch / device
        print(f"int8 peak unavailable: {ex}", file=sys.stderr)
        return None


def bench_gemm(kq, torch, peaks, args):
    out = []
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    i8_lib = int8_tensor_peak(torch)
    i8_mma = int8_mma_sync_peak(kq, torch)
    have = [v for v in (i8_lib, i8_mma) if v is not None]
    i8_peak = max(have) if have else None
    out.append({"int8_tensor_peak_tops": None if i8_peak is None else round(i8_peak, 1),
                "int8_mma_sync_tops": None if i8_mma is None else round(i8_mma, 1),
                "int8_cublaslt_tops": None if i8_lib is None else round(i8_lib, 1),
                "how": "measured, the larger of: kq_measure_mma_s8 (mma.sync m16n8k32 s8, 4 blocks x 8 warps per SM, "
                       "8 independent MMAs per warp, best of 5) and torch._int_mm (cuBLASLt int8 GEMM) 8192^3, best of 10",
                "fp16_tensor_peak_tflops": tc_peak, "fp16_how": "MEASURED_PEAKS.json bf16_tflops (cuBLAS, burst)"})

    def time_it(fn, reps):
        """ms per call of fn(r): calls r = 0..reps-1 captured in one CUDA graph
        (with the launch flags the headline uses), replayed in timed regions
        covering >= 100 ms; the median replay."""
        fn(0)
        torch.cuda.synchronize()
        g = graph_of(torch, lambda: [fn(r) for r in range(reps)])
        g.replay()
        torch.cuda.synchronize()
        times = time_regions(torch, g.replay, min_ms=100)
        del g
        return float(statistics.median(times)) / reps

    def dense(name, cfg_index, mats, outliers):
        M = 512
        wbytes = sum(m.weight_bytes for m in mats)
        copies = max(1, -(-260_000_000 // wbytes))  # weights of the rotation > 2x L2
        items = []
        for i, m in enumerate(mats):
            disk = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(cfg_index, 2 * i))
            packed0 = kq.kq_repack(m.fmt, torch.from_numpy(disk.reshape(-1)).cuda(), m.N, m.K)
            packed = [packed0] + [packed0.clone() for _ in range(copies - 1)]
            x = torch.from_numpy(synth.activations(M, m.K, synth.rng_for(cfg_index, 2 * i + 1), outliers)).cuda()
            a = kq.q8k_empty(M, m.K)
            y = torch.empty((M, m.N), dtype=torch.float32, device="cuda")
            ws_n = kq.kq_gemm_workspace_bytes(m.fmt, M, m.N, m.K)
            ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda") if ws_n else None
            items.append((m, packed, x, a, y, ws))
        torch.cuda.synchronize()

        def step(r):
            for m, packed, x, a, y, ws in items:
                kq.kq_quantize_q8k(x, out=a)
                kq.kq_gemm(m.fmt, packed[r % copies], m.N, m.K, a, y=y, workspace=ws)

        ms = time_it(step, args.gemm_reps)
        ops = sum(2 * M * m.N * m.K for m in mats)
        tops = ops / (ms * 1e-3) / 1e12
        out.append({"workload": name, "M": M, "ms": round(ms, 4), "tops": round(tops, 2),
                    "timing": f"median of timed graph replays of {args.gemm_reps} steps (>= 100 ms in all), "
                              f"{copies} rotating weight copies",
                    "frac_of_fp16_tensor_peak": round(tops / tc_peak, 4),
                    "frac_of_int8_tensor_peak": None if i8_peak is None else round(tops / i8_peak, 4),
                    "weight_gbs": round(sum(m.weight_bytes for m in mats) / (ms * 1e-3) / 1e9, 1)})
        del items
        torch.cuda.empty_cache()

    cfgs = synth.configs()
    dense("27B-shaped dense FFN Q4_K, M=512", 3, cfgs[3].matrices, True)
    dense("Qwen3-4B prefill pp512 all-Q5_K", 2, cfgs[2].matrices[:7], False)
    dense("Qwen3-4B prefill pp512 all-Q6_K", 2, cfgs[2].matrices[7:], False)

    # Q8_0 rail at M = 512: the 27B-shaped FFN in Q8_0 (gate, up, down), each
    # step quantizing its activations (kq_quantize_q8_0) and running the GEMM
    M = 512
    shapes = [(17408, 5120), (17408, 5120), (5120, 17408)]
    wbytes = sum(N * Kd * 34 // 32 for N, Kd in shapes)
    copies = max(1, -(-260_000_000 // wbytes))
    items = []
    for i, (N, Kd) in enumerate(shapes):
        disk = torch.from_numpy(synth.disk_weights_q8_0(N, Kd, synth.rng_for(3, 60 + i)).reshape(-1)).cuda()
        p0 = kq.kq_repack(synth.Q8_0, disk, N, Kd)
        del disk
        packed = [p0] + [p0.clone() for _ in range(copies - 1)]
        x = torch.from_numpy(synth.activations(M, Kd, synth.rng_for(3, 160 + i), outliers=True)).cuda()
        dq = torch.empty((M, Kd // 32), dtype=torch.float32, device="cuda")
        qq = torch.empty((M, Kd), dtype=torch.int8, device="cuda")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        items.append((N, Kd, packed, x, dq, qq, y))
    torch.cuda.synchronize()

    def q8_step(r):
        for N, Kd, packed, x, dq, qq, y in items:
            kq.kq_quantize_q8_0(x, d=dq, qs=qq)
            kq.kq_gemm_q8_0(packed[r % copies], N, Kd, dq, qq, y=y)

    ms = time_it(q8_step, args.gemm_reps)
    ops = sum(2 * M * N * Kd for N, Kd in shapes)
    tops = ops / (ms * 1e-3) / 1e12
    out.append({"workload": "27B-shaped dense FFN in Q8_0, M=512 (kq_quantize_q8_0 + kq_gemm_q8_0 per matrix)",
                "M": M, "ms": round(ms, 4), "tops": round(tops, 2),
                "timing": f"median of timed graph replays of {args.gemm_reps} steps (>= 100 ms in all), "
                          f"{copies} rotating weight copies",
                "frac_of_fp16_tensor_peak": round(tops / tc_peak, 4),
                "frac_of_int8_tensor_peak": None if i8_peak is None else round(tops / i8_peak, 4),
                "weight_gbs": round(wbytes / (ms * 1e-3) / 1e9, 1)})
    del items
    torch.cuda.empty_cache()

    # MoE grouped
    cfg = cfgs[4]
    T, E = cfg.M, cfg.experts
    row_token, _, offsets = synth.moe_routing(T, E, cfg.topk, synth.rng_for(4, 0))
    off_d = torch.from_numpy(offsets).cuda()
    x_tok = synth.activations(T, 2048, synth.rng_for(4, 1))
    items = []
    for i, m in enumerate(cfg.matrices):
        per = kq.kq_repack_bytes(m.fmt, m.N, m.K)
        packed = torch.empty(per * E, dtype=torch.uint8, device="cuda")
        for e in range(E):
            disk = synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(4, 10 + 1000 * i + e))
            kq.kq_repack(m.fmt, torch.from_numpy(disk.reshape(-1)).cuda(), m.N, m.K, packed=packed[e * per:(e + 1) * per])
        x = x_tok[row_token] if m.name != "down" else synth.activations(len(row_token), m.K, synth.rng_for(4, 2))
        xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        a = kq.q8k_empty(len(row_token), m.K)
        y = torch.empty((len(row_token), m.N), dtype=torch.float32, device="cuda")
        ws_n = kq.kq_gemm_workspace_bytes(m.fmt, len(row_token), m.N, m.K)
        ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda") if ws_n else None
        items.append((m, packed, xd, a, y, ws))
    torch.cuda.synchronize()

    def moe_step(r):
        for m, packed, x, a, y, ws in items:
            kq.kq_quantize_q8k(x, out=a)
            kq.kq_gemm_grouped(m.fmt, packed, E, off_d, m.N, m.K, a, y=y, workspace=ws)

    ms = time_it(moe_step, args.gemm_reps)
    rows = len(row_token)
    ops = sum(2 * rows * m.N * m.K for m in cfg.matrices)
    wbytes = sum(m.weight_bytes for m in cfg.matrices) * E
    out.append({"workload": "30B-A3B-shaped MoE grouped GEMM (128 experts, top-8, 512 tokens)", "rows": rows,
                "ms": round(ms, 4), "tops": round(ops / (ms * 1e-3) / 1e12, 2),
                "weight_gbs": round(wbytes / (ms * 1e-3) / 1e9, 1),
                "frac_of_hbm": round(wbytes / (ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]), 4)})
    del items
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)

REF_MIN_SECONDS = 10.0
REF_MAX_SECONDS = 60.0


class OracleLayers:
    """The headline workload for the CPU oracle: the same seeded layer copies
    (weights and input rows) as the GPU arm's DecodeLayers, in disk form."""

    def __init__(self, n_copies: int = DEFAULT_LAYER_COPIES, seed_cfg: int = 1):
        self.mats = synth.configs()[1].matrices
        self.copies = []
        for l in range(n_copies):
            disks = [synth.disk_weights(m.fmt, m.N, m.K, synth.rng_for(seed_cfg, 1000 * l + i))
                     for i, m in enumerate(self.mats)]
            xs = [synth.activations(1, k, synth.rng_for(seed_cfg, 1000 * l + 100 + j))
                  for j, (_, k) in enumerate(LAYER_INPUTS)]
            self.copies.append((disks, xs))
        self.weight_bytes = sum(m.weight_bytes for m in self.mats)

    def step(self, i: int):
        """One layer step with the oracle: quantize the four inputs, then the
        seven products (every output)."""
        import oracle
        disks, xs = self.copies[i % len(self.copies)]
        q = [oracle.quantize_q8k(x) for x in xs]
        for m, disk in zip(self.mats, disks):
            oracle.gemm(m.fmt, disk, *q[LAYER_USES[m.name]])


def cpu_oracle_regions(layers: OracleLayers, steps: int, warmup: int, min_seconds: float, max_seconds: float):
    """Times of regions of exactly `steps` oracle layer steps (after `warmup`
    untimed steps), repeated until they cover min_seconds (at least 3
    regions) or max_seconds has passed."""
    for i in range(warmup):
        layers.step(i)
    times, i0, t_start = [], warmup, time.perf_counter()
    while True:
        t0 = time.perf_counter()
        for i in range(steps):
            layers.step(i0 + i)
        times.append(time.perf_counter() - t0)
        i0 += steps
        if (len(times) >= 3 and sum(times) >= min_seconds) or time.perf_counter() - t_start >= max_seconds:
            return times


def cpu_baseline(seconds):
    import oracle
    layers = OracleLayers()
    times = cpu_oracle_regions(layers, 32, 2, seconds, 3 * seconds)
    el = float(statistics.median(times))
    return {"value": round(layers.weight_bytes * 32 / el / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "host_cpus": os.cpu_count(),
            "sample": f"{len(times)} regions of 32 layer steps of the headline workload (7 matrices, every output, "
                      f"rotating over the same {len(layers.copies)} layer copies), {sum(times):.1f} s wall, median "
                      f"region, OpenMP over weight rows"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    layers = OracleLayers()
    steps = args.steps
    # bounded: regions of exactly K steps until REF_MIN_SECONDS are covered
    # (at least 3 regions), at most ~REF_MAX_SECONDS
    times = cpu_oracle_regions(layers, steps, args.warmup, REF_MIN_SECONDS, REF_MAX_SECONDS)
    el = float(statistics.median(times))
    value = layers.weight_bytes * steps / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic (seeded random K-quant superblocks and N(0,1) activations)",
            "config": headline_config(world),
            "timing": {"how": "the CPU oracle (scalar C, OpenMP over weight rows) on the host cores: regions of "
                              "exactly K layer steps after W untimed ones, repeated until "
                              f"{REF_MIN_SECONDS:.0f} s are covered; "
                              "value and ms_per_step from the median region",
                       "regions": len(times), "median_ms": round(el * 1e3, 3), "total_s": round(sum(times), 2)},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{len(times)} regions of {steps} layer steps (the headline workload, every "
                                       f"output)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=DEFAULT_LAYER_COPIES, help="rotating layer copies (weights > L2)")
    ap.add_argument("--gemm-reps", type=int, default=20)
    ap.add_argument("--no-gemm", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
