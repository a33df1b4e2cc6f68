"""Benchmark of the small-M FP8 block-scaled linear layer on GB300.

Default workload: one decode pass at M = 8 tokens -- 256 FP8 GEMMs cycling
the four layer shapes 5,120 x 5,120, 34,816 x 5,120, 5,120 x 17,408 and
7,168 x 5,120 (N x K; 64 of each, every one with its own weights, 21.1 GB)
followed by the 248,320 x 5,120 output layer (1.27 GB): 22.4 GB of E4M3
weights with 128x128 fp32 block scales, bf16 activations cast per token per
128 K on the way in, bf16 output.  One step = one such pass through the
library's fused entry point (257 calls; the activation cast runs in the GEMM
prologue or as its own kernel, whichever the library's rule picks), replayed
from a CUDA graph with programmatic dependent launch between the layers.
The weights (22.4 GB) are far larger than L2, so every step reads them from
HBM.

Metric: us per GEMM and achieved HBM GB/s (algorithmic bytes: Wq + s_w +
X bf16 + Y bf16 per GEMM) as a fraction of the measured HBM peak.  ``value``
is the whole-job GB/s over all ranks.  The same JSON line carries, under
``configs``, the other workloads measured on the same weights: each layer
shape alone (64 distinct weights cycled), the output layer at M = 1 and 8
(FP8, with the greedy next-token choice, and the bf16 comparison GEMM), and
the pass at M = 1 ... 512.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode_pass|square_decode|mlp_up|mlp_down|vocab|tiny
                              |mx_<layer>]
                  [--m M] [--no-sweep] [--out-dir DIR]

``--workload mx_<layer>`` (mx_square_decode, ...) times the same layer in the
MX variant (its activation cast + MX GEMM per layer; our arm only).

Multi-GPU (torchrun): each rank runs its own replica on its own GPU (the
layer needs no exchange between GPUs); the barrier + max-over-ranks timing
gives whole-job throughput ("scaling": "weak").
``--impl reference`` times the CPU oracle (the plain fp64 restatement used as
the parity checker) on the host cores on a bounded sample of the same
workload.
"""
import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/GEMM and achieved HBM GB/s (% of GB300 peak) for FP8 block-scaled GEMM, M=1–64"
UNIT = "GB/s"
KERNEL_SOURCES = ["gemm_kernel.cuh", "ptx.cuh", "quant_math.cuh", "plan.cuh", "gemm_launch.cuh"]

# The decode pass: (N, K) of the four layer shapes, 64 distinct layers each in
# this cycling order, then the output layer.
PASS_SHAPES = ((5120, 5120), (34816, 5120), (5120, 17408), (7168, 5120))
PASS_REPEAT = 64
VOCAB = (248320, 5120)


# ---------------------------------------------------------------- workloads
def workload(name, m_override=None):
    """A layer workload; ``mx_<name>`` is the same layer in the MX variant."""
    from fp8_block_scaled_token_gb300 import synth
    cfg = dict(synth.WORKLOADS[name[3:] if name.startswith("mx_") else name])
    if m_override:
        cfg["M"] = m_override
    return cfg


def algorithmic_bytes(M, N, K, fused=True):
    """Bytes one GEMM must move at minimum: Wq + s_w + X (bf16, or Aq + s_a
    when pre-quantised) + Y bf16."""
    nb, kg = (N + 127) // 128, K // 128
    act = 2 * M * K if fused else M * K + 4 * M * kg
    return N * K + 4 * nb * kg + act + 2 * M * N


def bf16_bytes(M, N, K):
    return 2 * N * K + 2 * M * K + 2 * M * N


def mx_bytes(M, N, K):
    """Bytes of one MX layer (1x32 power-of-two scales): codes + one scale
    byte per 32 K per weight row + X bf16 + Y bf16."""
    return N * K + N * K // 32 + 2 * M * K + 2 * M * N


def pass_workload(M):
    """The decode-pass workload of the JSON line's config (both arms)."""
    return {"workload": "decode_pass M=%d: 256 GEMMs cycling %s (N x K, 64 distinct weights each) "
                        "+ the 248320x5120 output layer" % (M, ", ".join("%dx%d" % s for s in PASS_SHAPES)),
            "M": M, "gemms_per_step": len(pass_layers_shapes()),
            "weight_bytes": sum(N * K for N, K in pass_layers_shapes())}


def pass_layers_shapes():
    """(N, K) of the 257 GEMMs of one decode pass, in order."""
    return [PASS_SHAPES[i % 4] for i in range(4 * PASS_REPEAT)] + [VOCAB]


def pass_bytes(M):
    return sum(algorithmic_bytes(M, N, K) for N, K in pass_layers_shapes())


# ---------------------------------------------------------------- multi-rank helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world):
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_value(bytes_per_step, steps, world, seconds):
    """Aggregate GB/s: every rank moved bytes_per_step * steps in at most
    `seconds` (the max over ranks)."""
    return bytes_per_step * steps * world / seconds / 1e9


# ---------------------------------------------------------------- peaks, clocks, traffic
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region (read-only queries)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, out_dir=None):
        self.index = index
        self.proc = None
        base = out_dir or tempfile.mkdtemp(prefix="fp8bs_clocks_")
        self.path = os.path.join(base, "clocks_%s.csv" % str(index).replace("/", "_"))

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.6)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def gpu_query_id(dev):
    """nvidia-smi -i argument for a torch device: its UUID when torch knows
    it (indices differ under CUDA_VISIBLE_DEVICES), else its index."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    return str(dev.index if dev.index is not None else 0)


def _code_only(text):
    """C++ source without its comments and with whitespace runs collapsed:
    what the compiler sees, so a comment edit does not change the hash."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    """First 16 hex digits of the sha256 of the GEMM kernel's sources, their
    comments and whitespace removed (string literals in them hold no //)."""
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "fp8_block_scaled_token_gb300", "csrc", n)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(key):
    """DRAM bytes (read + write) of the GEMM kernel for `key` from the
    committed ncu summary (profiles/gemm_traffic.txt: "kernel_source_hash
    <h>" then "<key> <bytes> ..."), if it was taken on the current kernel
    source; else None."""
    p = os.path.join(ROOT, "profiles", "gemm_traffic.txt")
    if not os.path.exists(p):
        return None
    entries = {}
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 2 and not line.startswith("#"):
                entries[parts[0]] = parts[1]
    if entries.get("kernel_source_hash") != kernel_source_hash():
        return None
    v = entries.get(key)
    return None if v is None else int(v)


def kernel_runs():
    """The library's device-side launch counters (synchronises the device):
    every kernel of the library adds one to its slot when it starts."""
    import fp8_block_scaled_token_gb300 as fb
    out = (ctypes.c_ulonglong * 128)()
    rc = fb.lib().fp8bs_testhook_kernel_runs(0, 128, out)
    if rc != 0:
        raise RuntimeError("launch counters: " + fb.status_string(rc))
    return [int(v) for v in out]


# ---------------------------------------------------------------- CPU oracle timing
class OracleSample:
    """The CPU oracle on one layer shape: activation cast + fp64 GEMM over the
    first `ncols` output columns, weights quantised beforehand (as on the GPU
    path, where weight quantisation is offline)."""

    def __init__(self, M, N, K, seed, ncols=None):
        import numpy as np
        import torch

        import oracle
        from fp8_block_scaled_token_gb300 import synth
        self.o = oracle.default()
        self.threads = oracle.default_threads()
        self.M, self.N, self.K = M, N, K
        self.ncols = N if ncols is None else max(1, min(N, ncols))
        rows = min(N, ((self.ncols + 127) // 128) * 128)
        x = synth.activations(M, K, seed=seed)
        w = synth.weights(rows, K, seed=seed + 1000).numpy()
        self.xb = x.view(torch.int16).numpy().view(np.uint16)
        self.wq, self.ws = self.o.quant_weight(w)
        self.cols = np.arange(self.ncols, dtype=np.int32)

    def run_once(self):
        xq, xs = self.o.quant_act(self.xb)
        self.o.gemm_fp8(xq, xs, self.wq, self.ws, cols=self.cols, nthreads=self.threads)

    def bytes_per_run(self):
        n, K, M = self.ncols, self.K, self.M
        return n * K + 4 * ((n + 127) // 128) * (K // 128) + 2 * M * K + 2 * M * n


class OracleMix:
    """The oracle on a bounded sample of a workload made of several layer
    shapes: a slice of the output columns of every shape (an equal share of
    the time budget each, at most 8,192 columns), run back to back.  The
    oracle's cost per weight byte does not depend on the shape, so the
    sampled mix gives the rate of the whole workload."""

    def __init__(self, M, shapes, seconds, seed=1):
        probe = OracleSample(M, shapes[0][0], shapes[0][1], seed, ncols=128)
        probe.run_once()  # first run pays one-time costs
        t0 = time.perf_counter()
        probe.run_once()
        per_byte = (time.perf_counter() - t0) / probe.bytes_per_run()
        share = seconds / len(shapes)
        self.parts = []
        for i, (N, K) in enumerate(shapes):
            ncols = int(max(1, min(N, 8192, share / max(per_byte * K, 1e-12))))
            self.parts.append(OracleSample(M, N, K, seed + i, ncols=ncols))
        self.threads = probe.threads
        self.M = M
        self.shapes = shapes

    def run_once(self):
        for p in self.parts:
            p.run_once()

    def bytes_per_run(self):
        return sum(p.bytes_per_run() for p in self.parts)

    def describe(self):
        return ("oracle act-cast + fp64 GEMM at M=%d over the first %s output columns of the layer shapes %s, "
                "%d threads" % (self.M, "/".join(str(p.ncols) for p in self.parts),
                                ", ".join("%dx%d" % s for s in self.shapes), self.threads))


def oracle_rate(M, shapes, seconds, seed=1):
    """Time the oracle on a sample of the workload for about `seconds`.
    Returns (GB/s of algorithmic bytes, threads, sample text)."""
    mix = OracleMix(M, shapes, seconds / 3.0, seed)
    reps, t0 = 0, time.perf_counter()
    while True:
        mix.run_once()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    gbs = mix.bytes_per_run() * reps / el / 1e9
    return gbs, mix.threads, "%d runs of %s, %.1f s" % (reps, mix.describe(), el)


# ---------------------------------------------------------------- timing helpers
def graph_of(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()  # untimed: uploads the graph
    torch.cuda.synchronize()
    return g


def time_replays(g, reps, stream):
    """Seconds for `reps` replays of graph g, CUDA events on `stream`."""
    import torch
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        s.record(stream)
        for _ in range(reps):
            g.replay()
        e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / 1e3


class PassWeights:
    """The 257 quantised weight matrices of one decode pass, resident in HBM
    in the tiled layout (seeds 100 + i, the output layer 356)."""

    def __init__(self, dev):
        import torch

        import fp8_block_scaled_token_gb300 as fb
        from fp8_block_scaled_token_gb300 import synth
        self.layers = []
        for i, (N, K) in enumerate(pass_layers_shapes()):
            w = synth.weights(N, K, seed=100 + i, device=dev)
            self.layers.append((N, K) + fb.fp8_quant_weight_blocks(w, tiled=True))
            del w
        torch.cuda.synchronize()

    def of_shape(self, N, K):
        return [l for l in self.layers if l[0] == N and l[1] == K]


class PassRunner:
    """Buffers and the call sequence of one decode pass at M tokens."""

    def __init__(self, weights, M, dev, layers=None):
        import torch

        import fp8_block_scaled_token_gb300 as fb
        from fp8_block_scaled_token_gb300 import synth
        self.fb = fb
        self.layers = weights.layers if layers is None else layers
        self.M = M
        Ks = sorted({K for _, K, _, _ in self.layers})
        Ns = sorted({N for N, _, _, _ in self.layers})
        self.x = {K: synth.activations(M, K, seed=1, device=dev) for K in Ks}
        self.y = {N: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for N in Ns}
        wsz = max(fb.fp8_blockscaled_gemm_workspace_size(M, N, K) for N, K, _, _ in self.layers)
        self.work = fb.make_workspace(wsz, dev)
        self.bytes = sum(algorithmic_bytes(M, N, K) for N, K, _, _ in self.layers)
        self.flops = sum(2.0 * M * N * K for N, K, _, _ in self.layers)

    def run(self, flags=None, x=None):
        fb = self.fb
        f = fb.FLAG_OVERLAP_PREV if flags is None else flags
        xs = self.x if x is None else x
        for N, K, wq, ws in self.layers:
            fb.fp8_blockscaled_gemm_fused(xs[K], wq, ws, y=self.y[N], workspace=self.work, flags=f, n=N)


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.workload == "decode_pass":
        run_pass(args, world, rank, dev)
    else:
        run_layer(args, world, rank, dev)


def run_pass(args, world, rank, dev):
    import torch

    import fp8_block_scaled_token_gb300 as fb
    M = args.m or 8
    peak, peak_kind = measured_peaks()
    weights = PassWeights(dev)
    runner = PassRunner(weights, M, dev)
    stream = torch.cuda.Stream(device=dev)

    for _ in range(args.warmup):
        runner.run()
    torch.cuda.synchronize()
    g = graph_of(runner.run, stream)
    if fb.workspace_status(runner.work) != 0:
        raise RuntimeError("device-side timeout during warm-up")

    runs0 = kernel_runs()
    clocks = ClockSampler(gpu_query_id(dev), args.out_dir)
    clocks.start()
    barrier(world)
    elapsed = time_replays(g, args.steps, stream)
    barrier(world)
    clk = clocks.stop()
    runs1 = kernel_runs()
    launches = sum(b - a for a, b in zip(runs0, runs1))
    t_max = max_over_ranks(elapsed, world)
    if fb.workspace_status(runner.work) != 0:
        raise RuntimeError("device-side timeout in the timed region")

    steps = args.steps
    value = whole_job_value(runner.bytes, steps, world, t_max)
    per_pass_s = elapsed / steps
    achieved = runner.bytes / per_pass_s / 1e9

    # end to end through the public API, eagerly, with host buffers: the
    # step's activations copied in from pinned host memory and the output
    # layer's logits read back, every step
    x_host = {K: t.cpu().pin_memory() for K, t in runner.x.items()}
    x_dev = {K: torch.empty_like(t) for K, t in runner.x.items()}
    yv = runner.y[VOCAB[0]]
    y_host = torch.empty(tuple(yv.shape), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(steps, 100))

    def e2e_step():
        for K in x_dev:
            x_dev[K].copy_(x_host[K], non_blocking=True)
        runner.run(x=x_dev)
        y_host.copy_(yv, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(e2e_steps):
        e2e_step()
    e.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(s.elapsed_time(e) / 1e3, world)
    e2e_value = whole_job_value(runner.bytes, e2e_steps, world, e2e_s)
    h2d = sum(t.numel() * 2 for t in x_host.values())
    d2h = y_host.numel() * 2

    configs = []
    if not args.no_sweep:
        configs = sweep(weights, dev, stream, peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, threads, sample = oracle_rate(M, list(PASS_SHAPES) + [VOCAB], seconds=args.cpu_seconds)
        cpu = {"value": round(gbs, 6), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}

    if rank == 0:
        n_gemm = len(runner.layers)
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(t_max / steps * 1e3, 6),
            "us_per_gemm": round(t_max / steps / n_gemm * 1e6, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3xe4m3->f32",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) bf16 activations)",
            "config": {**pass_workload(M),
                       "kernel": "fp8_blockscaled_gemm_fused (activation cast + swap-AB tcgen05 split-K GEMM)",
                       "weights": "E4M3 tiled layout (one contiguous 16 KB run per 128x128 tile)",
                       "l2": "inputs larger than L2: 22.4 GB of distinct weights per step",
                       "timing": "CUDA graph of one pass replayed per step; PDL between launches; CUDA events",
                       "parallelism": "replica per GPU" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": profiled_traffic("pass_M%d" % M),
                         "peak_kind": peak_kind, "kernel": "gemm_small_m_kernel (with its activation cast)",
                         "scope": "per step: algorithmic bytes of the 257 GEMMs over the step's time",
                         "bytes_per_step": runner.bytes, "step_us": round(per_pass_s * 1e6, 3)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": round(e2e_s / e2e_steps * 1e3, 4),
                    "how": "257 eager calls of the public fused entry point per step (no graph), activations "
                           "copied in from pinned host memory and the output layer's logits read back"},
            "gpu_launches": launches,
            "gpu_launches_how": "the library's device-side launch counters, read before and after the timed region",
            "clocks": clk,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
        if args.out_dir:
            os.makedirs(args.out_dir, exist_ok=True)
            with open(os.path.join(args.out_dir, "bench_line.json"), "w") as fh:
                json.dump(line, fh, indent=1)


def sweep(weights, dev, stream, peak):
    """The other workloads on the pass's resident weights (printed to stderr
    as they complete, returned for the JSON line)."""
    import torch

    import fp8_block_scaled_token_gb300 as fb
    from fp8_block_scaled_token_gb300 import synth
    out = []

    def emit(d):
        out.append(d)
        print(json.dumps(d), file=sys.stderr, flush=True)

    def layer_row(name, M, N, K, us, nbytes):
        return {"workload": name, "M": M, "N": N, "K": K, "us": round(us, 3), "GB/s": round(nbytes / us / 1e3, 1),
                "frac": round(nbytes / us / 1e3 / peak, 4), "TFLOP/s": round(2.0 * M * N * K / us / 1e6, 1)}

    # each layer shape alone: its 64 distinct weights cycled in one graph
    names = {(5120, 5120): "square_decode", (34816, 5120): "mlp_up", (5120, 17408): "mlp_down",
             (7168, 5120): "attn_7168x5120"}
    for (N, K), name in names.items():
        for M in ((1, 8, 64, 128, 512) if name == "square_decode" else (8,)):
            r = PassRunner(weights, M, dev, layers=weights.of_shape(N, K))
            g = graph_of(r.run, stream)
            reps = max(1, 2000 // len(r.layers))
            us = time_replays(g, reps, stream) * 1e6 / (reps * len(r.layers))
            emit(layer_row(name, M, N, K, us, algorithmic_bytes(M, N, K)))
            del g, r
    # the output layer: FP8 plain, FP8 with the greedy choice (logits not stored)
    vN, vK = VOCAB
    vocab = weights.of_shape(vN, vK)
    for M in (1, 8):
        r = PassRunner(weights, M, dev, layers=vocab)
        g = graph_of(r.run, stream)
        us = time_replays(g, 50, stream) * 1e6 / 50
        emit(layer_row("vocab", M, vN, vK, us, algorithmic_bytes(M, vN, vK)))
        tok = torch.empty((M,), dtype=torch.int32, device=dev)
        lg = torch.empty((M,), dtype=torch.float32, device=dev)
        _, _, wq, ws = vocab[0]

        def greedy(r=r, tok=tok, lg=lg, wq=wq, ws=ws):
            fb.fp8_blockscaled_gemm_fused_greedy(r.x[vK], wq, ws, store_y=False, token=tok, logit=lg,
                                                 workspace=r.work, flags=fb.FLAG_OVERLAP_PREV, n=vN)
        g = graph_of(greedy, stream)
        us = time_replays(g, 50, stream) * 1e6 / 50
        emit(layer_row("vocab_greedy", M, vN, vK, us, algorithmic_bytes(M, vN, vK) - 2 * M * vN))
        del g, r
    # the bf16 comparison GEMM of the output layer (two distinct bf16 copies)
    wb = [fb.bf16_pack_weights_tiled(synth.weights(vN, vK, seed=300 + i, device=dev).to(torch.bfloat16))
          for i in range(2)]
    for M in (1, 8):
        x = synth.activations(M, vK, seed=4, device=dev)
        y = torch.empty((M, vN), dtype=torch.bfloat16, device=dev)
        work = fb.make_workspace(fb.bf16_gemm_ref_workspace_size(M, vN, vK), dev)

        def f(x=x, y=y, work=work):
            for w in wb:
                fb.bf16_gemm_ref(x, w, y=y, workspace=work, flags=fb.FLAG_OVERLAP_PREV, n=vN)
        g = graph_of(f, stream)
        us = time_replays(g, 25, stream) * 1e6 / 50
        emit(layer_row("vocab_bf16", M, vN, vK, us, bf16_bytes(M, vN, vK)))
        del g
    del wb
    torch.cuda.empty_cache()
    # the native block-scaled (MX) variant: activation cast + MX GEMM per
    # layer (a different numeric contract: 1x32 power-of-two scales), on 64
    # distinct square layers (also at 128 and 512 tokens, beside the FP8
    # square layer's rows) and on the output layer
    for (N, K), name, R, Ms in (((5120, 5120), "mx_square_decode", 64, (1, 8, 128, 512)),
                                (VOCAB, "mx_vocab", 2, (1, 8))):
        mx = [fb.fp8_mx_quant_weights(synth.weights(N, K, seed=400 + i, device=dev)) for i in range(R)]
        for M in Ms:
            x = synth.activations(M, K, seed=1, device=dev)
            xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
            xa = torch.empty(((M + 127) // 128 * (K // 128), 512), dtype=torch.uint8, device=dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            work = fb.make_workspace(fb.fp8_mx_gemm_workspace_size(M, N, K), dev)

            def f(x=x, xq=xq, xa=xa, y=y, work=work, mx=mx, N=N):
                for wq, wa in mx:
                    fb.fp8_mx_quant_act(x, xq=xq, xs_atoms=xa, flags=fb.FLAG_OVERLAP_PREV)
                    fb.fp8_mx_gemm(xq, xa, wq, wa, N, y=y, workspace=work, flags=fb.FLAG_OVERLAP_PREV)
            g = graph_of(f, stream)
            reps = max(1, 2000 // R) if R > 2 else 25
            us = time_replays(g, reps, stream) * 1e6 / (reps * R)
            emit(layer_row(name, M, N, K, us, mx_bytes(M, N, K)))
            del g
        del mx
    torch.cuda.empty_cache()
    # the whole pass at every token count
    for M in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512):
        r = PassRunner(weights, M, dev)
        g = graph_of(r.run, stream)
        reps = 20 if M <= 64 else 5
        s = time_replays(g, reps, stream) / reps
        emit({"workload": "decode_pass_257", "M": M, "ms": round(s * 1e3, 4),
              "GB/s": round(r.bytes / s / 1e9, 1), "frac": round(r.bytes / s / 1e9 / peak, 4),
              "TFLOP/s": round(r.flops / s / 1e12, 1)})
        del g, r
    torch.cuda.empty_cache()
    return out


def run_layer(args, world, rank, dev):
    """One layer shape: successive steps walk a ring of distinct weight
    layers whose total size is more than 4x the L2 cache."""
    import torch

    import fp8_block_scaled_token_gb300 as fb
    from fp8_block_scaled_token_gb300 import synth
    cfg = workload(args.workload, args.m)
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    mx = args.workload.startswith("mx_")  # the MX variant: its cast + MX GEMM per layer
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 1024 * 1024
    R = max(2, min(64, math.ceil(4 * l2 / (N * K))))
    layers = []
    for i in range(R):
        w = synth.weights(N, K, seed=100 + i, outlier_p=cfg.get("w_outlier_p", 0.0), device=dev)
        layers.append((N, K) + (fb.fp8_mx_quant_weights(w) if mx else fb.fp8_quant_weight_blocks(w, tiled=True)))
        del w
    x = synth.activations(M, K, seed=cfg["seed"], outlier_p=cfg.get("x_outlier_p", 0.0), device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    work = fb.make_workspace((fb.fp8_mx_gemm_workspace_size if mx else fb.fp8_blockscaled_gemm_workspace_size)(M, N, K),
                             dev)
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    xa = torch.empty(((M + 127) // 128 * (K // 128), 512), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def layer(xin, wq, ws, flags):
        if mx:
            fb.fp8_mx_quant_act(xin, xq=xq, xs_atoms=xa, flags=flags)
            fb.fp8_mx_gemm(xq, xa, wq, ws, N, y=y, workspace=work, flags=flags)
        else:
            fb.fp8_blockscaled_gemm_fused(xin, wq, ws, y=y, workspace=work, flags=flags, n=N)

    def ring():
        for _, _, wq, ws in layers:
            layer(x, wq, ws, fb.FLAG_OVERLAP_PREV)

    for _ in range(max(1, args.warmup // R + 1)):
        ring()
    g = graph_of(ring, stream)
    reps = max(1, args.steps // R)
    steps = reps * R
    runs0 = kernel_runs()
    clocks = ClockSampler(gpu_query_id(dev), args.out_dir)
    clocks.start()
    barrier(world)
    elapsed = time_replays(g, reps, stream)
    barrier(world)
    clk = clocks.stop()
    launches = sum(b - a for a, b in zip(runs0, kernel_runs()))
    t_max = max_over_ranks(elapsed, world)
    if fb.workspace_status(work) != 0:
        raise RuntimeError("device-side timeout in the timed region")
    nbytes = mx_bytes(M, N, K) if mx else algorithmic_bytes(M, N, K)
    peak, peak_kind = measured_peaks()
    achieved = nbytes / (elapsed / steps) / 1e9

    x_host = x.cpu().pin_memory()
    y_host = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    e2e_steps = min(steps, 2000)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    s.record()
    for i in range(e2e_steps):
        x_dev.copy_(x_host, non_blocking=True)
        _, _, wq, ws = layers[i % R]
        layer(x_dev, wq, ws, 0)
        y_host.copy_(y, non_blocking=True)
    e.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(s.elapsed_time(e) / 1e3, world)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not mx:
        gbs, threads, sample = oracle_rate(M, [(N, K)], seconds=args.cpu_seconds, seed=cfg["seed"])
        cpu = {"value": round(gbs, 6), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(whole_job_value(nbytes, steps, world, t_max), 3), "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(t_max / steps * 1e3, 6),
            "us_per_gemm": round(t_max / steps * 1e6, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3xe4m3->f32",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) bf16 activations)",
            "config": {"workload": "%s M=%d N=%d K=%d" % (args.workload, M, N, K), "M": M, "N": N, "K": K,
                       "weights_ring": R, "l2": "ring of %d distinct layers (%.0f MB) > 4x L2" % (R, R * N * K / 1e6),
                       "timing": "CUDA graph of %d launches replayed; PDL between launches; CUDA events" % R,
                       "parallelism": "replica per GPU" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": None if mx else profiled_traffic("M%d_N%d_K%d" % (M, N, K)),
                         "peak_kind": peak_kind, "bytes_per_launch": nbytes,
                         "launch_us": round(elapsed / steps * 1e6, 4)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(whole_job_value(nbytes, e2e_steps, world, e2e_s), 3), "unit": UNIT,
                    "h2d_bytes_per_step": 2 * M * K, "d2h_bytes_per_step": 2 * M * N, "steps": e2e_steps},
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- reference arm: the CPU oracle
def run_reference(args, world, rank):
    if rank != 0:
        return
    if args.workload.startswith("mx_"):
        raise SystemExit("bench.py: the reference arm times the oracle of the FP8 block-scaled layer; "
                         "the MX variant is a different numeric contract")
    if args.workload == "decode_pass":
        M = args.m or 8
        shapes = list(PASS_SHAPES) + [VOCAB]
        config = pass_workload(M)
    else:
        cfg = workload(args.workload, args.m)
        M, shapes = cfg["M"], [(cfg["N"], cfg["K"])]
        config = {"workload": "%s M=%d N=%d K=%d" % (args.workload, M, cfg["N"], cfg["K"]), "M": M, "N": cfg["N"],
                  "K": cfg["K"]}
    # size each step so that the warm-up and timed steps together stay
    # within about two minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    mix = OracleMix(M, shapes, budget)
    for _ in range(args.warmup):
        mix.run_once()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        mix.run_once()
    el = time.perf_counter() - t0
    value = mix.bytes_per_run() * args.steps / el / 1e9
    line = {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / max(1, args.steps) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) bf16 activations)",
            "config": config,
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "kind": "oracle", "cores": mix.threads,
                             "sample": "each step: " + mix.describe()},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_pass")
    ap.add_argument("--m", type=int, default=None)
    ap.add_argument("--no-sweep", action="store_true", help="skip the other workloads (configs key)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--out-dir", default=None,
                    help="directory for the clock samples and a copy of the JSON line (default: a temporary one)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1 and args.impl == "ours":
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
