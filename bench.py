"""Benchmark of the small-M FP8 block-scaled linear layer on GB300.

Default workload: the square decode layer, M = 8 tokens, N = K = 5120
(E4M3 weights with 128x128 fp32 block scales, bf16 activations cast per token
per 128 inside the GEMM, bf16 output).  One step = one batch of 8 tokens
through one such layer: the fused activation-cast + block-scaled GEMM, one
kernel launch.  Successive steps walk a ring of distinct weight layers whose
total size is more than 4x the L2 cache, so every step reads its weights from
HBM.  The timed region replays CUDA graphs of those launches (programmatic
dependent launch lets each GEMM start streaming its weights while the previous
one drains).

Metric: us per GEMM and achieved HBM GB/s (algorithmic bytes: Wq + s_w + X
bf16 + Y bf16) as a fraction of the measured HBM peak.  ``value`` is the
whole-job GB/s over all ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload square_decode|mlp_up|mlp_down|vocab|tiny] [--m M]
                  [--configs]   (also sweep the other workloads, to stderr)

Multi-GPU (torchrun): each rank runs its own replica on its own GPU (the
layer needs no exchange between GPUs); the barrier + max-over-ranks timing
gives whole-job throughput ("scaling": "weak").
``--impl reference`` times the CPU oracle (the plain fp64 restatement used as
the parity checker) on the host cores on a bounded sample of the same
workload.
"""
import argparse
import hashlib
import json
import math
import os
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


# ---------------------------------------------------------------- workloads
def workload(name, m_override=None):
    from fp8_block_scaled_token_gb300 import synth
    cfg = dict(synth.WORKLOADS[name])
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


def kernel_source_hash():
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "fp8_block_scaled_token_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(M, N, K):
    """DRAM bytes per launch of the GEMM from the committed ncu summary
    (profiles/gemm_traffic.txt: "kernel_source_hash <h>" then
    "M<m>_N<n>_K<k> <bytes per launch> ..."), if it was taken on the current
    kernel source; else None."""
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
    v = entries.get("M%d_N%d_K%d" % (M, N, K))
    return None if v is None else int(v)


# ---------------------------------------------------------------- CPU oracle timing
class OracleSample:
    """The CPU oracle on one layer: activation cast + fp64 GEMM over the first
    `ncols` output columns, weights quantised beforehand (as on the GPU path,
    where weight quantisation is offline)."""

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

    def describe(self):
        return "oracle act-cast + fp64 GEMM, M=%d K=%d over %d of %d output columns, %d threads" % (
            self.M, self.K, self.ncols, self.N, self.threads)


def oracle_rate(M, N, K, seconds, seed=1):
    """Time the oracle on the full layer for about `seconds` (at least one
    run).  Returns (GB/s of algorithmic bytes, threads, sample text)."""
    smp = OracleSample(M, N, K, seed)
    reps, t0 = 0, time.perf_counter()
    while True:
        smp.run_once()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    gbs = smp.bytes_per_run() * reps / el / 1e9
    return gbs, smp.threads, "%d runs of %s, %.1f s" % (reps, smp.describe(), el)


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import fp8_block_scaled_token_gb300 as fb
    from fp8_block_scaled_token_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workload(args.workload, args.m)
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 1024 * 1024
    layer_bytes = N * K
    R = max(2, min(64, math.ceil(4 * l2 / layer_bytes)))

    # resident inputs: R distinct quantised layers, one activation batch
    wqs, wss = [], []
    for i in range(R):
        w = synth.weights(N, K, seed=100 + i, outlier_p=cfg.get("w_outlier_p", 0.0), device=dev)
        wq, ws = fb.fp8_quant_weight_blocks(w, tiled=True)
        wqs.append(wq)
        wss.append(ws)
        del w
    x = synth.activations(M, K, seed=cfg["seed"], outlier_p=cfg.get("x_outlier_p", 0.0), device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K), dev)
    flags = fb.FLAG_OVERLAP_PREV
    torch.cuda.synchronize()

    def step(i):
        fb.fp8_blockscaled_gemm_fused(x, wqs[i % R], wss[i % R], y=y, workspace=work, flags=flags, n=N)

    # warm-up (eager), then capture one ring pass and the remainder as graphs
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    steps = args.steps
    full_reps, rem = divmod(steps, R)
    stream = torch.cuda.Stream(device=dev)
    g_ring = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ring, stream=stream):
        for i in range(R):
            step(i)
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                step(i)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g_ring.replay()            # untimed: uploads the graph
        if g_rem is not None:
            g_rem.replay()
    torch.cuda.synchronize()
    if fb.workspace_status(work) != 0:
        raise RuntimeError("device-side timeout during warm-up")

    clocks = ClockSampler(gpu_query_id(dev), args.out_dir)
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(full_reps):
            g_ring.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    elapsed = start.elapsed_time(end) / 1e3
    clk = clocks.stop()
    t_max = max_over_ranks(elapsed, world)
    if fb.workspace_status(work) != 0:
        raise RuntimeError("device-side timeout in the timed region")

    bytes_step = algorithmic_bytes(M, N, K, fused=True)
    value = whole_job_value(bytes_step, steps, world, t_max)
    per_launch_s = elapsed / steps
    achieved = bytes_step / per_launch_s / 1e9
    peak, peak_kind = measured_peaks()

    # eager (no graph) for context, same launches
    eager_steps = min(steps, 2000)
    torch.cuda.synchronize()
    start.record()
    for i in range(eager_steps):
        step(i)
    end.record()
    torch.cuda.synchronize()
    eager_us = start.elapsed_time(end) * 1e3 / eager_steps

    # end to end through the public API with host buffers: pinned X in, Y out, every step
    x_host = x.cpu().pin_memory()
    y_host = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    e2e_steps = min(steps, 5000)
    for i in range(3):
        x_dev.copy_(x_host, non_blocking=True)
        fb.fp8_blockscaled_gemm_fused(x_dev, wqs[i % R], wss[i % R], y=y, workspace=work, n=N)
        y_host.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    barrier(world)
    start.record()
    for i in range(e2e_steps):
        x_dev.copy_(x_host, non_blocking=True)
        fb.fp8_blockscaled_gemm_fused(x_dev, wqs[i % R], wss[i % R], y=y, workspace=work, n=N)
        y_host.copy_(y, non_blocking=True)
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(start.elapsed_time(end) / 1e3, world)
    e2e_value = whole_job_value(bytes_step, e2e_steps, world, e2e_s)

    # two-kernel path (standalone cast + GEMM) and bf16 baseline, for context
    extra = {}
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    xs = torch.empty((M, K // 128), dtype=torch.float32, device=dev)

    def step2(i):
        fb.fp8_quant_act(x, xq=xq, xs=xs, flags=flags)
        fb.fp8_blockscaled_gemm(xq, xs, wqs[i % R], wss[i % R], y=y, workspace=work, flags=flags, n=N)

    for i in range(20):
        step2(i)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        for i in range(R):
            step2(i)
    torch.cuda.synchronize()
    reps2 = max(1, min(full_reps, 2000 // R + 1))
    with torch.cuda.stream(stream):
        g2.replay()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(reps2):
            g2.replay()
        end.record(stream)
    torch.cuda.synchronize()
    extra["two_kernel_us_per_gemm"] = start.elapsed_time(end) * 1e3 / (reps2 * R)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, threads, sample = oracle_rate(M, N, K, seconds=args.cpu_seconds, seed=cfg["seed"])
        cpu = {"value": round(gbs, 6), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}

    if rank == 0:
        traffic = profiled_traffic(M, N, K)
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(t_max / steps * 1e3, 6),
            "us_per_gemm": round(t_max / steps * 1e6, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3xe4m3->f32",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) bf16 activations)",
            "config": {"workload": "%s M=%d N=%d K=%d" % (args.workload, M, N, K), "M": M, "N": N, "K": K,
                       "kernel": "fp8_blockscaled_gemm_fused (cast fused, swap-AB tcgen05, split-K)",
                       "weights": "E4M3 tiled layout (one contiguous 16 KB run per 128x128 tile)",
                       "weights_ring": R, "l2": "ring of %d distinct %.1f MB weight layers (%.0f MB) > 4x L2 (%.0f MB)" % (
                           R, layer_bytes / 1e6, R * layer_bytes / 1e6, l2 / 1e6),
                       "timing": "CUDA graphs of %d launches replayed; PDL between launches; CUDA events" % R,
                       "parallelism": "replica per GPU" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_kind": peak_kind,
                         "bytes_per_launch": bytes_step, "launch_us": round(per_launch_s * 1e6, 4)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": 2 * M * K,
                    "d2h_bytes_per_step": 2 * M * N, "steps": e2e_steps,
                    "us_per_step": round(e2e_s / e2e_steps * 1e6, 3)},
            "gpu_launches": steps,
            "clocks": clk,
            "context": {"eager_us_per_gemm": round(eager_us, 3), **{k: round(v, 3) for k, v in extra.items()}},
        }
        print(json.dumps(line), flush=True)

    if args.configs and rank == 0:
        sweep(args, dev)


# ---------------------------------------------------------------- extra configurations (stderr)
def time_graph(fn, reps_inner, reps_outer, stream):
    import torch
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(reps_inner):
            fn(i)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        torch.cuda.synchronize()
        s.record(stream)
        for _ in range(reps_outer):
            g.replay()
        e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / (reps_inner * reps_outer)


PASS_SHAPES = ((5120, 5120), (34816, 5120), (5120, 17408), (7168, 5120))  # (N, K)


def decode_pass(dev, stream, peak, Ms=(1, 2, 4, 8, 16, 32, 64, 128, 256, 512)):
    """One decode pass: 256 GEMMs cycling the four layer shapes, every one with
    its own weights (22.4 GB, seeds 100 + i), then the output layer; timed as
    one graph per token count M."""
    import torch

    import fp8_block_scaled_token_gb300 as fb
    from fp8_block_scaled_token_gb300 import synth
    layers = []
    for i in range(256):
        N, K = PASS_SHAPES[i % 4]
        w = synth.weights(N, K, seed=100 + i, device=dev)
        layers.append((N, K) + fb.fp8_quant_weight_blocks(w, tiled=True))
        del w
    vN, vK = workload("vocab")["N"], workload("vocab")["K"]
    w = synth.weights(vN, vK, seed=356, device=dev)
    layers.append((vN, vK) + fb.fp8_quant_weight_blocks(w, tiled=True))
    del w
    torch.cuda.synchronize()
    rows = []
    for M in Ms:
        xs = {K: synth.activations(M, K, seed=1, device=dev) for K in (5120, 17408)}
        ys = {N: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for N, _ in PASS_SHAPES + ((vN, vK),)}
        wsz = max(fb.fp8_blockscaled_gemm_workspace_size(M, N, K) for N, K, _, _ in layers)
        work = fb.make_workspace(wsz, dev)

        def f(i, xs=xs, ys=ys, work=work):
            for N, K, wq, ws in layers:
                fb.fp8_blockscaled_gemm_fused(xs[K], wq, ws, y=ys[N], workspace=work, flags=fb.FLAG_OVERLAP_PREV,
                                              n=N)
        us = time_graph(f, 1, 20, stream)
        b = sum(algorithmic_bytes(M, N, K) for N, K, _, _ in layers)
        flops = sum(2.0 * M * N * K for N, K, _, _ in layers)
        rows.append({"workload": "decode_pass_257", "M": M, "ms": round(us / 1e3, 4),
                     "GB/s": round(b / us / 1e3, 1), "frac": round(b / us / 1e3 / peak, 4),
                     "TFLOP/s": round(flops / us / 1e6, 1)})
        print(json.dumps(rows[-1]), file=sys.stderr, flush=True)
        del xs, ys, work
    del layers
    torch.cuda.empty_cache()
    return rows


def sweep(args, dev):
    import torch

    import fp8_block_scaled_token_gb300 as fb
    from fp8_block_scaled_token_gb300 import synth
    peak, _ = measured_peaks()
    stream = torch.cuda.Stream(device=dev)
    out = []
    l2 = 126 * 1024 * 1024
    for name, Ms in (("square_decode", (1, 8, 64, 128, 256, 512)), ("mlp_up", (8,)), ("mlp_down", (8,)),
                     ("vocab", (1, 8))):
        cfg = workload(name)
        N, K = cfg["N"], cfg["K"]
        R = max(1, min(32, math.ceil(4 * l2 / (N * K))))
        layers = []
        for i in range(R):
            w = synth.weights(N, K, seed=200 + i, outlier_p=cfg.get("w_outlier_p", 0.0), device=dev)
            layers.append(fb.fp8_quant_weight_blocks(w, tiled=True))
            del w
        for M in Ms:
            x = synth.activations(M, K, seed=cfg["seed"], outlier_p=cfg.get("x_outlier_p", 0.0), device=dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K), dev)

            def f(i, x=x, y=y, work=work, N=N):
                wq, ws = layers[i % R]
                fb.fp8_blockscaled_gemm_fused(x, wq, ws, y=y, workspace=work, flags=fb.FLAG_OVERLAP_PREV, n=N)
            us = time_graph(f, R, max(1, 400 // R), stream)
            b = algorithmic_bytes(M, N, K)
            out.append({"workload": name, "M": M, "N": N, "K": K, "us": round(us, 3),
                        "GB/s": round(b / us / 1e3, 1), "frac": round(b / us / 1e3 / peak, 4),
                        "TFLOP/s": round(2.0 * M * N * K / us / 1e6, 1)})
            print(json.dumps(out[-1]), file=sys.stderr, flush=True)
            if name == "vocab":
                # the output layer with the greedy token choice fused, logits not stored
                tok = torch.empty((M,), dtype=torch.int32, device=dev)
                lg = torch.empty((M,), dtype=torch.float32, device=dev)

                def g(i, x=x, work=work, N=N, tok=tok, lg=lg):
                    wq, ws = layers[i % R]
                    fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws, store_y=False, token=tok, logit=lg,
                                                         workspace=work, flags=fb.FLAG_OVERLAP_PREV, n=N)
                us = time_graph(g, R, max(1, 400 // R), stream)
                b = algorithmic_bytes(M, N, K) - 2 * M * N  # no Y written
                out.append({"workload": "vocab_greedy", "M": M, "N": N, "K": K, "us": round(us, 3),
                            "GB/s": round(b / us / 1e3, 1), "frac": round(b / us / 1e3 / peak, 4)})
                print(json.dumps(out[-1]), file=sys.stderr, flush=True)
        del layers
        torch.cuda.empty_cache()
    out += decode_pass(dev, stream, peak)
    # vocab layer in bf16 (the 16-bit baseline of the output layer)
    cfg = workload("vocab")
    N, K = cfg["N"], cfg["K"]
    wb = [fb.bf16_pack_weights_tiled(synth.weights(N, K, seed=300 + i, device=dev).to(torch.bfloat16))
          for i in range(2)]
    for M in (1, 8):
        x = synth.activations(M, K, seed=4, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        work = fb.make_workspace(fb.bf16_gemm_ref_workspace_size(M, N, K), dev)

        def f(i, x=x, y=y, work=work):
            fb.bf16_gemm_ref(x, wb[i % 2], y=y, workspace=work, flags=fb.FLAG_OVERLAP_PREV, n=N)
        us = time_graph(f, 2, 50, stream)
        b = bf16_bytes(M, N, K)
        out.append({"workload": "vocab_bf16", "M": M, "N": N, "K": K, "us": round(us, 3),
                    "GB/s": round(b / us / 1e3, 1), "frac": round(b / us / 1e3 / peak, 4)})
        print(json.dumps(out[-1]), file=sys.stderr, flush=True)
    if args.out_dir:
        os.makedirs(args.out_dir, exist_ok=True)
        with open(os.path.join(args.out_dir, "bench_configs.json"), "w") as fh:
            json.dump(out, fh, indent=1)


# ---------------------------------------------------------------- reference arm: the CPU oracle
def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = workload(args.workload, args.m)
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    # calibrate seconds per output column, then size each step so that the
    # warm-up and timed steps together stay within about two minutes
    probe = OracleSample(M, N, K, cfg["seed"], ncols=128)
    t0 = time.perf_counter()
    probe.run_once()
    per_col = (time.perf_counter() - t0) / 128
    budget = 120.0 / max(1, args.steps + args.warmup)
    smp = OracleSample(M, N, K, cfg["seed"], ncols=int(max(1, min(N, budget / per_col))))
    for _ in range(args.warmup):
        smp.run_once()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.run_once()
    el = time.perf_counter() - t0
    value = smp.bytes_per_run() * args.steps / el / 1e9
    sample = "each step: " + smp.describe()
    line = {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / max(1, args.steps) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) bf16 activations)",
            "config": {"workload": "%s M=%d N=%d K=%d" % (args.workload, M, N, K), "M": M, "N": N, "K": K},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "kind": "oracle", "cores": smp.threads,
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="square_decode")
    ap.add_argument("--m", type=int, default=None)
    ap.add_argument("--configs", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--out-dir", default=None,
                    help="directory for the clock samples and the --configs table (default: a temporary one)")
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
