"""Benchmark of the GB300 MXFP4 linear hot path: one Flux-12B MLP up-projection training
step (dual-quantize X, W, dY; fwd, dgrad and wgrad block-scaled GEMMs) per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--cpu-baseline-seconds S]

Prints one JSON line (rank 0).  `value` is the step's GEMM work (3 x 2MNK flops) divided
by the device time of the whole step, quantizers included, summed over all ranks' steps;
per-kernel times, the GEMM roofline and the dual-quantizer bandwidth come with it.
Under torchrun each rank runs its own replica of the step on its own GPU (the path has
no exchange step), so scaling is weak.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 GEMM TFLOPS + dual-quant GB/s at Flux-12B shapes; % of roofline"
DEFAULT_WORKLOAD = "flux12b_mlp_up_train_step_4608x12288x3072"
L2_FLUSH_BYTES = 256 << 20       # > 2x the 129 MB L2
HEAD_START_CYCLES = 20_000_000   # ~10 ms of GPU sleep before the first timed step
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25   # dense FP4 / dense bf16 tensor rate (nominal)
NOMINAL_FP8_OVER_BF16 = 4.5 / 2.25    # dense FP8 / dense bf16 tensor rate (nominal)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max_over_ranks(x: float, world: int, device="cpu") -> float:
    """Max of a per-rank float over all ranks of the default process group (the slowest
    rank sets the job's time).  device: "cpu" for gloo, the rank's GPU for NCCL."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(step_flops: int, steps: int, max_total_ms: float, world: int) -> float:
    """Weak scaling: every rank runs `steps` steps of the same workload; the job's
    throughput is all ranks' work over the slowest rank's time."""
    return world * step_flops * steps / (max_total_ms * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "source": "fallback"}


KERNEL_SOURCES = {
    "gemm_mxf4_kernel": ("gemm.cu", "epilogue.cuh", "ptx.cuh", "launch.h"),
    "gemm_mxf4_pair_kernel": ("gemm_pair.cu", "epilogue.cuh", "ptx.cuh", "launch.h"),
    "quantize_kernel": ("quantize.cu", "ptx.cuh", "launch.h"),
    "gemm_fp8_pair_kernel": ("gemm_fp8.cu", "epilogue.cuh", "ptx.cuh", "launch_fp8.h"),
}


def kernel_source_hash(kernel):
    """Hash of the sources a kernel is built from (a profile taken on other sources is
    stale)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mxfp4_block_scaled_quantize_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    ent = t.get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.samples = []
        self.proc = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [s for t, s in self.samples if self.window and self.window[0] - 0.15 <= t <= self.window[1] + 0.15]
        if not rows:
            rows = [s for _, s in self.samples[-3:]]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from mxfp4_block_scaled_quantize_gb300 import abi, workloads
    from mxfp4_block_scaled_quantize_gb300.linear import MXFP4Linear
    import __graft_entry__

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    abi.load()

    wl = workloads.WORKLOADS[args.workload]
    lin = wl.linears[0]
    M, N, K = lin.M, lin.N, lin.K
    t = wl.tensors(0)
    x, w = t["X"].to(dev), t["W"].to(dev)
    dy = t["dY"].to(dev) if lin.train else None
    fp8_bwd = bool(args.fp8_backward) and lin.train
    if args.fp8_backward and args.sr:
        raise SystemExit("--sr is a mode of the MXFP4 backward, not of --fp8-backward")
    layer = MXFP4Linear(M, N, K, train=lin.train, device=dev, backward="fp8" if fp8_bwd else "mxfp4")
    bias = (workloads.normal((N,), 0.02, 977).to(dev) if args.bias else None)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_src = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # Write a buffer larger than L2, then read another one: no input of the step is left
        # in L2, and neither is a dirty line whose write-back would land in the next step.
        flush.zero_()
        flush_src.sum()
    stream = torch.cuda.current_stream(dev)
    n_k = layer.launches_per_step
    names = (["quant_row_XW", "gemm_fwd", "quant_fp8_dY_X_W", "gemm_fp8_dgrad_wgrad"] if fp8_bwd else
             ["quant_dual_XW", "gemm_fwd", "quant_dual_dY", "gemm_dgrad_wgrad"]
             if lin.train else ["quant_row_XW", "gemm_fwd"])

    def sr_seed(k):
        return (0x5EED0000 + k) if args.sr else None

    def step_with_events(evs, k):
        evs[0].record(stream)
        layer.quantize_xw(x, w)
        evs[1].record(stream)
        layer.fwd_gemm(bias=bias)
        evs[2].record(stream)
        if lin.train:
            if fp8_bwd:
                layer.quantize_fp8_bwd(dy)
            else:
                layer.quantize_dy(dy, sr_seed=sr_seed(k))
            evs[3].record(stream)
            if fp8_bwd:
                layer.fp8_bwd_gemms()
            else:
                layer.bwd_gemms()
            evs[4].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()

    for i in range(args.warmup):
        flush_l2()
        layer.step(x, w, dy, bias=bias, sr_seed=sr_seed(i))
    torch.cuda.synchronize()
    if abi.mxfp4_last_device_error() != abi.MXFP4_OK:
        raise RuntimeError("device error word set during warm-up")

    def head_start():
        # Keep the GPU busy (outside every timed interval) while the host queues the first
        # steps, so no step waits on the host's launch calls.
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(HEAD_START_CYCLES)

    sampler = ClockSampler(local_rank)
    if rank == 0:
        sampler.start()
    # Timed region: the K steps, one event pair per step.  Nothing is recorded between a
    # step's kernels, so each kernel's launch overlaps the previous kernel's tail
    # (programmatic dependent launch); the L2 flush between steps is outside the pairs.
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_start = time.time()
    head_start()
    for k in range(args.steps):
        flush_l2()
        step_events[k][0].record(stream)
        layer.step(x, w, dy, bias=bias, sr_seed=sr_seed(k))
        step_events[k][1].record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    barrier()
    # Per-kernel pass (same steps, an event between every two kernels, which serializes
    # their launches): the kernel durations behind the roofline and bandwidth figures.
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    head_start()
    for k in range(args.steps):
        flush_l2()
        step_with_events(events[k], k)
    torch.cuda.synchronize()
    t_end2 = time.time()
    barrier()
    sampler.mark(t_start, t_end2)
    clocks = sampler.stop() if rank == 0 else None
    if abi.mxfp4_last_device_error() != abi.MXFP4_OK:
        raise RuntimeError("device error word set during the timed steps")

    per_kernel = [[ev[i].elapsed_time(ev[i + 1]) for ev in events] for i in range(len(names))]
    step_ms = [ev[0].elapsed_time(ev[1]) for ev in step_events]
    total_ms = reduce_max_over_ranks(sum(step_ms), world, dev)

    # ---- end to end: inputs from pinned host memory, results back to pinned host memory,
    #      through the layer's host-buffer step (copies overlapped with the kernels)
    hx, hw = t["X"].pin_memory(), t["W"].pin_memory()
    hdy = t["dY"].pin_memory() if lin.train else None
    outs = [layer.y] + ([layer.dx, layer.dw] if lin.train else [])
    houts = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    houts += [None] * (3 - len(houts))
    h2d = sum(a.numel() * a.element_size() for a in (hx, hw, hdy) if a is not None)
    d2h = sum(o.numel() * o.element_size() for o in houts if o is not None)
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        layer.step_host(hx, hw, hdy, *houts, bias=bias, sr_seed=sr_seed(0))
    torch.cuda.synchronize()
    e_ms = []
    for _ in range(e2e_steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        layer.step_host(hx, hw, hdy, *houts, bias=bias, sr_seed=sr_seed(0))
        e1.record(stream)
        e1.synchronize()
        e_ms.append(e0.elapsed_time(e1))
    e2e_ms = reduce_max_over_ranks(statistics.mean(e_ms), world, dev)

    if rank != 0:
        return None

    peaks = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * NOMINAL_FP4_OVER_BF16
    gemm_idx = [i for i, n in enumerate(names) if n.startswith("gemm")]
    quant_idx = [i for i, n in enumerate(names) if n.startswith("quant")]
    # algorithmic flops of each GEMM launch: the forward GEMM, and dgrad + wgrad together
    launch_flops = {"gemm_fwd": 2 * M * N * K, "gemm_dgrad_wgrad": 4 * M * N * K,
                    "gemm_fp8_dgrad_wgrad": 4 * M * N * K}
    if fp8_bwd:
        # the FP8 backward GEMM launch dominates; its peak is the FP8 one
        gemm_idx = [names.index("gemm_fp8_dgrad_wgrad")]
        fp4_peak = peaks["bf16_tflops"] * NOMINAL_FP8_OVER_BF16
    gemm_flops = sum(launch_flops[names[i]] for i in gemm_idx) / len(gemm_idx)   # per launch
    gemm_ms = statistics.mean([v for i in gemm_idx for v in per_kernel[i]])      # per launch
    gemm_tflops = gemm_flops / (gemm_ms * 1e-3) / 1e12

    # algorithmic bytes of each quantizer launch (padding excluded): bf16 read once, codes
    # and scales written once
    qbytes = {"quant_dual_XW": (M * K + N * K) * 3.0625, "quant_row_XW": (M * K + N * K) * 2.53125,
              "quant_dual_dY": M * N * 3.0625,
              "quant_fp8_dY_X_W": M * N * (2 + 2) + (M * K + N * K) * (2 + 1)}
    kern = {}
    for i, n in enumerate(names):
        ms = statistics.mean(per_kernel[i])
        ent = {"avg_us": round(ms * 1e3, 2), "min_us": round(min(per_kernel[i]) * 1e3, 2)}
        if n.startswith("gemm"):
            ent["tflops"] = round(launch_flops[n] / (ms * 1e-3) / 1e12, 1)
            ent["frac_of_fp4_peak"] = round(ent["tflops"] / fp4_peak, 4)
        else:
            nbytes = qbytes[n]
            ent["gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
            ent["frac_of_hbm"] = round(ent["gbs"] / peaks["hbm_gbs"], 4)
        kern[n] = ent
    q_bytes = sum(qbytes[names[i]] for i in quant_idx)
    q_ms = sum(statistics.mean(per_kernel[i]) for i in quant_idx)
    quant_gbs = q_bytes / (q_ms * 1e-3) / 1e9

    step_flops = lin.flops_step
    value = whole_job_tflops(step_flops, args.steps, total_ms, world)
    e2e_value = whole_job_tflops(step_flops, 1, e2e_ms, world)
    gemm_kernel = ("gemm_fp8_pair_kernel" if fp8_bwd else
                   "gemm_mxf4_pair_kernel" if M > 128 else "gemm_mxf4_kernel")
    traffic = profiled_traffic(gemm_kernel)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4_e2m1 (e8m0 block scales, fp32 accumulate, bf16 out)" + (
            "; backward fp8_e5m2 (tensorwise scales, fp32 accumulate)" if fp8_bwd else ""),
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, N(0,1e-3) grads)",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                   "step": ("row-quant X,W; fwd" + (" + bias" if args.bias else "") +
                            "; fp8 tensorwise quant dY, X, W; fp8 dgrad; fp8 wgrad") if fp8_bwd else
                           ("dual-quant X,W; fwd" + (" + bias" if args.bias else "") +
                            "; dual-quant dY" + (" (stochastic rounding)" if args.sr else "") +
                            "; dgrad; wgrad") if lin.train
                   else "row-quant X,W; fwd",
                   "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, then "
                         f"{L2_FLUSH_BYTES >> 20} MiB read)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": gemm_kernel,
                     "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp4_peak, 4),
                     "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 {peaks['bf16_tflops']} TFLOP/s x " + (
                         f"{NOMINAL_FP8_OVER_BF16:g} (nominal dense FP8/bf16 ratio)" if fp8_bwd else
                         f"{NOMINAL_FP4_OVER_BF16:g} (nominal dense FP4/bf16 ratio)"),
                     "algorithmic_flops_per_launch": int(gemm_flops)},
        "quant_roofline": {"bound": "hbm", "achieved": round(quant_gbs, 1),
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(quant_gbs / peaks["hbm_gbs"], 4),
                           "algorithmic_bytes_per_step": int(q_bytes), "peak_source": peaks["source"]},
        "kernels": kern,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": n_k * args.steps,
        "kernel_times": "second pass over the same steps with an event between kernels",
        "clocks": clocks,
        "device": torch.cuda.get_device_name(dev),
    }
    return line


# ---------------------------------------------------------------------------------------
# the CPU oracle on a bounded sample (cpu_baseline, and the reference arm)
# ---------------------------------------------------------------------------------------
def oracle_sample(workload_name, seconds, fp8_backward=False, threads=1):
    """Times the oracle on slices of the workload and extrapolates one full step.

    Sample: the oracle's quantizers (dual, or row-only; with fp8_backward, row-only MX for
    X and W plus tensorwise E5M2 of dY, X and W) on 128-row slabs of X, W and dY, and its
    fp64 GEMM on 8-row blocks of output against 512 columns; each part runs for about
    seconds/2 of wall time on `threads` host threads at once (the oracle's C functions
    release the GIL, so the threads run in parallel; each thread takes its own slabs and
    blocks).  Step time = wall time per quantized element x all quantized elements + wall
    time per MAC x all MACs of the step's GEMMs.
    """
    import concurrent.futures
    import numpy as np

    import oracle
    from mxfp4_block_scaled_quantize_gb300 import workloads

    wl = workloads.WORKLOADS[workload_name]
    lin = wl.linears[0]
    M, N, K = lin.M, lin.N, lin.K
    t = wl.tensors(0)
    bits = {k: workloads.bf16_bits(v) for k, v in t.items()}
    fp8 = fp8_backward and lin.train
    quant = oracle.quantize_dual if (lin.train and not fp8) else oracle.quantize_row
    threads = max(1, int(threads))

    def slab(k, w):
        rows = bits[k].shape[0]
        r0 = (128 * w) % max(1, rows - 127)
        return np.ascontiguousarray(bits[k][r0:r0 + 128])

    def quant_worker(w):
        slabs = {k: slab(k, w) for k in bits}
        elems = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds / 2:
            for k, sl in slabs.items():
                if fp8:   # row-only MX for X and W, tensorwise E5M2 for all three
                    if k != "dY":
                        quant(sl)
                    oracle.fp8_quantize_tw(sl, row=(k == "dY"), col=True)
                else:
                    quant(sl)
                elems += sl.size
        return elems

    wq, ws = oracle.quantize_row(np.ascontiguousarray(bits["W"][:512]))
    b = oracle.dequantize(wq, ws)

    def gemm_worker(w):
        xq, xs = oracle.quantize_row(slab("X", w)[:8])
        a = oracle.dequantize(xq, xs)
        macs = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds / 2:
            oracle.gemm_dequantized(a, b, want_abs=False)
            macs += a.shape[0] * b.shape[0] * a.shape[1]
        return macs

    with concurrent.futures.ThreadPoolExecutor(threads) as ex:
        t0 = time.perf_counter()
        q_elems = sum(ex.map(quant_worker, range(threads)))
        q_wall = time.perf_counter() - t0
        t0 = time.perf_counter()
        g_macs = sum(ex.map(gemm_worker, range(threads)))
        g_wall = time.perf_counter() - t0
    total_q = M * K + N * K + (M * N if lin.train else 0)
    if fp8:
        total_q = 2 * (M * K + N * K) + M * N
    total_macs = M * N * K * (3 if lin.train else 1)
    step_s = q_wall / q_elems * total_q + g_wall / g_macs * total_macs
    kind = "row-only MX + tensorwise E5M2" if fp8 else "dual" if lin.train else "row-only"
    return {
        "step_seconds": step_s,
        "value": lin.flops_step / step_s / 1e12,
        "sample": (f"oracle {kind} quantizer on 128-row slabs of X, W{', dY' if lin.train else ''} "
                   f"({int(q_elems)} elements) and fp64 GEMM on 8x512 output blocks at "
                   f"K={oracle.padded(K)} ({int(g_macs)} MACs), on {threads} host thread(s); one "
                   f"full step extrapolated per element / per MAC of wall time"),
        "cores": threads,
        "kind": "oracle",
    }


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle.build
    oracle.build.build()
    per = max(2.0, args.cpu_baseline_seconds / max(1, args.steps))
    cores = host_cores()
    for _ in range(args.warmup):
        oracle_sample(args.workload, 0.2, args.fp8_backward, cores)
    vals = [oracle_sample(args.workload, per, args.fp8_backward, cores) for _ in range(args.steps)]
    step_s = statistics.mean(v["step_seconds"] for v in vals)
    value = vals[0]["value"] if len(vals) == 1 else statistics.mean(v["value"] for v in vals)
    from mxfp4_block_scaled_quantize_gb300 import workloads
    lin = workloads.WORKLOADS[args.workload].linears[0]
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "M": lin.M, "N": lin.N, "K": lin.K,
                   "parallelism": "host cores of rank 0"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": vals[0]["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--sr", action="store_true",
                    help="dY is quantized with stochastic rounding (the gradient quantizer's "
                         "`use_sr`), a new Philox seed every step")
    ap.add_argument("--fp8-backward", action="store_true",
                    help="the hybrid backward: dY, X, W quantized tensorwise to FP8 E5M2 and "
                         "dgrad / wgrad as FP8 GEMMs (the layer's mxfp4_backward_precision 'fp8')")
    ap.add_argument("--bias", action="store_true",
                    help="the forward adds the layer's bf16 bias inside the GEMM (the "
                         "`output + bias` that follows the GEMM in the layer's forward)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, world, local_rank = dist_env()

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        # the oracle on every host core, and on one (half of the time budget each)
        cores = host_cores()
        base = oracle_sample(args.workload, args.cpu_baseline_seconds / 2, args.fp8_backward, cores)
        one = oracle_sample(args.workload, args.cpu_baseline_seconds / 2, args.fp8_backward, 1)
        line["cpu_baseline"] = {"value": base["value"], "unit": "TFLOP/s", "cores": base["cores"],
                                "kind": "oracle", "sample": base["sample"],
                                "single_core_value": one["value"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
