"""Benchmark of the GB300 MXFP4 linear hot path at Flux-12B shapes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--cpu-baseline-seconds S] [--no-extras]
                    [--sr | --fp8-backward] [--recipes] [--bias] [--extra NAME]

One step is one training step of every MXFP4 linear of the workload, in the order of a
block's training step: each linear's forward (X and W quantized in one launch, then
Y = X . W^T), then each linear's backward in reverse order (dY quantized, then dgrad and
wgrad in one GEMM launch).  The default workload is Flux-12B's single-stream block:
linear1 X[4608,3072] . W1[21504,3072]^T and linear2 H[4608,15360] . W2[3072,15360]^T,
3.131 TFLOP per step.

Prints one JSON line (rank 0).  `value` is the step's GEMM work divided by the device time
of the whole step, quantizers included, summed over all ranks' steps.  With it: per-kernel
medians and means, the GEMM roofline, the quantizer bandwidth, the same step replayed as a
CUDA graph, an end-to-end step from pinned host buffers through the library's host-step
entry point, and (N = 1, `extras`) the Flux QKV forward with row-only quantization, the
quantizer bandwidth sweep, the forward GEMM that writes its output's MXFP4 blobs and the QKV
gradient's quantization with the norm + RoPE backward in its read (`--extra NAME` runs one
of these alone and prints only its line).  Under torchrun each rank runs its own replica of the step on
its own GPU (the path has no exchange step), so scaling is weak.  `--impl reference`
times the CPU oracle on a bounded sample of the same workload instead.
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
DEFAULT_WORKLOAD = "flux12b_single_block_linears_train"
L2_FLUSH_BYTES = 256 << 20       # > 2x the 129 MB L2
HEAD_START_CYCLES = 20_000_000   # ~10 ms of GPU sleep before the first timed step
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25   # dense FP4 / dense bf16 tensor rate (nominal)
NOMINAL_FP8_OVER_BF16 = 4.5 / 2.25    # dense FP8 / dense bf16 tensor rate (nominal)
SPEC_FP4_TFLOPS = 15000.0        # dense FP4 per GB300 GPU (GB300 NVL72: 1.08 EF / 72)
SPEC_HBM_GBS = 8000.0            # HBM3e, nominal (~8 TB/s)
MMA_MXF4_ISSUE_TFLOPS = 9690.0   # back-to-back kind::mxf4 M256 N256 K64 on all SMs (measured)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
RHT_SIGNS = 0xA5C3                       # sign mask of the column-blob transform (--recipes)
DUAL_BYTES = 2 + 2 * (0.5 + 1 / 32)      # per element: bf16 read, two blobs written
ROW_BYTES = 2 + 0.5 + 1 / 32


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
    "gemm_mxf4_pair_kernel": ("gemm_pair.cu", "epilogue.cuh", "mx_encode.cuh", "ptx.cuh", "launch.h"),
    "quantize_kernel": ("quantize.cu", "mx_encode.cuh", "ptx.cuh", "launch.h"),
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


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    ent = t.get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel) or ent.get("workload") != workload:
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
# algorithmic work of each stage of a step
# ---------------------------------------------------------------------------------------
def op_work(name, lin):
    """(flops, bytes) of one stage `name` of linear `lin`: GEMM stages count 2MNK flops per
    GEMM with the logical K; quantizer stages count the bf16 read plus the codes and scale
    bytes written, padding excluded."""
    M, N, K = lin.M, lin.N, lin.K
    kind = name.split(".", 1)[1]
    return {
        "quant_dual_XW": (0, (M * K + N * K) * DUAL_BYTES),
        "quant_row_XW": (0, (M * K + N * K) * ROW_BYTES),
        "quant_dual_dY": (0, M * N * DUAL_BYTES),
        "quant_fp8_dY_X_W": (0, M * N * (2 + 2) + (M * K + N * K) * (2 + 1)),
        "gemm_fwd": (2 * M * N * K, 0),
        "gemm_dgrad_wgrad": (4 * M * N * K, 0),
        "gemm_fp8_dgrad_wgrad": (4 * M * N * K, 0),
    }[kind]


def summarize(ms_list):
    return {"median_us": round(statistics.median(ms_list) * 1e3, 2),
            "mean_us": round(statistics.mean(ms_list) * 1e3, 2),
            "min_us": round(min(ms_list) * 1e3, 2)}


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from mxfp4_block_scaled_quantize_gb300 import abi, workloads
    from mxfp4_block_scaled_quantize_gb300.linear import MXFP4Block
    import __graft_entry__

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    abi.load()

    wl = workloads.WORKLOADS[args.workload]
    lins = wl.linears
    train = lins[0].train
    fp8_bwd = bool(args.fp8_backward) and train
    if args.fp8_backward and args.sr:
        raise SystemExit("--sr is a mode of the MXFP4 backward, not of --fp8-backward")
    host_t = [wl.tensors(i) for i in range(len(lins))]
    inputs = [{k: v.to(dev) for k, v in t.items()} for t in host_t]
    if args.recipes and fp8_bwd:
        raise SystemExit("--recipes is a mode of the MXFP4 backward")
    block = MXFP4Block([(l.name, l.M, l.N, l.K) for l in lins], train=train, device=dev,
                       backward="fp8" if fp8_bwd else "mxfp4", weight_2d=args.recipes,
                       rht_signs=RHT_SIGNS if (args.recipes and train) else None)
    bias = ([workloads.normal((l.N,), 0.02, 977 + i).to(dev) for i, l in enumerate(lins)]
            if args.bias else None)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_src = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    lin_of = {l.name: l for l in lins}

    def flush_l2():
        # Write a buffer larger than L2, then read another one: no input of the step is left
        # in L2, and neither is a dirty line whose write-back would land in the next step.
        flush.zero_()
        flush_src.sum()
    stream = torch.cuda.current_stream(dev)

    def sr_seed(k):
        return (0x5EED0000 + k) if args.sr else None

    def ops(k):
        return block.ops(inputs, bias, sr_seed(k))
    names = [n for n, _, _ in ops(0)]
    launches_per_step = sum(n for _, _, n in ops(0))

    def run_step(k):
        for _, fn, _ in ops(k):
            fn()

    def barrier():
        if world > 1:
            dist.barrier()

    def head_start():
        # Keep the GPU busy (outside every timed interval) while the host queues the first
        # steps, so no step waits on the host's launch calls.
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(HEAD_START_CYCLES)

    for i in range(args.warmup):
        flush_l2()
        run_step(i)
    torch.cuda.synchronize()
    if abi.mxfp4_last_device_error() != abi.MXFP4_OK:
        raise RuntimeError("device error word set during warm-up")

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
        run_step(k)
        step_events[k][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    # Per-kernel pass (same steps, an event between every two stages, which serializes
    # their launches): the kernel durations behind the roofline and bandwidth figures.
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    head_start()
    for k in range(args.steps):
        flush_l2()
        evs = events[k]
        evs[0].record(stream)
        for i, (_, fn, _) in enumerate(ops(k)):
            fn()
            evs[i + 1].record(stream)
    torch.cuda.synchronize()
    # CUDA-graph pass: one step captured once and replayed, which takes the host's launch
    # calls out of the picture (the same kernels and arguments; with --sr every replay uses
    # the first step's seed).
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            run_step(0)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            run_step(0)
        torch.cuda.synchronize()
        for _ in range(2):
            flush_l2()
            g.replay()
        gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        head_start()
        for k in range(args.steps):
            flush_l2()
            gev[k][0].record(stream)
            g.replay()
            gev[k][1].record(stream)
        torch.cuda.synchronize()
        gms = [a.elapsed_time(b) for a, b in gev]
        graph = {"ms_per_step_median": round(statistics.median(gms), 4),
                 "ms_per_step_mean": round(statistics.mean(gms), 4)}
    except Exception as e:   # reported, not hidden: the eager numbers stand on their own
        graph = {"error": f"{type(e).__name__}: {e}"[:200]}
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

    # ---- end to end: inputs from pinned host memory, results back to pinned host memory
    plain = not (fp8_bwd or args.sr or args.bias or args.recipes)
    hin = [{k: v.pin_memory() for k, v in t.items()} for t in host_t]
    houts = []
    for L in block.layers:
        outs = [L.y] + ([L.dx, L.dw] if train else [])
        houts.append([torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs])
    h2d = sum(v.numel() * v.element_size() for t in hin for v in t.values())
    d2h = sum(o.numel() * o.element_size() for os_ in houts for o in os_)

    def e2e_step():
        if plain:
            # the library's own host-buffer step (mxfp4_linear_step_host, one C-ABI call)
            block.step_host(hin, houts)
        else:
            # the options are not in the host-step entry point: per layer, torch copies on
            # copy streams around the layer's C-ABI calls
            for L, t, o, i in zip(block.layers, hin, houts, range(len(lins))):
                o3 = list(o) + [None] * (3 - len(o))
                L.step_host(t["X"], t["W"], t.get("dY"), *o3, bias=bias[i] if bias else None,
                            sr_seed=sr_seed(0))

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for _ in range(e2e_steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e_ms.append(e0.elapsed_time(e1))
    e2e_latency_ms = reduce_max_over_ranks(statistics.median(e_ms), world, dev)
    e2e_ms = e2e_latency_ms
    if plain:
        # A loop of steps through the pipelined host step: each step's copies in, kernels and
        # copies out are all in the timed region, and consecutive steps overlap one step's
        # copies out with the next step's copies in and kernels.
        for _ in range(2):
            block.step_host_pipelined(hin, houts)
        block.host_wait()
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(e2e_steps):
            block.step_host_pipelined(hin, houts)
        block.host_wait()
        p1.record(stream)
        p1.synchronize()
        e2e_ms = reduce_max_over_ranks(p0.elapsed_time(p1) / e2e_steps, world, dev)
    if abi.mxfp4_last_device_error() != abi.MXFP4_OK:
        raise RuntimeError("device error word set during the end-to-end steps")

    extras = run_extras(args, dev, flush_l2, head_start) if (rank == 0 and world == 1 and args.extras) else None

    if rank != 0:
        return None

    peaks = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * NOMINAL_FP4_OVER_BF16
    gemm_peak = peaks["bf16_tflops"] * (NOMINAL_FP8_OVER_BF16 if fp8_bwd else NOMINAL_FP4_OVER_BF16)
    kern = {}
    gemm_flops = gemm_ms = q_bytes = q_ms = 0.0
    n_gemm = 0
    for i, n in enumerate(names):
        flops, nbytes = op_work(n, lin_of[n.split(".")[0]])
        ent = summarize(per_kernel[i])
        ms = statistics.mean(per_kernel[i])
        if flops:
            ent["tflops"] = round(flops / (ms * 1e-3) / 1e12, 1)
            peak = gemm_peak if "fp8" in n else fp4_peak
            ent["frac_of_peak"] = round(ent["tflops"] / peak, 4)
            if "fp8" in n or not fp8_bwd:
                gemm_flops += flops
                gemm_ms += ms
                n_gemm += 1
        else:
            ent["gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
            ent["frac_of_hbm"] = round(ent["gbs"] / peaks["hbm_gbs"], 4)
            q_bytes += nbytes
            q_ms += ms
        kern[n] = ent
    gemm_tflops = gemm_flops / (gemm_ms * 1e-3) / 1e12
    quant_gbs = q_bytes / (q_ms * 1e-3) / 1e9

    step_flops = sum(l.flops_step for l in lins)
    value = whole_job_tflops(step_flops, args.steps, total_ms, world)
    e2e_value = whole_job_tflops(step_flops, 1, e2e_ms, world)
    gemm_kernel = ("gemm_fp8_pair_kernel" if fp8_bwd else
                   "gemm_mxf4_pair_kernel" if min(l.M for l in lins) > 128 else "gemm_mxf4_kernel")
    traffic = profiled_traffic(gemm_kernel, args.workload)
    mode = ("; backward fp8 (tensorwise E5M2 of dY, X, W; fp8 dgrad + wgrad)" if fp8_bwd else
            "; dY stochastically rounded" if args.sr else "") + ("; bias fused" if args.bias else "") + (
            f"; recipes: W in 32x32 blocks, col blobs of X and dY Hadamard-transformed (signs {RHT_SIGNS:#06x})"
            if args.recipes else "")

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "ms_per_step_median": round(statistics.median(step_ms), 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4_e2m1 (e8m0 block scales, fp32 accumulate, bf16 out)" + (
            "; backward fp8_e5m2 (tensorwise scales, fp32 accumulate)" if fp8_bwd else ""),
        "data": "synthetic (seeded N(0,1) / GELU-like activations, N(0,0.02) weights, N(0,1e-3) grads)",
        "config": {"workload": args.workload,
                   "linears": [{"name": l.name, "M": l.M, "N": l.N, "K": l.K} for l in lins],
                   "gemm_tflop_per_step": round(step_flops / 1e12, 4),
                   "step": ("forwards in order (quant X+W, fwd GEMM), backwards in reverse order "
                            "(quant dY, dgrad+wgrad GEMM)" if train else "quant X+W (row-only), fwd GEMM") + mode,
                   "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, then "
                         f"{L2_FLUSH_BYTES >> 20} MiB read)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": gemm_kernel,
                     "achieved": round(gemm_tflops, 1), "peak": round(gemm_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / gemm_peak, 4),
                     "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 {peaks['bf16_tflops']} TFLOP/s x " + (
                         f"{NOMINAL_FP8_OVER_BF16:g} (nominal dense FP8/bf16 ratio)" if fp8_bwd else
                         f"{NOMINAL_FP4_OVER_BF16:g} (nominal dense FP4/bf16 ratio)"),
                     "frac_of_spec_15pf": None if fp8_bwd else round(gemm_tflops / SPEC_FP4_TFLOPS, 4),
                     "frac_of_mxf4_issue_ceiling": None if fp8_bwd else round(gemm_tflops / MMA_MXF4_ISSUE_TFLOPS, 4),
                     "launches_per_step": n_gemm,
                     "algorithmic_flops_per_launch": int(gemm_flops / max(1, n_gemm))},
        "quant_roofline": {"bound": "hbm", "achieved": round(quant_gbs, 1),
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(quant_gbs / peaks["hbm_gbs"], 4),
                           "frac_of_spec_8tbs": round(quant_gbs / SPEC_HBM_GBS, 4),
                           "algorithmic_bytes_per_step": int(q_bytes), "peak_source": peaks["source"]},
        "kernels": kern,
        "graph": graph,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "single_step_latency_ms": round(e2e_latency_ms, 4),
                "path": ("mxfp4_linear_step_host_pipelined (one C-ABI call per step, %d steps in a loop, "
                         "consecutive steps overlapped; pinned host buffers)" % e2e_steps) if plain
                        else "per layer: torch copies on copy streams + the layer's C-ABI calls"},
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_note": "library kernels in the timed step pass (L2 flushes are torch's)",
        "kernel_times": "second pass over the same steps with an event between stages",
        "extras": extras,
        "clocks": clocks,
        "device": torch.cuda.get_device_name(dev),
    }
    return line


EXTRAS = ("qkv_fwd", "quant_sweep", "fwd_gemm_with_output_blobs", "qkv_bwd_norm_rope")


def run_extras(args, dev, flush_l2, head_start, only=None):
    """Lines for the other Flux configs, timed the same way: the QKV projection forward with
    row-only quantization (X[4608,3072], W[9216,3072]), the quantizer bandwidth sweep
    (dual quantization of M x K bf16 tensors for every M in {4608, 18432, 4600} and K in
    {3072, 12288, 15360}; the largest, 18432 x 15360, moves 867 MB), the forward GEMM that
    quantizes its own output against the GEMM plus a quantizer launch, and the QKV
    gradient's quantization with the norm + RoPE backward in its staging read.  `only`
    names one of them (`EXTRAS`) to run it alone."""
    import torch

    from mxfp4_block_scaled_quantize_gb300 import abi

    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    n = max(5, min(args.steps, 50))
    ctx = (dev, stream, flush_l2, head_start, peaks, n)
    parts = {"qkv_fwd": _extra_qkv_fwd, "quant_sweep": _extra_quant_sweep,
             "fwd_gemm_with_output_blobs": _extra_fwd_gemm_output_blobs,
             "qkv_bwd_norm_rope": _extra_qkv_bwd_norm_rope}
    out = {}
    for name in EXTRAS:
        if only is None or only == name:
            out.update(parts[name](*ctx))
    if abi.mxfp4_last_device_error() != abi.MXFP4_OK:
        raise RuntimeError("device error word set during the extra lines")
    return out


def _extra_qkv_fwd(dev, stream, flush_l2, head_start, peaks, n):
    import torch

    from mxfp4_block_scaled_quantize_gb300 import workloads
    from mxfp4_block_scaled_quantize_gb300.linear import MXFP4Block

    out = {}
    # QKV forward (row-only X, W, then the forward GEMM)
    wl = workloads.FLUX_QKV_FWD
    lin = wl.linears[0]
    t = {k: v.to(dev) for k, v in wl.tensors(0).items()}
    blk = MXFP4Block([(lin.name, lin.M, lin.N, lin.K)], train=False, device=dev)
    ops = blk.ops([t])
    for _ in range(3):
        for _, fn, _ in ops:
            fn()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(n)]
    head_start()
    for k in range(n):
        flush_l2()
        evs[k][0].record(stream)
        for i, (_, fn, _) in enumerate(ops):
            fn()
            evs[k][i + 1].record(stream)
    torch.cuda.synchronize()
    q_ms = [e[0].elapsed_time(e[1]) for e in evs]
    g_ms = [e[1].elapsed_time(e[2]) for e in evs]
    qb = (lin.M * lin.K + lin.N * lin.K) * ROW_BYTES
    out[wl.name] = {
        "quant_row_XW": dict(summarize(q_ms), gbs=round(qb / (statistics.mean(q_ms) * 1e-3) / 1e9, 1),
                             frac_of_hbm=round(qb / (statistics.mean(q_ms) * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)),
        "gemm_fwd": dict(summarize(g_ms), tflops=round(lin.flops_fwd / (statistics.mean(g_ms) * 1e-3) / 1e12, 1)),
        "step_tflops": round(lin.flops_fwd / ((statistics.mean(q_ms) + statistics.mean(g_ms)) * 1e-3) / 1e12, 1),
    }
    del blk, t
    return out


def _extra_quant_sweep(dev, stream, flush_l2, head_start, peaks, n):
    import torch

    from mxfp4_block_scaled_quantize_gb300 import abi, workloads

    # quantizer sweep: dual quantization, inputs drawn on the device from a seed (the values
    # do not change the work; the bit-exact sweep lives in the parity tests)
    sweep = {}
    gen = torch.Generator(device=dev)
    for M in workloads.SWEEP_M:
        for K in workloads.SWEEP_K:
            gen.manual_seed(M * 100003 + K)
            x = torch.randn((M, K), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
            outs = abi.quantize(x, dual=True)
            ms = []
            for k in range(n + 3):
                flush_l2()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                abi.mxfp4_quantize_dual(x, M, K, x.stride(0), *outs, abi.MXFP4_SCALE_TC)
                e1.record(stream)
                if k >= 3:
                    ms.append((e0, e1))
            torch.cuda.synchronize()
            ms = [a.elapsed_time(b) for a, b in ms]
            nbytes = M * K * DUAL_BYTES
            gbs = nbytes / (statistics.median(ms) * 1e-3) / 1e9
            sweep[f"{M}x{K}"] = {"median_us": round(statistics.median(ms) * 1e3, 2), "mb": round(nbytes / 1e6, 1),
                                 "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                                 "frac_of_spec_8tbs": round(gbs / SPEC_HBM_GBS, 4)}
            del x, outs
    return {"quant_dual_sweep": sweep}


def _extra_fwd_gemm_output_blobs(dev, stream, flush_l2, head_start, peaks, n):
    import torch

    from mxfp4_block_scaled_quantize_gb300 import abi, workloads

    # The forward GEMM whose epilogue writes its output's dual MXFP4 blobs (what the next
    # layer's forward would quantize), against the GEMM followed by the dual quantizer over
    # its output: the single-stream block's linear1, 4608 x 21504 x 3072.
    wl = workloads.FLUX_SINGLE_BLOCK
    lin = wl.linears[0]
    t = wl.tensors(0)
    aq, a_s = abi.quantize(t["X"].to(dev), dual=False)
    bq, b_s = abi.quantize(t["W"].to(dev), dual=False)
    del t
    c = torch.empty((lin.M, lin.N), dtype=torch.bfloat16, device=dev)
    rq, rs = abi.alloc_blob(lin.M, lin.N, device=dev)
    cq, cs = abi.alloc_blob(lin.N, lin.M, device=dev)
    args_g = (aq, a_s, bq, b_s, lin.M, lin.N, lin.K)

    def fused():
        abi.mxfp4_gemm_quantize(*args_g, None, c, lin.N, rq, rs, cq, cs)

    def unfused():
        abi.mxfp4_gemm(*args_g, c, lin.N, abi.MXFP4_OUT_BF16)
        abi.mxfp4_quantize_dual(c, lin.M, lin.N, lin.N, rq, rs, cq, cs, abi.MXFP4_SCALE_TC)

    def fused_row():
        abi.mxfp4_gemm_quantize(*args_g, None, c, lin.N, rq, rs, None, None)

    def plain():
        abi.mxfp4_gemm(*args_g, c, lin.N, abi.MXFP4_OUT_BF16)
    res = {}
    for name, fn in (("gemm_only", plain), ("gemm_then_quantize", unfused), ("gemm_quantize_fused", fused),
                     ("gemm_quantize_fused_row_only", fused_row)):
        for _ in range(3):
            fn()
        ms = []
        for _ in range(n):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ms.append((e0, e1))
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in ms]
        res[name] = dict(summarize(ms), tflops=round(lin.flops_fwd / (statistics.median(ms) * 1e-3) / 1e12, 1))
    res["shape"] = f"{lin.M}x{lin.N}x{lin.K}"
    del aq, a_s, bq, b_s, c, rq, rs, cq, cs
    return {"fwd_gemm_with_output_blobs": res}


def _extra_qkv_bwd_norm_rope(dev, stream, flush_l2, head_start, peaks, n):
    import torch

    from mxfp4_block_scaled_quantize_gb300 import abi

    # The QKV projection's gradient quantization with the QK RMSNorm + interleaved RoPE
    # backward in the staging read (the pages' QKV packer prologue): Flux QKV, 4608 tokens,
    # 24 heads of 128 (d(mixed_qkv) [4608, 9216]), against the plain dual quantizer over a
    # d(mixed_qkv) already in HBM.
    M, H = 4608, 24
    K = 3 * H * 128
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    g = (torch.randn((M, K), generator=gen, device=dev) * 1e-3).to(torch.bfloat16)
    x = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
    rstd = torch.rand((M, H, 2), generator=gen, device=dev) + 0.5
    wq = torch.rand((128,), generator=gen, device=dev) + 0.5
    wk = torch.rand((128,), generator=gen, device=dev) + 0.5
    theta = (torch.rand((M, 64), generator=gen, device=dev) - 0.5) * 6.283
    cos_t, sin_t = torch.cos(theta).contiguous(), torch.sin(theta).contiguous()
    rq, rs = abi.alloc_blob(M, K, device=dev)
    cq, cs = abi.alloc_blob(K, M, device=dev)

    def prolog():
        abi.mxfp4_quantize_dual_qk_norm_rope_bwd(g, x, M, H, rstd, wq, wk, cos_t, sin_t, rq, rs, cq, cs)

    def plain_dual():
        abi.mxfp4_quantize_dual(g, M, K, K, rq, rs, cq, cs, abi.MXFP4_SCALE_TC)
    res = {}
    for name, fn in (("fused_norm_rope_bwd_quantize", prolog), ("plain_dual_quantize", plain_dual)):
        for _ in range(3):
            fn()
        ms = []
        for _ in range(n):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ms.append((e0, e1))
        torch.cuda.synchronize()
        res[name] = summarize([a.elapsed_time(b) for a, b in ms])
    # algorithmic bytes of the fused kernel: g read, x read for q and k, both blobs written
    nb = M * K * (2 + 2 * 2 / 3 + 2 * (0.5 + 1 / 32)) + M * 64 * 8 + M * H * 8
    gbs = nb / (res["fused_norm_rope_bwd_quantize"]["median_us"] * 1e-6) / 1e9
    res["fused_gbs"] = round(gbs, 1)
    res["fused_frac_of_hbm"] = round(gbs / peaks["hbm_gbs"], 4)
    res["shape"] = f"d(mixed_qkv) {M}x{K}, {H} heads of 128"
    del g, x, rstd, wq, wk, cos_t, sin_t, rq, rs, cq, cs
    return {"qkv_bwd_quantize_with_norm_rope_prologue": res}


def run_extra_alone(args):
    """One extra line alone (`--extra NAME`), on the first GPU: what a profiler capture of
    one of those kernels runs, without the step and the CPU baseline around it."""
    import torch

    from mxfp4_block_scaled_quantize_gb300 import abi
    import __graft_entry__

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    __graft_entry__.build()
    abi.load()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_src = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        flush_src.sum()

    def head_start():
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(HEAD_START_CYCLES)
    res = run_extras(args, dev, flush_l2, head_start, only=args.extra)
    return {"extra": args.extra, "n_gpus": 1, "steps": max(5, min(args.steps, 50)),
            "device": torch.cuda.get_device_name(dev), "result": res}


# ---------------------------------------------------------------------------------------
# the CPU oracle on a bounded sample (cpu_baseline, and the reference arm)
# ---------------------------------------------------------------------------------------
_SAMPLE_BITS = {}


def _sample_bits(workload_name):
    """The first 512 rows of every tensor of the workload as bf16 bits (drawn once)."""
    if workload_name not in _SAMPLE_BITS:
        from mxfp4_block_scaled_quantize_gb300 import workloads
        wl = workloads.WORKLOADS[workload_name]
        _SAMPLE_BITS[workload_name] = [
            {k: workloads.bf16_bits(v[:512]) for k, v in wl.tensors(i).items()}
            for i in range(len(wl.linears))]
    return _SAMPLE_BITS[workload_name]


def oracle_sample(workload_name, seconds, fp8_backward=False, threads=1):
    """Times the oracle on slices of the workload and extrapolates one full step.

    Sample: the oracle's quantizers (dual, or row-only; with fp8_backward, row-only MX for
    X and W plus tensorwise E5M2 of dY, X and W) on 128-row slabs of each linear's X, W and
    dY, and its fp64 GEMM on 8-row blocks of output against 512 columns; each part runs for
    about seconds/2 of wall time on `threads` host threads at once (the oracle's C functions
    release the GIL, so the threads run in parallel; each thread takes its own slabs and
    blocks).  Step time = wall time per quantized element x all quantized elements + wall
    time per MAC x all MACs of the step's GEMMs, summed over the linears.
    """
    import concurrent.futures
    import numpy as np

    import oracle
    from mxfp4_block_scaled_quantize_gb300 import workloads

    wl = workloads.WORKLOADS[workload_name]
    lins = wl.linears
    train = lins[0].train
    fp8 = fp8_backward and train
    quant = oracle.quantize_dual if (train and not fp8) else oracle.quantize_row
    threads = max(1, int(threads))
    bits = _sample_bits(workload_name)

    def slab(li, k, w):
        b = bits[li][k]
        rows = b.shape[0]
        r0 = (128 * w) % max(1, rows - 127)
        return np.ascontiguousarray(b[r0:r0 + 128])

    per_elem_bytes = ROW_BYTES if quant is oracle.quantize_row else DUAL_BYTES

    def quant_worker(w):
        slabs = [(k, slab(li, k, w)) for li in range(len(lins)) for k in bits[li]]
        elems = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds / 2:
            for k, sl in slabs:
                if fp8:   # row-only MX for X and W, tensorwise E5M2 for all three
                    if k != "dY":
                        quant(sl)
                    oracle.fp8_quantize_tw(sl, row=(k == "dY"), col=True)
                else:
                    quant(sl)
                elems += sl.size
        return elems

    wq, ws = oracle.quantize_row(bits[0]["W"])
    b = oracle.dequantize(wq, ws)
    kp = b.shape[1]

    def gemm_worker(w):
        xq, xs = oracle.quantize_row(slab(0, "X", w)[:8])
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
    total_q = total_macs = 0
    for l in lins:
        if fp8:
            total_q += 2 * (l.M * l.K + l.N * l.K) + l.M * l.N
        else:
            total_q += l.M * l.K + l.N * l.K + (l.M * l.N if train else 0)
        total_macs += l.M * l.N * l.K * (3 if train else 1)
    step_s = q_wall / q_elems * total_q + g_wall / g_macs * total_macs
    kind = "row-only MX + tensorwise E5M2" if fp8 else "dual" if train else "row-only"
    return {
        "step_seconds": step_s,
        "value": sum(l.flops_step for l in lins) / step_s / 1e12,
        "quant_gbs": None if fp8 else q_elems * per_elem_bytes / q_wall / 1e9,
        "gemm_gflops": 2 * g_macs / g_wall / 1e9,
        "sample": (f"oracle {kind} quantizer on 128-row slabs of every linear's X, W"
                   f"{', dY' if train else ''} ({int(q_elems)} elements) and fp64 GEMM on 8x512 "
                   f"output blocks at K={kp} ({int(g_macs)} MACs), on {threads} host thread(s); "
                   f"one full step extrapolated per element / per MAC of wall time"),
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
    lins = workloads.WORKLOADS[args.workload].linears
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
        "config": {"workload": args.workload,
                   "linears": [{"name": l.name, "M": l.M, "N": l.N, "K": l.K} for l in lins],
                   "parallelism": "host cores of rank 0"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": vals[0]["sample"],
                         "quant_gbs": vals[0]["quant_gbs"], "gemm_gflops": vals[0]["gemm_gflops"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the QKV-forward and quantizer-sweep lines")
    ap.add_argument("--extra", choices=EXTRAS, default=None,
                    help="run only this extra line (one GPU, no step, no CPU baseline)")
    ap.add_argument("--sr", action="store_true",
                    help="dY is quantized with stochastic rounding (the gradient quantizer's "
                         "`use_sr`), a new Philox seed every step")
    ap.add_argument("--fp8-backward", action="store_true",
                    help="the hybrid backward: dY, X, W quantized tensorwise to FP8 E5M2 and "
                         "dgrad / wgrad as FP8 GEMMs (the layer's mxfp4_backward_precision 'fp8')")
    ap.add_argument("--recipes", action="store_true",
                    help="the pages' quantization recipes: W with one scale per 32x32 block in both "
                         "packings, the col blobs of X and dY Hadamard-transformed (with --sr: dY "
                         "stochastically rounded after the transform, the gradient recipe with use_sr)")
    ap.add_argument("--bias", action="store_true",
                    help="the forward adds the layer's bf16 bias inside the GEMM (the "
                         "`output + bias` that follows the GEMM in the layer's forward)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, world, local_rank = dist_env()

    if args.extra is not None:
        if args.impl != "ours" or world > 1:
            raise SystemExit("--extra runs our arm on one GPU")
        print(json.dumps(run_extra_alone(args)), flush=True)
        return

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
                                "quant_gbs": base["quant_gbs"], "gemm_gflops": base["gemm_gflops"],
                                "single_core_value": one["value"],
                                "single_core_quant_gbs": one["quant_gbs"],
                                "single_core_gemm_gflops": one["gemm_gflops"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
