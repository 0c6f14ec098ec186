#!/usr/bin/env python3
"""Benchmark of the W4A16 weight-streaming GEMM on GB300 (one JSON line on stdout).

Step = one pass of the hot path over one batch: the single-stream decode GEMV workload, M = 1
activation row through two matrices (K x N = 5120 x 5120 and 17408 x 5120, group 128), each
y = x . dequant(W) through the C ABI (w4a16_gemm). The metric is the effective weight-stream
rate, weight bytes (0.5 B per weight + fp16 scales) / step time, beside TFLOP/s.

Timing: W untimed warm-up steps; the K timed steps are one CUDA-graph replay bracketed by a
barrier and torch.cuda.synchronize(), timed with CUDA events on the launching stream. Every
step reads the next of R device copies of the weights (R x weight bytes > 4 x L2), so no step
finds its weights in L2. `e2e` repeats the K steps through the C ABI with host buffers
(w4a16_gemm_host): each step copies x from pinned host memory and reads y back.

--impl reference times the CPU oracle (fp64, oracle/) on the same metric; under torchrun only
rank 0 runs it. --workload selects another configuration (for profiles); --sweep prints the
dense-layer sweep table to stderr.
"""
from __future__ import annotations

import argparse
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

import w4a16_inputs as inputs  # noqa: E402

METRIC = "W4A16 GEMM weight-stream GB/s & TFLOP/s vs GB300 roofline, M=1..1024"
GROUP = inputs.GROUP
L2_BYTES = 129 * 1024 * 1024  # GB300 L2 (queried at run time when a device is present)

WORKLOADS = {
    "decode": ("single-stream decode GEMV", inputs.WORKLOADS["decode_gemv"]),
    "verify": ("single-stream speculative verify", inputs.WORKLOADS["spec_verify"]),
    "batched": ("batched verify", inputs.WORKLOADS["batched_verify"]),
    "oracle_scale": ("oracle-scale GEMM", inputs.WORKLOADS["oracle_scale"]),
    "head": ("output-head GEMV", inputs.WORKLOADS["output_head"]),
    "head_verify": ("output-head verify", inputs.WORKLOADS["output_head_verify"]),
}


# ------------------------------------------------------------------------------ accounting
def weight_bytes(K: int, N: int, group: int = GROUP) -> int:
    """Packed weights (4 bits each) + fp16 scales: what one step must stream from HBM."""
    return K * N // 2 + (K // group) * N * 2


def activation_bytes(M: int, K: int, N: int) -> int:
    """fp16 x read + fp16 y written."""
    return 2 * M * K + 2 * M * N


def gemm_flops(M: int, K: int, N: int) -> int:
    """Two FLOPs (multiply, add) per weight per activation row."""
    return 2 * M * N * K


def bound_tokens_per_s(bandwidth_bytes_s: float, bytes_per_token: float) -> float:
    """Single-stream ceiling: every weight read once per token."""
    return bandwidth_bytes_s / bytes_per_token


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each workload's dominant
# kernel from one ncu capture (summaries under profiles/), with the SHA-256 prefix of the kernel
# sources it was taken from: a figure is reported only while those sources are unchanged.
MEASURED_TRAFFIC = {
    "path=gemv M=1 N=5120 K=17408 ": (46_027_008, ("gemv.cu", "common.cuh"), "7f97cbde400939bb",
                                      "profiles/gemv_decode_m1_17408x5120.md"),
    "path=tc M=16 N=34816 K=5120 ": (95_082_240, ("tc_gemm.cu", "common.cuh"), "e5db09846ea61779",
                                     "profiles/tc_gemm_verify_m16_5120x34816.md"),
    "path=tc M=256 N=34816 K=5120 ": (97_315_840, ("tc_gemm.cu", "common.cuh"), "e5db09846ea61779",
                                      "profiles/tc_gemm_batched_m256_5120x34816.md"),
}


def measured_traffic(plan: str):
    """(bytes per launch, summary file) if a capture of this launch's current kernel exists."""
    import hashlib
    for prefix, (nbytes, files, digest, summary) in MEASURED_TRAFFIC.items():
        if not plan.startswith(prefix):
            continue
        m = hashlib.sha256()
        for f in files:
            with open(os.path.join(ROOT, "w4a16_weight_streaming_gb300", "csrc", f), "rb") as fh:
                m.update(fh.read())
        if m.hexdigest()[:16] == digest:
            return nbytes, summary
    return None, None


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100", "-i",
                 str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        # NCCL between the GPUs of one node; gloo where there is no GPU (the CPU reference arm
        # and the multi-process tests)
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def dist_max(dist, value: float, device) -> float:
    """Maximum of `value` over the ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch

    if dist.get_backend() != "nccl":
        device = "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------ CPU oracle timing
def oracle_prepare(mats, cols: int):
    """The workload's inputs restricted to the first `cols` columns of every matrix (a bounded
    sample for the CPU oracle)."""
    prepared = []
    for (M, K, N, seed) in mats:
        d = inputs.generate(M, K, N, GROUP, seed=seed)
        c = min(cols, N)
        prepared.append((d["x"], np.ascontiguousarray(d["qweight"][:, :c]), np.ascontiguousarray(d["scales"][:, :c]),
                         weight_bytes(K, c)))
    return prepared


def oracle_pass(prepared, nthreads: int) -> int:
    """One pass of the fp64 oracle over the sample; returns the weight bytes it covered."""
    import oracle

    nbytes = 0
    for (x, qw, sc, wb) in prepared:
        oracle.gemm(x, qw, sc, GROUP, nthreads=nthreads)
        nbytes += wb
    return nbytes


def oracle_sample(mats, cols: int, target_s: float, nthreads: int):
    """Times the oracle on the sample, repeated for about target_s seconds.
    Returns (GB/s of weights processed, seconds, repetitions)."""
    import oracle

    oracle.build()
    prepared = oracle_prepare(mats, cols)
    oracle_pass(prepared, nthreads)  # warm
    reps, nbytes, t0 = 0, 0, time.perf_counter()
    while True:
        nbytes += oracle_pass(prepared, nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return nbytes / el / 1e9, el, reps


def run_reference(args, rank: int):
    if rank != 0:
        return
    import oracle

    oracle.build()
    name, mats = WORKLOADS[args.workload]
    nthreads = oracle.default_threads()
    cols = 256
    prepared = oracle_prepare(mats, cols)
    for _ in range(args.warmup):
        oracle_pass(prepared, nthreads)
    t0 = time.perf_counter()
    total_bytes = 0
    for _ in range(args.steps):
        total_bytes += oracle_pass(prepared, nthreads)
    el = time.perf_counter() - t0
    value = total_bytes / el / 1e9
    sample = f"first {cols} columns of each matrix per step, all M rows, fp64 oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(name, mats, extra={"columns_per_matrix": cols}),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(name, mats, extra=None):
    cfg = {"workload": f"{name}: M={mats[0][0]}, K x N = " + ", ".join(f"{K}x{N}" for (_, K, N, _) in mats)
           + f", group {GROUP}",
           "M": mats[0][0], "matrices": [{"K": K, "N": N, "seed": s} for (_, K, N, s) in mats], "group": GROUP}
    if extra:
        cfg.update(extra)
    return cfg


# ------------------------------------------------------------------------------ GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--sweep", action="store_true", help="also print the dense-layer sweep table to stderr")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    dist, rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank)
        if dist is not None:
            dist.destroy_process_group()
        return

    import torch

    import w4a16_weight_streaming_gb300 as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", L2_BYTES) or L2_BYTES
    peaks = measured_peaks()
    name, mats = WORKLOADS[args.workload]

    # ---- inputs: canonical weights on the host -> R repacked device copies per matrix
    step_wbytes = sum(weight_bytes(K, N) for (_, K, N, _) in mats)
    R = max(2, -(-4 * l2 // step_wbytes))
    bufs = []
    for (M, K, N, seed) in mats:
        d = inputs.generate(M, K, N, GROUP, seed=seed)
        qw = torch.from_numpy(d["qweight"]).to(dev)
        sc = torch.from_numpy(d["scales"].view(np.int16)).to(dev)
        copies = [W.repack(qw, sc, GROUP) for _ in range(R)]
        x_host = torch.from_numpy(d["x"].view(np.int16)).view(torch.float16).pin_memory()
        x = x_host.to(dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        y_host = torch.empty((M, N), dtype=torch.float16).pin_memory()
        bufs.append(dict(M=M, K=K, N=N, copies=copies, x=x, y=y, x_host=x_host, y_host=y_host))
        del qw, sc
    torch.cuda.synchronize()

    def step(i: int):
        for b in bufs:
            qr, sr = b["copies"][i % R]
            W.gemm(b["x"], qr, sr, b["N"], b["K"], GROUP, y=b["y"])

    plans = []
    for b in bufs:
        qr, sr = b["copies"][0]
        W.gemm(b["x"], qr, sr, b["N"], b["K"], GROUP, y=b["y"])
        plans.append(W.w4a16_last_dispatch())
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after warm-up: {W.status_string(st)}")

    # ---- capture K steps (and, per matrix, K launches alone for the per-kernel roofline)
    cap_stream = torch.cuda.Stream(device=dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cap_stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap_stream, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()
        return g

    g_step = capture(lambda: [step(i) for i in range(args.steps)])
    per_matrix_graphs = []
    for j, b in enumerate(bufs):
        def one(b=b):
            for i in range(args.steps):
                qr, sr = b["copies"][i % R]
                W.gemm(b["x"], qr, sr, b["N"], b["K"], GROUP, y=b["y"])
        per_matrix_graphs.append(capture(one))
    g_step.replay()  # upload + warm
    torch.cuda.synchronize()

    def timed_replay(g) -> float:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        return e0.elapsed_time(e1)  # ms

    # keep the GPU busy around the timed region so the clock samples reflect load
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.perf_counter() + 0.8
    while time.perf_counter() < t_end:
        g_step.replay()
    ms_total = timed_replay(g_step)
    t_end = time.perf_counter() + 0.3
    while time.perf_counter() < t_end:
        g_step.replay()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms_total = dist_max(dist, ms_total, dev)
    ms_step = ms_total / args.steps

    kernel_ms = []
    for g in per_matrix_graphs:
        kernel_ms.append(timed_replay(g) / args.steps)
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after timing: {W.status_string(st)}")

    flops_step = sum(gemm_flops(b["M"], b["K"], b["N"]) for b in bufs)
    value = world * step_wbytes / (ms_step * 1e-3) / 1e9
    tflops = world * flops_step / (ms_step * 1e-3) / 1e12

    # ---- dominant kernel roofline (the matrix with the longest launches)
    j = int(np.argmax(kernel_ms))
    b = bufs[j]
    alg = weight_bytes(b["K"], b["N"]) + activation_bytes(b["M"], b["K"], b["N"])
    fl = gemm_flops(b["M"], b["K"], b["N"])
    t_k = kernel_ms[j] * 1e-3
    # arithmetic intensity decides which roof binds: ridge = peak flops / peak bytes
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if fl / alg < ridge:
        roof = {"bound": "hbm", "achieved": alg / t_k / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": fl / t_k / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"], roof["traffic_source"] = measured_traffic(plans[j])
    roof["kernel"] = plans[j]
    roof["us_per_launch"] = kernel_ms[j] * 1e3
    roof["algorithmic_bytes"] = alg
    roof["peak_source"] = peaks["source"] + (" (burst copy)" if roof["bound"] == "hbm" else " (bf16 burst; fp16 same rate)")

    # ---- end to end through the C ABI with host buffers: w4a16_gemm_host queues, per matrix, the
    # copy of x from pinned host memory, the GEMM and the copy of y back to pinned host memory
    h2d = sum(bb["x"].numel() * 2 for bb in bufs)
    d2h = sum(bb["y"].numel() * 2 for bb in bufs)
    stream = torch.cuda.current_stream().cuda_stream
    calls = [[(bb["x_host"].data_ptr(), bb["x"].data_ptr(), qr.data_ptr(), sr.data_ptr(), bb["y"].data_ptr(),
               bb["y_host"].data_ptr(), bb["M"], bb["N"], bb["K"], GROUP, stream) for (qr, sr) in bb["copies"]]
             for bb in bufs]

    def e2e_step(i: int):
        for c in calls:
            rc = W.w4a16_gemm_host(*c[i % R])
            if rc != W.OK:
                raise RuntimeError(f"w4a16_gemm_host: {W.status_string(rc)}")

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        e2e_step(i)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = dist_max(dist, e0.elapsed_time(e1), dev) / args.steps
    e2e = {"value": world * step_wbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        nthreads = oracle.default_threads()
        cols = 256
        gbs, el, reps = oracle_sample(mats, cols, args.cpu_seconds, nthreads)
        cpu = {"value": gbs, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
               "sample": f"fp64 oracle on the first {cols} columns of each matrix, {reps} repetitions, {el:.1f} s"}

    if args.sweep and rank == 0:
        sweep(W, dev, peaks, l2)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f16", "data": "synthetic",
                "config": workload_config(name, mats, extra={
                    "l2": f"each step reads the next of {R} weight copies ({R * step_wbytes / 1e6:.0f} MB, "
                          f"> 4x the {l2 / 1e6:.0f} MB L2)",
                    "timing": "CUDA graph of K steps, CUDA events", "plans": plans,
                    "parallelism": "replicas" if world > 1 else "single GPU"}),
                "tflops": tflops, "us_per_matrix": [k * 1e3 for k in kernel_ms],
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps * len(bufs), "clocks": clocks,
                "peaks": {k: v for k, v in peaks.items()}}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def sweep(W, dev, peaks, l2):
    """Dense-layer sweep: every matrix at every M, L2-cold, CUDA-graph timed. Table on stderr."""
    import torch

    rows = []
    reps = 50
    layer_us = {}
    for mname, K, N in inputs.SWEEP_MATRICES:
        qweight, scales = inputs.generate_weights(K, N, GROUP, seed=inputs.SWEEP_SEED)
        qw = torch.from_numpy(qweight).to(dev)
        sc = torch.from_numpy(scales.view(np.int16)).to(dev)
        wb = weight_bytes(K, N)
        R = max(2, -(-4 * l2 // wb))
        copies = [W.repack(qw, sc, GROUP) for _ in range(R)]
        del qw, sc
        for M in inputs.SWEEP_M:
            x = torch.from_numpy(inputs.generate_x(M, K, seed=1000 + M).view(np.int16)).view(torch.float16).to(dev)
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            for i in range(3):
                W.gemm(x, copies[i % R][0], copies[i % R][1], N, K, GROUP, y=y)
            plan = W.w4a16_last_dispatch()
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream(device=dev)
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                for i in range(reps):
                    W.gemm(x, copies[i % R][0], copies[i % R][1], N, K, GROUP, y=y)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) / reps * 1e3
            alg = wb + activation_bytes(M, K, N)
            fl = gemm_flops(M, K, N)
            t_mem = alg / (peaks["hbm_gbs"] * 1e9)
            t_tc = fl / (peaks["bf16_tflops"] * 1e12)
            frac = max(t_mem, t_tc) / (us * 1e-6)
            rows.append(dict(matrix=mname, K=K, N=N, M=M, us=us, weight_gbs=wb / (us * 1e-6) / 1e9,
                             tflops=fl / (us * 1e-6) / 1e12, roofline_frac=frac,
                             bound="hbm" if t_mem >= t_tc else "tensor", plan=plan))
            layer_us[M] = layer_us.get(M, 0.0) + us
            del g
        del copies
        torch.cuda.empty_cache()
    print(f"{'matrix':8s} {'M':>5s} {'us':>9s} {'wGB/s':>8s} {'TFLOP/s':>8s} {'roof%':>6s} bound  plan",
          file=sys.stderr)
    for r in rows:
        print(f"{r['matrix']:8s} {r['M']:5d} {r['us']:9.2f} {r['weight_gbs']:8.0f} {r['tflops']:8.1f} "
              f"{100 * r['roofline_frac']:6.1f} {r['bound']:6s} {r['plan']}", file=sys.stderr)
    total_wb = sum(weight_bytes(K, N) for _, K, N in inputs.SWEEP_MATRICES)
    for M in inputs.SWEEP_M:
        print(f"layer step M={M:5d}: {layer_us[M]:9.2f} us  ({total_wb / (layer_us[M] * 1e-6) / 1e9:7.0f} weight GB/s)",
              file=sys.stderr)
    print("SWEEP_JSON " + json.dumps({"rows": rows, "layer_us": layer_us}), file=sys.stderr)


if __name__ == "__main__":
    main()
