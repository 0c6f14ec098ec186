#!/usr/bin/env python3
"""Benchmark of the W4A16 weight-streaming GEMM on GB300 (one JSON line on stdout).

Default workload: the dense-layer sweep. The four matrices of one dense layer (K x N = 5120 x 7168
fused qkv, 5120 x 5120 o, 5120 x 34816 fused gate+up, 17408 x 5120 down; group 128) at every M in
{1, 2, 4, ..., 1024}. One step = one pass of the hot path over all 44 (M, matrix) GEMMs, in layer
order (for each M: qkv, o, gate+up, down), each y = x . dequant(W) through the C ABI. `value` =
weight bytes streamed per step / step time (effective weight-stream GB/s of the whole sweep);
`tflops` likewise; `rows` gives every (matrix, M) launch on its own: mean us (plain CUDA graph),
median / p10 / p90 us (per-launch event pairs), weight GB/s, TFLOP/s, roofline fraction, bound and
plan.

Timing: W untimed warm-up steps; the K timed steps are K replays of a CUDA graph of one step,
bracketed by a barrier and torch.cuda.synchronize(), timed with CUDA events on the launching stream.
L2: every weight matrix exists in R device copies and consecutive uses of one copy are at least 4 x
L2 bytes of other weights apart, so no launch finds its weights in L2. `e2e` repeats steps through
w4a16_gemm_host with host buffers (x copied in from pinned host memory, y copied back, every GEMM of
the step, the independent GEMMs spread over eight streams). More objects, outside the timed step:
`decode_step_chain` (64 dense layers in one CUDA graph per decode step, at B = 1 .. 64 streams),
`nvfp4` (the same four matrices with NVFP4 weights at M = 1, 16, 256, and their chain) and `w4a8`
(the same int4 weights with int8 activations at M = 1, 8, 16, 256, the quantisation timed beside
each row, and their chain with the quantisation inside the step).

--workload picks one of the single configurations instead (decode, verify, batched, head, ...):
the same line for that configuration. --impl reference times the CPU oracle (fp64, oracle/) on a
bounded sample of the same workload; under torchrun only rank 0 runs it.
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
    """Packed weights (4 bits each) + fp16 scales: what one launch must stream from HBM."""
    return K * N // 2 + (K // group) * N * 2


def activation_bytes(M: int, K: int, N: int) -> int:
    """fp16 x read + fp16 y written."""
    return 2 * M * K + 2 * M * N


def gemm_flops(M: int, K: int, N: int) -> int:
    """Two FLOPs (multiply, add) per weight per activation row."""
    return 2 * M * N * K


def roofline_seconds(M: int, K: int, N: int, peaks: dict) -> tuple[float, float]:
    """(t_mem, t_tensor): the weight + activation bytes at the HBM peak, the FLOPs at the tensor peak."""
    t_mem = (weight_bytes(K, N) + activation_bytes(M, K, N)) / (peaks["hbm_gbs"] * 1e9)
    t_tc = gemm_flops(M, K, N) / (peaks["bf16_tflops"] * 1e12)
    return t_mem, t_tc


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a launch shape from one
# ncu capture (summaries under profiles/), with the SHA-256 prefix of the kernel sources it was
# taken from: a figure is reported only while those sources are unchanged.
MEASURED_TRAFFIC: dict[str, tuple[int, tuple[str, ...], str, str]] = {
    # both launches of the GEMM: the whole waves of unsplit tiles and the K-split tail
    "path=tc M=1024 N=34816 K=5120 ": (128_174_848, ("tc_gemm.cu", "common.cuh"), "bfb3c13eb1fadf53",
                                       "profiles/tc_gemm_mt256_m1024_5120x34816_traffic.md"),
}


def source_digest(files) -> str:
    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "w4a16_weight_streaming_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def measured_traffic(plan: str):
    """(bytes per launch, summary file) if a capture of this launch's current kernel exists."""
    for prefix, (nbytes, files, digest, summary) in MEASURED_TRAFFIC.items():
        if plan.startswith(prefix) and source_digest(files) == digest:
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


# ------------------------------------------------------------------------------ the work of a step
def sweep_rows():
    """(name, M, K, N) of every GEMM of one sweep step, in execution order (layer order per M)."""
    return [(name, M, K, N) for M in inputs.SWEEP_M for (name, K, N) in inputs.SWEEP_MATRICES]


def workload_rows(mats):
    return [(f"{K}x{N}", M, K, N) for (M, K, N, _) in mats]


def describe(workload: str):
    """(config dict, rows) of a workload name."""
    if workload == "sweep":
        rows = sweep_rows()
        mats = ", ".join(f"{n} {K}x{N}" for (n, K, N) in inputs.SWEEP_MATRICES)
        cfg = {"workload": f"dense-layer sweep: M in {inputs.SWEEP_M} x ({mats}), K x N, group {GROUP}, "
                           f"seed {inputs.SWEEP_SEED} (x of each M from seed 1000+M)",
               "M": inputs.SWEEP_M, "matrices": [{"name": n, "K": K, "N": N} for (n, K, N) in inputs.SWEEP_MATRICES],
               "group": GROUP, "seed": inputs.SWEEP_SEED}
        return cfg, rows
    name, mats = WORKLOADS[workload]
    cfg = {"workload": f"{name}: M={mats[0][0]}, K x N = " + ", ".join(f"{K}x{N}" for (_, K, N, _) in mats)
                       + f", group {GROUP}",
           "M": mats[0][0], "matrices": [{"K": K, "N": N, "seed": s} for (_, K, N, s) in mats], "group": GROUP}
    return cfg, workload_rows(mats)


def parse_only(spec: str | None):
    """--only "name:M,name:M": the sweep rows to keep (None = all)."""
    if not spec:
        return None
    keep = set()
    for item in spec.split(","):
        name, m = item.split(":")
        keep.add((name.strip(), int(m)))
    return keep


def host_inputs(workload: str, cols: int | None = None, only=None):
    """Host-side inputs of every row: list of dict(name, M, K, N, x, qweight, scales) with the
    weights restricted to the first `cols` columns when given (bounded oracle samples)."""
    out = []
    if workload == "sweep":
        weights = {}
        for (name, K, N) in inputs.SWEEP_MATRICES:
            if only is not None and not any(n == name for (n, _) in only):
                continue
            qw, sc = inputs.generate_weights(K, N, GROUP, seed=inputs.SWEEP_SEED)
            if cols is not None:
                qw, sc = np.ascontiguousarray(qw[:, :cols]), np.ascontiguousarray(sc[:, :cols])
            weights[name] = (qw, sc)
        xs = {}
        for (name, M, K, N) in sweep_rows():
            if only is not None and (name, M) not in only:
                continue
            if (M, K) not in xs:
                xs[(M, K)] = inputs.generate_x(M, K, seed=1000 + M)
            qw, sc = weights[name]
            out.append(dict(name=name, M=M, K=K, N=N, x=xs[(M, K)], qweight=qw, scales=sc))
        return out
    _, mats = WORKLOADS[workload]
    for (M, K, N, seed) in mats:
        d = inputs.generate(M, K, N, GROUP, seed=seed)
        qw, sc = d["qweight"], d["scales"]
        if cols is not None:
            qw, sc = np.ascontiguousarray(qw[:, :cols]), np.ascontiguousarray(sc[:, :cols])
        out.append(dict(name=f"{K}x{N}", M=M, K=K, N=N, x=d["x"], qweight=qw, scales=sc))
    return out


# ------------------------------------------------------------------------------ CPU oracle timing
def oracle_pass(items, nthreads: int) -> int:
    """One pass of the fp64 oracle over the sample; returns the weight bytes it covered."""
    import oracle

    nbytes = 0
    for it in items:
        oracle.gemm(it["x"], it["qweight"], it["scales"], GROUP, nthreads=nthreads)
        nbytes += weight_bytes(it["K"], it["qweight"].shape[1])
    return nbytes


def column_sample(items, cols: int):
    """The same rows with every weight matrix cut to its first `cols` columns."""
    return [dict(it, qweight=np.ascontiguousarray(it["qweight"][:, :cols]),
                 scales=np.ascontiguousarray(it["scales"][:, :cols])) for it in items]


def oracle_sample(items, cols: int, target_s: float, nthreads: int):
    """The oracle on a bounded sample of the rows, repeated for about target_s seconds.
    Returns (GB/s of weights processed, seconds, repetitions)."""
    import oracle

    oracle.build()
    items = column_sample(items, cols)
    oracle_pass(items, nthreads)  # warm
    reps, nbytes, t0 = 0, 0, time.perf_counter()
    while True:
        nbytes += oracle_pass(items, nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return nbytes / el / 1e9, el, reps


def oracle_single_thread_configs(budget_s: float = 4.0):
    """The oracle on ONE thread for the three smallest configurations (oracle-scale in full, decode
    and verify on a column sample), as us per call extrapolated to the full matrix."""
    import oracle

    oracle.build()
    res = []
    for key, cols in (("oracle_scale", None), ("decode", 128), ("verify", 32)):
        items = host_inputs(key, cols)
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle_pass(items, 1)
            reps += 1
            if time.perf_counter() - t0 >= budget_s / 3:
                break
        el = (time.perf_counter() - t0) / reps
        frac = sum(it["qweight"].shape[1] for it in items) / sum(it["N"] for it in items)
        res.append({"config": key, "threads": 1, "columns_timed": cols or "all",
                    "s_per_call_full_matrix": el / frac, "weight_gbs": sum(
                        weight_bytes(it["K"], it["qweight"].shape[1]) for it in items) / el / 1e9})
    return res


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                low = line.lower()
                if low.startswith("model name") or low.startswith("cpu part"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_reference(args, rank: int):
    if rank != 0:
        return
    import oracle

    oracle.build()
    cfg, rows = describe(args.workload)
    nthreads = oracle.default_threads()
    cols = 4 if args.workload == "sweep" else 256
    items = host_inputs(args.workload, cols)
    for _ in range(args.warmup):
        oracle_pass(items, nthreads)
    t0 = time.perf_counter()
    total_bytes = 0
    for _ in range(args.steps):
        total_bytes += oracle_pass(items, nthreads)
    el = time.perf_counter() - t0
    value = total_bytes / el / 1e9
    sample = (f"fp64 oracle on the first {cols} columns of every matrix, every M row of every GEMM of the "
              f"step, {nthreads} threads")
    cfg = dict(cfg, columns_per_matrix=cols)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle", "sample": sample,
                             "cpu": cpu_model()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ the decode-step chain
CHAIN_LAYERS = 64
CHAIN_B = [1, 8, 16, 32, 64]


def measure_layer_chain(W, dev, sources, peaks, timed, capture, layers=CHAIN_LAYERS, reps=5, nvfp4_scale=None,
                        batches=None, w4a8=False):
    """The dense layers of one decode step as one CUDA graph: per layer qkv and o from the layer input,
    gate+up from o, silu(gate) * up, down -> the next layer's input (attention itself is not part of
    this path). Every layer streams its own device copy of the four matrices (layers x 170 MB in
    total, far beyond L2). Each B is timed over `reps` graph replays and set against the pages' step
    model t_step(B) = max(W / BW, B * F / P) with W the weight bytes and F = 2 x weights per position
    (no recurrent state or KV traffic in this path). nvfp4_scale: the sources are repacked NVFP4
    weights with that tensor scale (weight bytes counted in the canonical NVFP4 format). w4a8: int4
    weights with int8 activations: every GEMM input is quantised per token first (h once for qkv and
    o, then o and act), inside the timed step."""
    import torch

    names = [n for (n, _, _) in inputs.SWEEP_MATRICES]
    dims = {n: (K, N) for (n, K, N) in inputs.SWEEP_MATRICES}
    copies = {n: [tuple(t.clone() for t in sources[n]) for _ in range(layers)] for n in names}
    hidden = dims["o"][0]
    inter = dims["down"][0]
    nv = nvfp4_scale is not None
    wbytes = layers * sum((nvfp4_weight_bytes(K, N) if nv else weight_bytes(K, N)) for (K, N) in dims.values())
    weights_per_pos = layers * sum(K * N for (K, N) in dims.values())
    def gemm(x, w, N, K, y):
        if nv:
            W.gemm_nvfp4(x, *w, nvfp4_scale, N, K, y=y)
        else:
            W.gemm(x, *w, N, K, GROUP, y=y)

    out = []
    for B in (batches or CHAIN_B):
        h = [torch.zeros((B, hidden), dtype=torch.float16, device=dev) for _ in range(2)]
        h[0].normal_()
        qkv = torch.empty((B, dims["qkv"][1]), dtype=torch.float16, device=dev)
        o = torch.empty((B, hidden), dtype=torch.float16, device=dev)
        gu = torch.empty((B, 2 * inter), dtype=torch.float16, device=dev)
        act = torch.empty((B, inter), dtype=torch.float16, device=dev)

        def qbuf(K, consumers):  # int8 activations, their fp16 copy (tile path only), per-token scales
            tiles = any(W.w4a16_plan_for_w4a8(B, N, K, GROUP).path == W.PATH_TC for N in consumers)
            return (torch.empty((B, K), dtype=torch.int8, device=dev),
                    torch.empty((B, K), dtype=torch.float16, device=dev) if tiles else None,
                    torch.empty(B, dtype=torch.float32, device=dev))
        if w4a8:
            qh = qbuf(hidden, (dims["qkv"][1], hidden))
            qo = qbuf(hidden, (2 * inter,))
            qa = qbuf(inter, (hidden,))

        def step():
            for li in range(layers):
                x, y = h[li % 2], h[(li + 1) % 2]
                if w4a8:  # quantise each input once, in the call of its first GEMM
                    W.quantize_gemm_w4a8(x, *copies["qkv"][li], dims["qkv"][1], hidden, GROUP, out=qh, y=qkv)
                    W.gemm_w4a8(*qh, *copies["o"][li], hidden, hidden, GROUP, y=o)
                    W.quantize_gemm_w4a8(o, *copies["gate_up"][li], 2 * inter, hidden, GROUP, out=qo, y=gu)
                    W.silu_mul(gu, act)
                    W.quantize_gemm_w4a8(act, *copies["down"][li], hidden, inter, GROUP, out=qa, y=y)
                    continue
                gemm(x, copies["qkv"][li], dims["qkv"][1], hidden, qkv)
                gemm(x, copies["o"][li], hidden, hidden, o)
                gemm(o, copies["gate_up"][li], 2 * inter, hidden, gu)
                W.silu_mul(gu, act)
                gemm(act, copies["down"][li], hidden, inter, y)

        step()  # plans resolved outside the capture
        torch.cuda.synchronize()
        g = capture(step)
        g.replay()
        torch.cuda.synchronize()
        ms = timed(g.replay, reps) / reps
        del g
        t_mem = wbytes / (peaks["hbm_gbs"] * 1e9)
        t_tc = B * 2.0 * weights_per_pos / (peaks["bf16_tflops"] * 1e12)
        out.append({"B": B, "us_per_step": ms * 1e3, "tokens_per_s": B / (ms * 1e-3),
                    "weight_gbs": wbytes / (ms * 1e-3) / 1e9, "model_us": max(t_mem, t_tc) * 1e6,
                    "model_frac": max(t_mem, t_tc) / (ms * 1e-3), "bound": "hbm" if t_mem >= t_tc else "tensor"})
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after the layer chain: {W.status_string(st)}")
    del copies
    torch.cuda.empty_cache()
    kps = (8 if w4a8 else 5) * layers
    return {"layers": layers, "kernels_per_step": kps, "weight_bytes_per_step": wbytes,
            "weights": "NVFP4 (E2M1 + E4M3 per 16 k + fp32 tensor scale)" if nv else "int4, fp16 scales per 128 k",
            "activations": "int8 per token (quantised in the step)" if w4a8 else "fp16",
            "what": "per layer: qkv(h), o(h), gate_up(o), silu(gate)*up, down -> next h; one CUDA graph per step, "
                    "programmatic dependent launch between the kernels; model t_step(B) = max(W/BW, B*2*weights/P) "
                    "with the measured peaks", "rows": out}


NVFP4_M = [1, 16, 256]
E2E_STREAMS = 8  # streams the end-to-end step spreads its independent GEMMs over (measured: 3 -> 775,
#                 4 -> 837, 6 -> 912, 8 -> 933 GB/s)


def nvfp4_weight_bytes(K: int, N: int) -> int:
    """Canonical NVFP4 bytes: 4-bit codes + one E4M3 byte per 16 weights (0.5625 B per weight)."""
    return K * N // 2 + (K // 16) * N


def nvfp4_device_bytes(K: int, N: int) -> int:
    """What the device layout streams: 4-bit codes + one fp16 scale per 16 weights (0.625 B)."""
    return K * N // 2 + (K // 16) * N * 2


def measure_nvfp4(W, dev, peaks, timed, capture, l2, n_launches=100, keep=None):
    """The dense-layer matrices with NVFP4 weights at M = 1, 16, 256: per row a CUDA graph of
    `n_launches` launches cycling over enough repacked copies that they exceed 4 x L2; roofline
    fraction against the canonical NVFP4 bytes (the device layout's fp16 scales add 0.0625 B per
    weight, reported as device_gbs)."""
    import torch

    rows = []
    for (name, K, N) in inputs.SWEEP_MATRICES:
        if keep is not None and not any(n == name for (n, _) in keep):
            continue
        qw, s8, g = inputs.generate_nvfp4_weights(K, N, seed=inputs.SWEEP_SEED)
        q = torch.from_numpy(qw).to(dev)
        sc = torch.from_numpy(s8).to(dev)
        R = max(2, -(-4 * l2 // nvfp4_device_bytes(K, N)))
        copies = [W.repack_nvfp4(q, sc) for _ in range(R)]
        del q, sc
        for M in NVFP4_M:
            if keep is not None and (name, M) not in keep:
                continue
            x = torch.from_numpy(inputs.generate_x(M, K, seed=1000 + M).view(np.int16)).view(torch.float16).to(dev)
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            W.gemm_nvfp4(x, *copies[0], g, N, K, y=y)
            plan = W.w4a16_last_dispatch()
            torch.cuda.synchronize()
            gr = capture(lambda: [W.gemm_nvfp4(x, *copies[i % R], g, N, K, y=y) for i in range(n_launches)])
            gr.replay()
            us = timed(gr.replay) / n_launches * 1e3
            del gr
            wb = nvfp4_weight_bytes(K, N)
            t_mem = (wb + activation_bytes(M, K, N)) / (peaks["hbm_gbs"] * 1e9)
            t_tc = gemm_flops(M, K, N) / (peaks["bf16_tflops"] * 1e12)
            rows.append(dict(matrix=name, M=M, K=K, N=N, us=us, weight_gbs=wb / (us * 1e-6) / 1e9,
                             device_gbs=nvfp4_device_bytes(K, N) / (us * 1e-6) / 1e9,
                             tflops=gemm_flops(M, K, N) / (us * 1e-6) / 1e12,
                             roofline_frac=max(t_mem, t_tc) / (us * 1e-6), bound="hbm" if t_mem >= t_tc else "tensor",
                             plan=plan))
        del copies
        torch.cuda.empty_cache()
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after the NVFP4 rows: {W.status_string(st)}")
    layer = {}
    total = sum(nvfp4_weight_bytes(K, N) for (_, K, N) in inputs.SWEEP_MATRICES)
    for M in NVFP4_M if keep is None else []:
        us = sum(r["us"] for r in rows if r["M"] == M)
        layer[str(M)] = {"us": us, "weight_gbs": total / (us * 1e-6) / 1e9}
    return {"format": "E2M1 codes, one E4M3 scale per 16 k, fp32 tensor scale; fp16 activations",
            "bytes_per_weight": 0.5625, "device_bytes_per_weight": 0.625, "layer_step": layer, "rows": rows}


W4A8_M = [1, 8, 16, 256]


def measure_w4a8(W, dev, peaks, timed, capture, l2, n_launches=100, keep=None):
    """The dense-layer matrices with int4 weights and int8 activations at M = 1, 8, 16, 256: per row
    a CUDA graph of `n_launches` GEMM launches cycling over enough repacked copies that they exceed
    4 x L2, and beside it the per-token quantisation of that row's input ([M, K], its own graph).
    Roofline bytes: the weights plus int8 x and fp16 y."""
    import torch

    rows = []
    for (name, K, N) in inputs.SWEEP_MATRICES:
        if keep is not None and not any(n == name for (n, _) in keep):
            continue
        qw, sc = inputs.generate_weights(K, N, GROUP, seed=inputs.SWEEP_SEED)
        q = torch.from_numpy(qw).to(dev)
        s = torch.from_numpy(sc.view(np.int16)).to(dev)
        R = max(2, -(-4 * l2 // weight_bytes(K, N)))
        copies = [W.repack(q, s, GROUP) for _ in range(R)]
        del q, s
        for M in W4A8_M:
            if keep is not None and (name, M) not in keep:
                continue
            x = torch.from_numpy(inputs.generate_x(M, K, seed=1000 + M).view(np.int16)).view(torch.float16).to(dev)
            act = W.quantize_x_int8(x, with_f16=W.w4a16_plan_for_w4a8(M, N, K, GROUP).path == W.PATH_TC)
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            W.gemm_w4a8(*act, *copies[0], N, K, GROUP, y=y)
            plan = W.w4a16_last_dispatch()
            torch.cuda.synchronize()
            gr = capture(lambda: [W.gemm_w4a8(*act, *copies[i % R], N, K, GROUP, y=y) for i in range(n_launches)])
            gr.replay()
            us = timed(gr.replay) / n_launches * 1e3
            del gr
            gq = capture(lambda: [W.quantize_x_int8(x, out=act) for _ in range(n_launches)])
            gq.replay()
            us_q = timed(gq.replay) / n_launches * 1e3
            del gq
            # quantisation and GEMM in one call (two kernels, the GEMM with programmatic dependent launch)
            W.quantize_gemm_w4a8(x, *copies[0], N, K, GROUP, out=act, y=y)
            plan_qg = W.w4a16_last_dispatch()
            gf = capture(lambda: [W.quantize_gemm_w4a8(x, *copies[i % R], N, K, GROUP, out=act, y=y)
                                  for i in range(n_launches)])
            gf.replay()
            us_qg = timed(gf.replay) / n_launches * 1e3
            del gf
            wb = weight_bytes(K, N)
            ab = M * K + 2 * M * N
            t_mem = (wb + ab) / (peaks["hbm_gbs"] * 1e9)
            t_tc = gemm_flops(M, K, N) / (peaks["bf16_tflops"] * 1e12)
            rows.append(dict(matrix=name, M=M, K=K, N=N, us=us, us_quantize=us_q, us_quantize_gemm=us_qg,
                             quantize_gemm_plan=plan_qg, weight_gbs=wb / (us * 1e-6) / 1e9,
                             tflops=gemm_flops(M, K, N) / (us * 1e-6) / 1e12,
                             roofline_frac=max(t_mem, t_tc) / (us * 1e-6), bound="hbm" if t_mem >= t_tc else "tensor",
                             plan=plan))
        del copies
        torch.cuda.empty_cache()
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after the W4A8 rows: {W.status_string(st)}")
    layer = {}
    total = sum(weight_bytes(K, N) for (_, K, N) in inputs.SWEEP_MATRICES)
    for M in W4A8_M if keep is None else []:
        us = sum(r["us"] for r in rows if r["M"] == M)
        layer[str(M)] = {"us": us, "weight_gbs": total / (us * 1e-6) / 1e9}
    return {"format": "int4 weights (fp16 scales per 128 k), int8 activations per token",
            "quantisation": "sx = amax / 127, xq = rne(x / sx) in binary32; us_quantize times it alone",
            "layer_step": layer, "rows": rows}


# ------------------------------------------------------------------------------ GPU arm
def percentile(v, q):
    return float(np.percentile(np.asarray(v, dtype=np.float64), q))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["sweep"] + sorted(WORKLOADS), default="sweep")
    ap.add_argument("--launches", type=int, default=200, help="per-row launches for median / p10 / p90")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-streams", type=int, default=E2E_STREAMS,
                    help="streams the end-to-end step spreads its independent GEMMs over")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--table", action="store_true", help="also print the per-row table to stderr")
    ap.add_argument("--no-chain", action="store_true", help="skip the 64-layer decode-step chain")
    ap.add_argument("--no-nvfp4", action="store_true", help="skip the NVFP4-weight rows")
    ap.add_argument("--no-w4a8", action="store_true", help="skip the int8-activation rows")
    ap.add_argument("--w4a8-rows", default=None, help='int8-activation rows to run, e.g. "down:1" (profiling)')
    ap.add_argument("--nvfp4-rows", default=None,
                    help='NVFP4 rows to run, e.g. "gate_up:16" (M in 1, 16, 256; with --only: profiling)')
    ap.add_argument("--only", default=None, help='sweep rows to run, e.g. "o:16,gate_up:256" (profiling)')
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
    cfg, _ = describe(args.workload)

    # ---- inputs: canonical weights on the host -> repacked device copies per matrix. Every launch
    # of the step reads its own copy, and a matrix has enough copies that its copies cycle through
    # more than 4 x L2 bytes: no launch finds its weights in L2.
    only = parse_only(args.only) if args.workload == "sweep" else None
    if only is not None:
        cfg = dict(cfg, only=sorted(f"{n}:{m}" for (n, m) in only))
    items = host_inputs(args.workload, only=only)
    mats = {}
    for it in items:
        if it["name"] in mats:
            continue
        wb = weight_bytes(it["K"], it["N"])
        uses = sum(1 for jt in items if jt["name"] == it["name"])
        R = max(uses + 1, -(-4 * l2 // wb))
        qw = torch.from_numpy(it["qweight"]).to(dev)
        sc = torch.from_numpy(it["scales"].view(np.int16)).to(dev)
        mats[it["name"]] = dict(K=it["K"], N=it["N"], wb=wb, copies=[W.repack(qw, sc, GROUP) for _ in range(R)])
        del qw, sc
    step_wbytes = 0
    use_count = {n: 0 for n in mats}
    for it in items:
        it["x_host"] = torch.from_numpy(it["x"].view(np.int16)).view(torch.float16).pin_memory()
        it["xd"] = it["x_host"].to(dev)
        it["yd"] = torch.empty((it["M"], it["N"]), dtype=torch.float16, device=dev)
        it["y_host"] = torch.empty((it["M"], it["N"]), dtype=torch.float16).pin_memory()
        it["copy"] = use_count[it["name"]]  # the step's own copy of this matrix for this GEMM
        use_count[it["name"]] += 1
        step_wbytes += mats[it["name"]]["wb"]
    torch.cuda.synchronize()

    def launch(it, copy):
        qr, sr = mats[it["name"]]["copies"][copy]
        W.gemm(it["xd"], qr, sr, it["N"], it["K"], GROUP, y=it["yd"])

    def step():
        for it in items:
            launch(it, it["copy"])

    for it in items:
        launch(it, it["copy"])
        it["plan"] = W.w4a16_last_dispatch()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after warm-up: {W.status_string(st)}")

    cap_stream = torch.cuda.Stream(device=dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cap_stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap_stream, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()
        return g

    def timed(fn_replay, reps: int = 1) -> float:
        """ms of `reps` calls of fn_replay, CUDA events on the current stream, barrier + sync around."""
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn_replay()
        e1.record()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        return e0.elapsed_time(e1)

    # ---- the timed region: K replays of the one-step graph
    g_step = capture(step)
    g_step.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.perf_counter() + 0.8  # keep the GPU busy so the clock samples reflect load
    while time.perf_counter() < t_end:
        g_step.replay()
    ms_total = timed(g_step.replay, args.steps)
    t_end = time.perf_counter() + 0.3
    while time.perf_counter() < t_end:
        g_step.replay()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms_total = dist_max(dist, ms_total, dev)
    ms_step = ms_total / args.steps
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after timing: {W.status_string(st)}")

    # ---- every row on its own: a plain graph of n launches cycling over the matrix's copies (mean),
    # then the same launches with an event pair around each (median, p10, p90 of single launches)
    n = max(args.launches, 20)
    have_ext = True
    rows = []
    for it in items:
        R = len(mats[it["name"]]["copies"])
        g = capture(lambda it=it: [launch(it, i % R) for i in range(n)])
        g.replay()
        mean_us = timed(g.replay) / n * 1e3
        del g
        per = []
        if have_ext:
            try:
                evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n + 1)]

                def evloop(it=it, evs=evs):
                    for i in range(n):
                        evs[i].record()
                        launch(it, i % R)
                    evs[n].record()

                g = capture(evloop)
                g.replay()
                torch.cuda.synchronize()
                per = [evs[i].elapsed_time(evs[i + 1]) * 1e3 for i in range(n)]
                del g
            except (TypeError, RuntimeError):
                have_ext = False
                per = []
        M, K, N = it["M"], it["K"], it["N"]
        t_mem, t_tc = roofline_seconds(M, K, N, peaks)
        wb = mats[it["name"]]["wb"]
        rows.append(dict(matrix=it["name"], M=M, K=K, N=N, us=mean_us,
                         us_median=statistics.median(per) if per else None,
                         us_p10=percentile(per, 10) if per else None, us_p90=percentile(per, 90) if per else None,
                         weight_gbs=wb / (mean_us * 1e-6) / 1e9, tflops=gemm_flops(M, K, N) / (mean_us * 1e-6) / 1e12,
                         roofline_frac=max(t_mem, t_tc) / (mean_us * 1e-6), bound="hbm" if t_mem >= t_tc else "tensor",
                         plan=it["plan"]))
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after the per-row timing: {W.status_string(st)}")

    # ---- one cold launch (L2 flushed by a write larger than L2, then one launch outside any graph)
    flush = torch.empty(int(2 * l2), dtype=torch.uint8, device=dev)
    cold = {}
    for it in items:
        if it["M"] != 1 and args.workload == "sweep" and only is None:
            continue
        flush.fill_(1)
        torch.cuda.synchronize()
        cold[f"{it['name']} M={it['M']}"] = timed(lambda it=it: launch(it, 0)) * 1e3
    del flush

    # ---- dominant kernel: the row with the largest share of the step
    j = int(np.argmax([r["us"] for r in rows]))
    r = rows[j]
    alg = weight_bytes(r["K"], r["N"]) + activation_bytes(r["M"], r["K"], r["N"])
    fl = gemm_flops(r["M"], r["K"], r["N"])
    t_k = r["us"] * 1e-6
    if r["bound"] == "hbm":
        roof = {"bound": "hbm", "achieved": alg / t_k / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": fl / t_k / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"], roof["traffic_source"] = measured_traffic(r["plan"])
    roof["kernel"] = r["plan"]
    roof["us_per_launch"] = r["us"]
    roof["share_of_step"] = r["us"] / (ms_step * 1e3)
    roof["algorithmic_bytes"] = alg
    roof["algorithmic_flops"] = fl
    roof["peak_source"] = peaks["source"] + (" (burst copy)" if roof["bound"] == "hbm"
                                             else " (bf16 cuBLAS burst; fp16 runs at the same tensor rate)")
    t_roof_step = sum(max(*roofline_seconds(x["M"], x["K"], x["N"], peaks)) for x in rows)

    # ---- end to end through the C ABI with host buffers: per GEMM, w4a16_gemm_host queues the copy of
    # x from pinned host memory, the GEMM and the copy of y back to pinned host memory. The step's
    # GEMMs are independent, so they go round-robin to E2E_STREAMS streams (one call each, as a user
    # would issue them): one GEMM's copies overlap another's kernel. The streams join the timing
    # stream before and after every step.
    h2d = sum(it["xd"].numel() * 2 for it in items)
    d2h = sum(it["yd"].numel() * 2 for it in items)
    e2e_streams = [torch.cuda.Stream(device=dev) for _ in range(max(1, args.e2e_streams))]
    calls = []
    for i, it in enumerate(items):
        qr, sr = mats[it["name"]]["copies"][it["copy"]]
        calls.append((it["x_host"].data_ptr(), it["xd"].data_ptr(), qr.data_ptr(), sr.data_ptr(),
                      it["yd"].data_ptr(), it["y_host"].data_ptr(), it["M"], it["N"], it["K"], GROUP,
                      e2e_streams[i % len(e2e_streams)].cuda_stream))

    def e2e_step():
        cur = torch.cuda.current_stream()
        for s in e2e_streams:
            s.wait_stream(cur)
        for c in calls:
            rc = W.w4a16_gemm_host(*c)
            if rc != W.OK:
                raise RuntimeError(f"w4a16_gemm_host: {W.status_string(rc)}")
        for s in e2e_streams:
            cur.wait_stream(s)

    e2e_step()
    torch.cuda.synchronize()
    ne = max(1, args.e2e_steps)
    e2e_ms = dist_max(dist, timed(e2e_step, ne), dev) / ne
    e2e = {"value": world * step_wbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": ne, "streams": len(e2e_streams)}
    st = W.w4a16_device_status()
    if st != W.OK:
        raise RuntimeError(f"device status after the end-to-end steps: {W.status_string(st)}")

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        nthreads = oracle.default_threads()
        cols = 16 if args.workload == "sweep" else 256
        gbs, el, reps = oracle_sample(items, cols, args.cpu_seconds, nthreads)
        cpu = {"value": gbs, "unit": "GB/s", "cores": nthreads, "kind": "oracle", "cpu": cpu_model(),
               "sample": f"fp64 oracle on the first {cols} columns of every matrix, every M row of every GEMM "
                         f"of the step, {reps} repetitions, {el:.1f} s",
               "single_thread": oracle_single_thread_configs()}

    # ---- the decode-step chain (64 dense layers, one CUDA graph per step), sweep workload only
    chain = None
    if args.workload == "sweep" and not args.no_chain and only is None:
        chain = measure_layer_chain(W, dev, {n: m["copies"][0] for n, m in mats.items()}, peaks, timed, capture)

    nvfp4 = None
    nv_keep = parse_only(args.nvfp4_rows)
    if args.workload == "sweep" and not args.no_nvfp4 and (only is None or nv_keep is not None):
        nvfp4 = measure_nvfp4(W, dev, peaks, timed, capture, l2, keep=nv_keep)
        if nv_keep is None and not args.no_chain:
            src = {}
            for (name, K, N) in inputs.SWEEP_MATRICES:
                qw, s8, g = inputs.generate_nvfp4_weights(K, N, seed=inputs.SWEEP_SEED)
                src[name] = W.repack_nvfp4(torch.from_numpy(qw).to(dev), torch.from_numpy(s8).to(dev))
            nvfp4["decode_step_chain"] = measure_layer_chain(W, dev, src, peaks, timed, capture, nvfp4_scale=g)
            del src
            torch.cuda.empty_cache()

    w4a8 = None
    a8_keep = parse_only(args.w4a8_rows)
    if args.workload == "sweep" and not args.no_w4a8 and (only is None or a8_keep is not None):
        w4a8 = measure_w4a8(W, dev, peaks, timed, capture, l2, keep=a8_keep)
        if a8_keep is None and not args.no_chain:
            w4a8["decode_step_chain"] = measure_layer_chain(W, dev, {n: m["copies"][0] for n, m in mats.items()},
                                                            peaks, timed, capture, w4a8=True)
            torch.cuda.empty_cache()

    if args.table and rank == 0:
        print(f"{'matrix':8s} {'M':>5s} {'us':>9s} {'med':>8s} {'p10':>8s} {'p90':>8s} {'wGB/s':>7s} "
              f"{'TFLOP/s':>8s} {'roof%':>6s} bound  plan", file=sys.stderr)
        for x in rows:
            f = lambda v: f"{v:8.2f}" if v is not None else "       -"  # noqa: E731
            print(f"{x['matrix']:8s} {x['M']:5d} {x['us']:9.2f} {f(x['us_median'])} {f(x['us_p10'])} "
                  f"{f(x['us_p90'])} {x['weight_gbs']:7.0f} {x['tflops']:8.1f} {100 * x['roofline_frac']:6.1f} "
                  f"{x['bound']:6s} {x['plan']}", file=sys.stderr)
        if nvfp4:
            for x in nvfp4["rows"]:
                print(f"nvfp4 {x['matrix']:8s} {x['M']:5d} {x['us']:9.2f} us {x['weight_gbs']:7.0f} GB/s "
                      f"{x['tflops']:8.1f} TFLOP/s {100 * x['roofline_frac']:6.1f}% {x['bound']}", file=sys.stderr)
        if nvfp4 and nvfp4.get("decode_step_chain"):
            for c in nvfp4["decode_step_chain"]["rows"]:
                print(f"nvfp4 chain B={c['B']:3d}: {c['us_per_step']:9.1f} us/step {c['tokens_per_s']:9.0f} tok/s "
                      f"{c['weight_gbs']:6.0f} GB/s model {c['model_us']:8.1f} us ({100 * c['model_frac']:.1f}%)",
                      file=sys.stderr)
        if w4a8:
            for x in w4a8["rows"]:
                print(f"w4a8 {x['matrix']:8s} {x['M']:5d} {x['us']:9.2f} us (quantise {x['us_quantize']:5.2f} us, "
                      f"quantise+GEMM call {x['us_quantize_gemm']:6.2f} us) "
                      f"{x['weight_gbs']:7.0f} GB/s {x['tflops']:8.1f} TFLOP/s {100 * x['roofline_frac']:6.1f}% "
                      f"{x['bound']}", file=sys.stderr)
        if w4a8 and w4a8.get("decode_step_chain"):
            for c in w4a8["decode_step_chain"]["rows"]:
                print(f"w4a8 chain B={c['B']:3d}: {c['us_per_step']:9.1f} us/step {c['tokens_per_s']:9.0f} tok/s "
                      f"{c['weight_gbs']:6.0f} GB/s model {c['model_us']:8.1f} us ({100 * c['model_frac']:.1f}%)",
                      file=sys.stderr)
        if chain:
            for c in chain["rows"]:
                print(f"chain B={c['B']:3d}: {c['us_per_step']:9.1f} us/step {c['tokens_per_s']:9.0f} tok/s "
                      f"{c['weight_gbs']:6.0f} GB/s model {c['model_us']:8.1f} us ({100 * c['model_frac']:.1f}%, "
                      f"{c['bound']})", file=sys.stderr)

    if rank == 0:
        layer = {}
        if args.workload == "sweep" and only is None:
            total_wb = sum(weight_bytes(K, N) for (_, K, N) in inputs.SWEEP_MATRICES)
            for M in inputs.SWEEP_M:
                us = sum(x["us"] for x in rows if x["M"] == M)
                layer[str(M)] = {"us": us, "weight_gbs": total_wb / (us * 1e-6) / 1e9}
        flops_step = sum(gemm_flops(x["M"], x["K"], x["N"]) for x in rows)
        line = {"metric": METRIC, "value": world * step_wbytes / (ms_step * 1e-3) / 1e9, "unit": "GB/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
                "data": "synthetic",
                "config": dict(cfg, **{
                    "l2": "inputs larger than L2: every launch reads its own weight copy; a matrix's copies cycle "
                          f"through more than 4x the {l2 / 1e6:.0f} MB L2 (no flush needed)",
                    "timing": "K replays of a CUDA graph of one step, CUDA events on the launching stream",
                    "parallelism": "replicas" if world > 1 else "single GPU"}),
                "value_is": "weight bytes streamed per step / step time (all GEMMs of the step)",
                "tflops": world * flops_step / (ms_step * 1e-3) / 1e12,
                "step_roofline_frac": t_roof_step / (ms_step * 1e-3),
                "layer_step": layer, "rows": rows, "cold_launch_us": cold, "decode_step_chain": chain,
                "nvfp4": nvfp4, "w4a8": w4a8,
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps * sum(2 if "tail_items=" in r["plan"] else 1 for r in rows),
                "clocks": clocks,
                "peaks": {k: v for k, v in peaks.items()}}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
