"""Shared helpers of the GPU parity tests: move seeded inputs to the device, run the C-ABI GEMM,
compare with the CPU oracle under the acceptance bound |y - y_ref| <= 2^-10 |y_ref| + 2^-10 sum|x w|."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def lib():
    import __graft_entry__

    __graft_entry__.build_library()
    import w4a16_weight_streaming_gb300 as W

    return W


def to_dev(d: dict, dev="cuda"):
    qw = torch.from_numpy(np.ascontiguousarray(d["qweight"])).to(dev)
    sc = torch.from_numpy(np.ascontiguousarray(d["scales"]).view(np.int16)).to(dev)
    x = torch.from_numpy(np.ascontiguousarray(d["x"]).view(np.int16)).to(dev).view(torch.float16)
    return x, qw, sc


def x_to_dev(x_bits: np.ndarray, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(dev).view(torch.float16)


def run_gemm(W, x, qw_r, sc_r, N, K, G, plan=None, stream=None):
    y = W.gemm(x, qw_r, sc_r, N, K, G, plan=plan, stream=stream)
    torch.cuda.synchronize()
    st = W.w4a16_device_status()
    assert st == W.OK, W.status_string(st)
    return y


def y_f64(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def assert_parity(y: np.ndarray, y_ref: np.ndarray, abs_ref: np.ndarray, what: str):
    ok, worst, nbad = oracle.within_tolerance(y, y_ref, abs_ref)
    assert ok, f"{what}: {nbad} of {y.size} elements outside the bound (worst err/bound {worst:.3f})"
    return worst
