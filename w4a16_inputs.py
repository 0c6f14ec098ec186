"""Seeded synthetic inputs for the W4A16 GEMM, shared by the tests, the bench and the oracle runs.

This module holds no arithmetic of the method: it only draws random numbers and writes them in
the workload's canonical storage format. The oracle (``oracle/``) and the CUDA library each
read that format with their own code.

Recipe (one ``torch.Generator('cpu')`` per matrix, seeded, draws in this order):
  1. q ~ U{0..15}, shape [K, N]            (``torch.randint(0, 16, dtype=uint8)``)
  2. U ~ U[0, 1), shape [K/G, N], fp32     (``torch.rand``)
  3. x ~ N(0, 1), shape [M, K], fp32       (``torch.randn``)
  scales = fp16_rne(0.002 * (1 + U)) computed in fp32; x = fp16_rne(x).
  qweight int32 [K/8, N]: nibble j of word [k/8, n] holds q[8*(k/8) + j, n] (low nibble first).

The workloads below are the decode / verify shapes of a 27B-class dense layer: hidden 5120,
MLP width 17,408 (gate+up fused: 34,816 columns), fused qkv 7,168 columns, output projection
5120x5120, group 128 along K.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch

GROUP = 128

# name -> list of (M, K, N, seed)
WORKLOADS = {
    "oracle_scale": [(4, 1024, 1024, 0)],
    "decode_gemv": [(1, 5120, 5120, 1), (1, 17408, 5120, 1)],
    "spec_verify": [(16, 5120, 34816, 2)],
    "batched_verify": [(256, 5120, 34816, 3), (256, 17408, 5120, 3)],
    # the output head (vocabulary projection) of the same model: one decode row, and a verify step
    "output_head": [(1, 5120, 248320, 5)],
    "output_head_verify": [(16, 5120, 248320, 5)],
}
SWEEP_MATRICES = [("qkv", 5120, 7168), ("o", 5120, 5120), ("gate_up", 5120, 34816), ("down", 17408, 5120)]
SWEEP_M = [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024]
SWEEP_SEED = 4


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """uint8 q[K, N] (values 0..15) -> canonical int32 qweight[K/8, N], low nibble first."""
    q = np.asarray(q)
    K, N = q.shape
    assert K % 8 == 0
    q3 = q.reshape(K // 8, 8, N)
    words = np.zeros((K // 8, N), np.uint32)
    for j in range(8):
        words |= (q3[:, j, :].astype(np.uint32) & np.uint32(0xF)) << np.uint32(4 * j)
    return words.view(np.int32)


def half_bits(t: torch.Tensor) -> np.ndarray:
    """fp16 torch tensor -> its uint16 bit patterns (numpy)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def generate_weights(K: int, N: int, group: int = GROUP, seed: int = 0, gen: torch.Generator | None = None):
    """(qweight int32 [K/8, N], scales uint16-bits [K/G, N]) drawn as in the module recipe."""
    g = gen if gen is not None else torch.Generator("cpu").manual_seed(seed)
    q = torch.randint(0, 16, (K, N), generator=g, dtype=torch.uint8)
    u = torch.rand((K // group, N), generator=g, dtype=torch.float32)
    scales = (0.002 * (1.0 + u)).to(torch.float16)
    return pack_nibbles(q.numpy()), half_bits(scales)


# NVFP4 weights: 4-bit E2M1 codes, one E4M3 scale pattern per 16 weights along K, one fp32 tensor
# scale. Codes are drawn uniformly from all 16 patterns; scale patterns uniformly from
# [0x30, 0x40) (values 0.5 .. 1.875: every exponent/mantissa combination of that binade pair);
# the tensor scale is 1/256, so that |g * w| <= 6 * 1.875 / 256 ~ 0.044, the range of the int4
# workload's weights.
NVFP4_BLOCK = 16
NVFP4_TENSOR_SCALE = 1.0 / 256.0


def generate_nvfp4_weights(K: int, N: int, seed: int = 0, gen: torch.Generator | None = None):
    """(qweight int32 [K/8, N] of E2M1 codes, scales8 uint8 [K/16, N] of E4M3 patterns, g float)."""
    g = gen if gen is not None else torch.Generator("cpu").manual_seed(seed)
    q = torch.randint(0, 16, (K, N), generator=g, dtype=torch.uint8)
    s8 = torch.randint(0x30, 0x40, (K // NVFP4_BLOCK, N), generator=g, dtype=torch.uint8)
    return pack_nibbles(q.numpy()), s8.numpy().copy(), NVFP4_TENSOR_SCALE


def generate(M: int, K: int, N: int, group: int = GROUP, seed: int = 0):
    """dict(x uint16 [M, K], qweight int32 [K/8, N], scales uint16 [K/G, N]) for one matrix."""
    g = torch.Generator("cpu").manual_seed(seed)
    qweight, scales = generate_weights(K, N, group, gen=g)
    x = torch.randn((M, K), generator=g, dtype=torch.float32).to(torch.float16)
    return {"x": half_bits(x), "qweight": qweight, "scales": scales, "M": M, "K": K, "N": N, "group": group,
            "seed": seed}


def generate_x(M: int, K: int, seed: int) -> np.ndarray:
    """Activations only, fp16 bits [M, K], from their own generator (sweep rows of several M)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return half_bits(torch.randn((M, K), generator=g, dtype=torch.float32).to(torch.float16))


def digest(*arrays: np.ndarray) -> str:
    """SHA-256 over the raw bytes of the given arrays (records which inputs a run used)."""
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()[:16]
