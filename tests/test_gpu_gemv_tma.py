"""The TMA-fed CUDA-core GEMV (path 4, M <= 4) against the CPU oracle.

Same acceptance bound as every GEMM test: |y - y_ref| <= 2^-10 |y_ref| + 2^-10 sum_k |x w| per
element; one-hot rows bit-exact. Shapes cover a partial last stage (K not a multiple of the stage),
a ragged 96-column last tile, scale groups that straddle stages, and cluster splits."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import w4a16_inputs as inputs
from gpu_util import assert_parity, lib, run_gemm, to_dev, x_to_dev, y_f64

pytestmark = pytest.mark.gpu

GT = 4


@pytest.fixture(scope="module")
def W():
    return lib()


def _repacked(W, d, G):
    x, qw, sc = to_dev(d)
    qw_r, sc_r = W.repack(qw, sc, G)
    return x, qw_r, sc_r


PLANS = [dict(path=GT), dict(path=GT, split_k=1), dict(path=GT, split_k=3), dict(path=GT, split_k=5, k_chunk=128),
         dict(path=GT, split_k=2, k_chunk=256, stages=2), dict(path=GT, split_k=1, k_chunk=128, stages=7)]


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("K", [1024, 1216])
def test_rows_and_partial_stages(W, M, K):
    N, G = 352, 64  # three tiles, the last 96 wide; K = 1216 leaves a partial last stage
    d = inputs.generate(M, K, N, G, seed=40 + M + K)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    x, qw_r, sc_r = _repacked(W, d, G)
    for plan in PLANS:
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert "path=gemv_tma" in W.w4a16_last_dispatch()
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("G,K", [(32, 1536), (128, 1536), (256, 1536), (384, 1536), (96, 1920), (160, 1920)])
def test_group_sizes(W, G, K):
    M, N = 2, 256
    d = inputs.generate(M, K, N, G, seed=G)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    x, qw_r, sc_r = _repacked(W, d, G)
    for plan in (dict(path=GT, k_chunk=128, split_k=2), dict(path=GT, k_chunk=256, split_k=3)):
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_one_hot_rows_are_exact(W):
    K, N, G = 1024, 256, 128
    ks = [0, 7, 300, 1023]
    d = inputs.generate(len(ks), K, N, G, seed=41)
    x_bits = np.zeros((len(ks), K), dtype=np.uint16)
    for m, k in enumerate(ks):
        x_bits[m, k] = 0x3C00
    w_ref = np.asarray(oracle.dequant(d["qweight"], d["scales"], G)).astype(np.float16).view(np.uint16)
    _, qw, sc = to_dev(d)
    qw_r, sc_r = W.repack(qw, sc, G)
    for plan in (dict(path=GT, split_k=1), dict(path=GT, split_k=4)):
        y = run_gemm(W, x_to_dev(x_bits), qw_r, sc_r, N, K, G, plan=plan).cpu().numpy().view(np.uint16)
        for m, k in enumerate(ks):
            same = (y[m] == w_ref[k]) | (((y[m] | w_ref[k]) & 0x7FFF) == 0)
            assert same.all(), f"row {m} (k={k})"


def test_zero_scales_give_zero(W):
    M, K, N, G = 3, 1024, 256, 128
    d = inputs.generate(M, K, N, G, seed=42)
    d["scales"] = np.zeros_like(d["scales"])
    x, qw_r, sc_r = _repacked(W, d, G)
    y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=dict(path=GT, split_k=2))
    assert (y.float().abs().cpu().numpy() == 0).all()


@pytest.mark.parametrize("M,K,N,seed", inputs.WORKLOADS["decode_gemv"])
def test_decode_workload_sampled(W, M, K, N, seed):
    G = 128
    d = inputs.generate(M, K, N, G, seed=seed)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = y_f64(run_gemm(W, x, qw_r, sc_r, N, K, G, plan=dict(path=GT)))
    ns = np.arange(0, N, 37, dtype=np.int64)
    ms = np.zeros_like(ns)
    y_ref, abs_ref = oracle.gemm_sampled(d["x"], d["qweight"], d["scales"], G, ms, ns)
    assert_parity(y[ms, ns], y_ref, abs_ref, W.w4a16_last_dispatch())


def test_rejects_more_than_four_rows(W):
    M, K, N, G = 5, 1024, 256, 128
    d = inputs.generate(M, K, N, G, seed=43)
    x, qw_r, sc_r = _repacked(W, d, G)
    with pytest.raises(W.W4A16Error):
        W.gemm(x, qw_r, sc_r, N, K, G, plan=dict(path=GT))
