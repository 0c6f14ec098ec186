"""The persistent tensor-core streaming path (path 3, M <= 64) against the CPU oracle.

Same acceptance bound as every GEMM test: |y - y_ref| <= 2^-10 |y_ref| + 2^-10 sum_k |x w| per
element; one-hot rows and zero scales bit-exact. The shapes make each persistent cluster walk
several 128-column tiles (both TMEM accumulator buffers and both split-K partial buffers are
reused), split K unevenly across cluster ranks, and end on a ragged 96-column tile."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import assert_parity, lib, run_gemm, to_dev, x_to_dev, y_f64

pytestmark = pytest.mark.gpu

STREAM = 3


@pytest.fixture(scope="module")
def W():
    return lib()


def _case(M, K, N, G, seed):
    d = inputs.generate(M, K, N, G, seed=seed)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    return d, y_ref, abs_ref


def _repacked(W, d, G):
    x, qw, sc = to_dev(d)
    qw_r, sc_r = W.repack(qw, sc, G)
    return x, qw_r, sc_r


def _pid(p):
    return "-".join(f"{k[:2]}{v}" for k, v in p.items() if k != "path")


ORACLE_SCALE = [
    dict(path=STREAM),
    dict(path=STREAM, split_k=1, clusters=1),
    dict(path=STREAM, split_k=1, clusters=3),
    dict(path=STREAM, split_k=2, clusters=3),
    dict(path=STREAM, split_k=3, clusters=2),
    dict(path=STREAM, split_k=8, clusters=1, k_chunk=128),
    dict(path=STREAM, split_k=4, clusters=2, k_chunk=256, stages=2, tmem_stages=2),
    dict(path=STREAM, split_k=1, clusters=2, k_chunk=128, stages=3, tmem_stages=7),
    dict(path=STREAM, m_tile=32, split_k=2, clusters=4),
    dict(path=STREAM, m_tile=64, split_k=5, clusters=2, k_chunk=128),
    dict(path=STREAM, m_tile=64, mma_issuers=4, split_k=2, clusters=3),
    dict(path=STREAM, m_tile=64, mma_issuers=2, k_chunk=128, tmem_stages=4, split_k=1, clusters=5),
    dict(path=STREAM, m_tile=32, mma_issuers=4, k_chunk=128, tmem_stages=4, split_k=3, clusters=2),
]


@pytest.mark.parametrize("plan", ORACLE_SCALE, ids=_pid)
def test_oracle_scale(W, plan):
    M, K, N, G = 4, 1024, 1024, 128  # 8 column tiles
    d, y_ref, abs_ref = _case(M, K, N, G, seed=0)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
    assert "path=stream" in W.w4a16_last_dispatch()
    assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


EDGE_M = [1, 2, 3, 7, 8, 15, 16, 17, 31, 32, 33, 48, 63, 64]


@pytest.fixture(scope="module")
def edge_matrix(W):
    K, N, G = 1280, 352, 128  # 10 chunks of 128 / 5 of 256; 3 tiles, the last 96 wide
    d = inputs.generate(max(EDGE_M), K, N, G, seed=12)
    x_all, qw_r, sc_r = _repacked(W, d, G)
    return d, x_all, qw_r, sc_r, K, N, G


@pytest.mark.parametrize("M", EDGE_M)
def test_edge_rows(W, edge_matrix, M):
    d, x_all, qw_r, sc_r, K, N, G = edge_matrix
    y_ref, abs_ref = oracle.gemm(d["x"][:M], d["qweight"], d["scales"], G)
    x = x_all[:M].contiguous()
    for plan in (dict(path=STREAM), dict(path=STREAM, split_k=1, clusters=1),
                 dict(path=STREAM, split_k=3, clusters=2, k_chunk=128), dict(path=STREAM, split_k=5, clusters=1)):
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_many_tiles_per_cluster(W):
    """Each cluster walks 11 tiles: the accumulator and partial-tile buffers are reused many times."""
    M, K, N, G = 16, 2048, 4096, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=21)
    x, qw_r, sc_r = _repacked(W, d, G)
    for plan in (dict(path=STREAM, split_k=1, clusters=3), dict(path=STREAM, split_k=2, clusters=3),
                 dict(path=STREAM, split_k=4, clusters=3, k_chunk=128, stages=4)):
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("G", [32, 64, 256])
def test_group_sizes(W, G):
    M, K, N = 5, 1024, 384
    d, y_ref, abs_ref = _case(M, K, N, G, seed=G + 1)
    x, qw_r, sc_r = _repacked(W, d, G)
    for plan in (dict(path=STREAM, k_chunk=128), dict(path=STREAM, k_chunk=256, split_k=2, clusters=2)):
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_one_hot_rows_are_exact(W):
    """x row m is the unit vector e_k: y[m][n] must equal the dequantised weight w[k][n] bit for bit."""
    K, N, G = 1024, 256, 128
    ks = [0, 1, 7, 8, 127, 128, 300, 511, 512, 777, 1000, 1023, 64, 65, 255, 256]
    d = inputs.generate(len(ks), K, N, G, seed=5)
    x_bits = np.zeros((len(ks), K), dtype=np.uint16)
    for m, k in enumerate(ks):
        x_bits[m, k] = 0x3C00  # 1.0
    w = oracle.dequant(d["qweight"], d["scales"], G)  # [K][N], every value an fp16 number
    w_ref = np.asarray(w).astype(np.float16).view(np.uint16)
    _, qw, sc = to_dev(d)
    qw_r, sc_r = W.repack(qw, sc, G)
    xd = x_to_dev(x_bits)
    for plan in (dict(path=STREAM, split_k=1, clusters=1), dict(path=STREAM, split_k=4, clusters=2)):
        y = run_gemm(W, xd, qw_r, sc_r, N, K, G, plan=plan).cpu().numpy().view(np.uint16)
        for m, k in enumerate(ks):
            got, want = y[m], w_ref[k]
            same = (got == want) | (((got | want) & 0x7FFF) == 0)  # +0 and -0 both accepted
            assert same.all(), f"row {m} (k={k}): {int((~same).sum())} columns differ"


def test_zero_scales_give_zero(W):
    M, K, N, G = 9, 1024, 256, 128
    d = inputs.generate(M, K, N, G, seed=6)
    d["scales"] = np.zeros_like(d["scales"])
    x, qw_r, sc_r = _repacked(W, d, G)
    y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=dict(path=STREAM, split_k=2, clusters=2))
    assert (y.float().abs().cpu().numpy() == 0).all()


def test_deterministic(W):
    M, K, N, G = 16, 5120, 1024, 128
    d = inputs.generate(M, K, N, G, seed=8)
    x, qw_r, sc_r = _repacked(W, d, G)
    plan = dict(path=STREAM, split_k=4, clusters=2)
    y1 = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan).clone()
    y2 = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
    assert torch.equal(y1, y2)


def test_stream_plan_fields(W):
    M, K, N, G = 16, 1024, 512, 128
    d = inputs.generate(M, K, N, G, seed=10)
    x, qw_r, sc_r = _repacked(W, d, G)
    run_gemm(W, x, qw_r, sc_r, N, K, G, plan=dict(path=STREAM, split_k=2, clusters=2))
    disp = W.w4a16_last_dispatch()
    for field in ("path=stream", "m_tile=16", "split_k=2", "clusters=2", "issuers=4", "acc_buffers="):
        assert field in disp, disp


def test_invalid_stream_plans_are_rejected(W):
    M, K, N, G = 65, 1024, 256, 128
    d = inputs.generate(M, K, N, G, seed=9)
    x, qw_r, sc_r = _repacked(W, d, G)
    with pytest.raises(W.W4A16Error):
        W.gemm(x, qw_r, sc_r, N, K, G, plan=dict(path=STREAM))  # more rows than one resident block
    with pytest.raises(W.W4A16Error):
        W.gemm(x[:16].contiguous(), qw_r, sc_r, N, K, G, plan=dict(path=STREAM, k_chunk=64))
    with pytest.raises(W.W4A16Error):
        W.gemm(x[:16].contiguous(), qw_r, sc_r, N, K, G, plan=dict(path=STREAM, split_k=9))  # more ranks than K chunks
