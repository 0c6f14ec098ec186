"""The debug-bounds build (libw4a16_debug.so): every kernel checks each global-memory index and each
bulk-copy source range against its buffer before the access and reports W4A16_ERR_BOUNDS instead of
touching memory out of range. Small shapes on every kernel family run through it here with a clean
status word and results that match the CPU oracle (and the normal build, bit for bit)."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import assert_parity, lib, to_dev, y_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def W():
    return lib()


@pytest.fixture(scope="module")
def D(W):
    d = W.load_debug_bounds()
    assert d.w4a16_debug_bounds() == 1 and W.lib.w4a16_debug_bounds() == 0
    return d


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _status(D):
    return D.w4a16_device_status(_stream())


PLANS = [dict(path=1), dict(path=1, split_k=3), dict(path=1, split_k=16), dict(path=2, split_k=1),
         dict(path=2, split_k=3), dict(path=2, m_tile=16, k_chunk=256, split_k=2),
         dict(path=2, m_tile=16, dequant_warps=8, split_k=2), dict(path=2, m_tile=64, mma_issuers=2, k_chunk=256),
         dict(path=2, m_tile=128, split_k=2), dict(path=2, m_tile=256, split_k=3)]


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: "-".join(f"{k}{v}" for k, v in p.items()))
def test_every_kernel_family_runs_clean(W, D, plan):
    M = 5 if plan["path"] == 1 else 37
    K, N, G = 1280, 352, 128  # ragged last column tile, uneven splits
    d = inputs.generate(M, K, N, G, seed=700 + M)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    x, qw, sc = to_dev(d)
    qw_r = torch.empty(N * K // 8, dtype=torch.int32, device="cuda")
    sc_r = torch.empty((K // G) * N, dtype=torch.int16, device="cuda")
    assert D.w4a16_repack(qw.data_ptr(), sc.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), N, K, G, _stream()) == 0
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    p = W.Plan(**plan)
    assert D.w4a16_gemm_ex(x.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), y.data_ptr(), M, N, K, G,
                           ctypes.byref(p), _stream()) == 0
    torch.cuda.synchronize()
    assert _status(D) == W.OK
    assert_parity(y_f64(y), y_ref, abs_ref, f"debug-bounds build {plan}")
    y_norm = W.gemm(x, *W.repack(qw, sc, G), N, K, G, plan=plan)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_norm.view(torch.int16))


def test_repack_round_trip_and_activation_run_clean(W, D):
    K, N, G = 512, 96, 64
    d = inputs.generate(1, K, N, G, seed=710)
    _, qw, sc = to_dev(d)
    qw_r = torch.empty(N * K // 8, dtype=torch.int32, device="cuda")
    sc_r = torch.empty((K // G) * N, dtype=torch.int16, device="cuda")
    qw2 = torch.empty_like(qw)
    sc2 = torch.empty_like(sc)
    s = _stream()
    assert D.w4a16_repack(qw.data_ptr(), sc.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), N, K, G, s) == 0
    assert D.w4a16_unrepack(qw_r.data_ptr(), sc_r.data_ptr(), qw2.data_ptr(), sc2.data_ptr(), N, K, G, s) == 0
    gu = torch.randn((3, 2 * 40), device="cuda").half()
    act = torch.empty((3, 40), dtype=torch.float16, device="cuda")
    assert D.w4a16_silu_mul(gu.data_ptr(), act.data_ptr(), 3, 40, s) == 0
    torch.cuda.synchronize()
    assert _status(D) == W.OK
    assert torch.equal(qw2, qw) and torch.equal(sc2, sc)
    assert torch.equal(act.view(torch.int16), W.silu_mul(gu).view(torch.int16))


@pytest.mark.parametrize("plan", [dict(path=2, m_tile=256, split_k=1), dict(path=2, m_tile=256, split_k=1, tail_split=2),
                                  dict(path=2, m_tile=128, split_k=1)], ids=["persistent", "tail", "persistent128"])
def test_persistent_grid_and_tail_run_clean(W, D, plan):
    """153 work items of 128 columns (the last 96 wide): a persistent grid of one CTA per SM, or
    152 unsplit items and a K-split tail, through the index-checking build."""
    M, K, N, G = 200, 256, 19552, 128
    d = inputs.generate(M, K, N, G, seed=720)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    x, qw, sc = to_dev(d)
    qw_r = torch.empty(N * K // 8, dtype=torch.int32, device="cuda")
    sc_r = torch.empty((K // G) * N, dtype=torch.int16, device="cuda")
    assert D.w4a16_repack(qw.data_ptr(), sc.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), N, K, G, _stream()) == 0
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    p = W.Plan(**plan)
    assert D.w4a16_gemm_ex(x.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), y.data_ptr(), M, N, K, G,
                           ctypes.byref(p), _stream()) == 0
    torch.cuda.synchronize()
    assert _status(D) == W.OK
    what = ctypes.create_string_buffer(512)
    D.w4a16_last_dispatch(what, 512)
    assert (b"tail_split=2" in what.value) == ("tail_split" in plan), what.value
    assert_parity(y_f64(y), y_ref, abs_ref, f"debug-bounds build {plan}")
    y_norm = W.gemm(x, *W.repack(qw, sc, G), N, K, G, plan=plan)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_norm.view(torch.int16))


@pytest.mark.parametrize("M,split", [(1, 1), (2, 3)])
def test_gemv_batch_depth_runs_clean(W, D, M, split):
    """The GEMV with 8 blocks in flight per warp (one or two rows) through the index-checking build."""
    K, N, G = 1280, 352, 128
    d = inputs.generate(M, K, N, G, seed=730 + M)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    x, qw, sc = to_dev(d)
    qw_r = torch.empty(N * K // 8, dtype=torch.int32, device="cuda")
    sc_r = torch.empty((K // G) * N, dtype=torch.int16, device="cuda")
    assert D.w4a16_repack(qw.data_ptr(), sc.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), N, K, G, _stream()) == 0
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    p = W.Plan(path=1, split_k=split)
    assert D.w4a16_gemm_ex(x.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), y.data_ptr(), M, N, K, G,
                           ctypes.byref(p), _stream()) == 0
    torch.cuda.synchronize()
    assert _status(D) == W.OK
    what = ctypes.create_string_buffer(512)
    D.w4a16_last_dispatch(what, 512)
    assert b"unroll=8" in what.value, what.value
    assert_parity(y_f64(y), y_ref, abs_ref, f"debug-bounds build GEMV M={M} split {split}")
