"""NVFP4 weights on the GPU against the CPU oracle.

The RTX 5090 runs of "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s" (ai.satyajit.si), section "One
weight read, shared by every stream", keep the weights in NVFP4: E2M1 codes, one E4M3 scale per 16
weights along K, one fp32 tensor scale; activations stay fp16 here. Checked:
  * the device layout (w4a16_repack_nvfp4) bit for bit against the oracle's statement of it, and
    the round trip through w4a16_unrepack_nvfp4;
  * y on every element at the acceptance bound for both paths (CUDA-core GEMV, every tile kernel,
    split-K, ragged column tiles), the full-size workloads, one-hot rows exactly, zero scales;
  * every NVFP4 kernel family through the debug-bounds build."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import assert_parity, lib, x_to_dev, y_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def W():
    return lib()


def _dev_weights(W, qw, s8):
    q = torch.from_numpy(np.ascontiguousarray(qw)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(s8)).cuda()
    return W.repack_nvfp4(q, s)


def _case(M, K, N, seed):
    qw, s8, g = inputs.generate_nvfp4_weights(K, N, seed=seed)
    x = inputs.generate_x(M, K, seed=seed + 1)
    return qw, s8, g, x


def _run(W, x_bits, r, g, N, K, plan=None):
    y = W.gemm_nvfp4(x_to_dev(x_bits), r[0], r[1], g, N, K, plan=plan)
    torch.cuda.synchronize()
    st = W.w4a16_device_status()
    assert st == W.OK, W.status_string(st)
    assert "weights=nvfp4" in W.w4a16_last_dispatch()
    return y


def test_repack_matches_oracle_layout_and_round_trips(W):
    rng = np.random.default_rng(11)
    for (K, N) in [(128, 96), (1024, 352), (5120, 544)]:
        q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
        # every finite E4M3 pattern of both signs except -0 (whose E4M3 inverse is not unique)
        pats = np.array([b for b in range(256) if b not in (0x7F, 0xFF, 0x80)], np.uint8)
        s8 = rng.choice(pats, size=(K // 16, N)).astype(np.uint8)
        qw = inputs.pack_nibbles(q)
        wr_ref, sr_ref = oracle.repack_nvfp4(qw, s8)
        r = _dev_weights(W, qw, s8)
        torch.cuda.synchronize()
        assert np.array_equal(r[0].cpu().numpy().view(np.uint32), wr_ref)
        assert np.array_equal(r[1].cpu().numpy().view(np.uint16), sr_ref)
        qw2, s82 = W.unrepack_nvfp4(r[0], r[1], N, K)
        torch.cuda.synchronize()
        assert W.w4a16_device_status() == W.OK
        assert np.array_equal(qw2.cpu().numpy(), qw) and np.array_equal(s82.cpu().numpy(), s8)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
def test_gemv_rows(W, M):
    K, N = 1024, 352  # ragged last column tile
    qw, s8, g, x = _case(M, K, N, seed=20 + M)
    y_ref, a_ref = oracle.gemm_nvfp4(x, qw, s8, g)
    r = _dev_weights(W, qw, s8)
    for split in (1, 3, 16):
        y = _run(W, x, r, g, N, K, plan=dict(path=1, split_k=split))
        assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


# every instantiated (m_tile, k_chunk, mma_issuers, dequant_warps) tile kernel
TILES = [(16, 128, 4, 16), (16, 256, 4, 16), (32, 128, 4, 16), (32, 256, 4, 16), (64, 128, 4, 16),
         (64, 256, 4, 16), (64, 256, 2, 16), (128, 128, 2, 16), (128, 128, 1, 16), (256, 128, 1, 16),
         (16, 128, 4, 8), (32, 128, 4, 8), (64, 128, 2, 8)]


@pytest.mark.parametrize("mt,kc,ni,dw", TILES)
def test_every_tile(W, mt, kc, ni, dw):
    M, K, N = mt - 3, 1280 if kc == 128 else 1024, 352
    qw, s8, g, x = _case(M, K, N, seed=mt + kc + ni + dw)
    y_ref, a_ref = oracle.gemm_nvfp4(x, qw, s8, g)
    r = _dev_weights(W, qw, s8)
    for split in (1, 3):
        plan = dict(path=2, m_tile=mt, k_chunk=kc, mma_issuers=ni, dequant_warps=dw, split_k=split)
        if dw == 8:
            plan["tmem_stages"] = 2
        y = _run(W, x, r, g, N, K, plan=plan)
        assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("path", [1, 2])
def test_one_hot_rows_are_exact(W, path):
    # x = e_k returns fp16(g * e2m1 * e4m3) exactly: one product, g a power of two
    K, N, g = 1024, 256, 0.5
    qw, s8, _, _ = _case(1, K, N, seed=31)
    ks = [0, 15, 16, 17, 127, 128, 512, 1023]  # (at most 8 rows: the GEMV's limit)
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    w = oracle.dequant_nvfp4(qw, s8)
    want = np.stack([g * w[k] for k in ks]).astype(np.float16)
    r = _dev_weights(W, qw, s8)
    plan = dict(path=1) if path == 1 else dict(path=2, m_tile=16)
    y = _run(W, x.view(np.uint16), r, g, N, K, plan=plan)
    got = y.cpu().numpy()
    # bit for bit, except that a zero weight (code 8 is -0) sums to +0 in fp32: +-0 are equal here
    nz = want.astype(np.float32) != 0
    assert np.array_equal(got.view(np.uint16)[nz], want.view(np.uint16)[nz])
    assert np.all(got.astype(np.float32)[~nz] == 0)


def test_zero_scales_and_tensor_scale(W):
    K, N, M = 512, 128, 4
    qw, s8, _, x = _case(M, K, N, seed=41)
    r0 = _dev_weights(W, qw, np.zeros_like(s8))
    for path in (1, 2):
        y = _run(W, x, r0, 1.0, N, K, plan=dict(path=path))
        assert np.all(y.float().cpu().numpy() == 0.0)
    r = _dev_weights(W, qw, s8)
    y1 = _run(W, x, r, 1.0, N, K, plan=dict(path=2))
    y4 = _run(W, x, r, 4.0, N, K, plan=dict(path=2))
    # a power-of-two tensor scale scales the fp32 sum exactly (no overflow at these sizes)
    assert np.array_equal(y4.float().cpu().numpy(), 4.0 * y1.float().cpu().numpy())
    with pytest.raises(W.W4A16Error):
        W.gemm_nvfp4(x_to_dev(x), r[0], r[1], float("nan"), N, K)


@pytest.mark.parametrize("M,K,N", [(1, 5120, 5120), (1, 17408, 5120), (16, 5120, 34816)])
def test_full_size_every_element(W, M, K, N):
    qw, s8, g, x = _case(M, K, N, seed=50 + M)
    y_ref, a_ref = oracle.gemm_nvfp4(x, qw, s8, g)
    r = _dev_weights(W, qw, s8)
    y = _run(W, x, r, g, N, K)
    assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


def test_batched_sampled(W):
    M, K, N = 256, 5120, 34816
    qw, s8, g, x = _case(M, K, N, seed=60)
    r = _dev_weights(W, qw, s8)
    y = _run(W, x, r, g, N, K)
    rng = np.random.default_rng(61)
    ms = np.concatenate([rng.integers(0, M, 1500), [0, M - 1, M - 1]])
    ns = np.concatenate([rng.integers(0, N, 1500), [N - 1, 0, N - 1]])
    y_ref, a_ref = oracle.gemm_nvfp4_sampled(x, qw, s8, g, ms, ns)
    got = y_f64(y)[ms, ns]
    assert_parity(got, y_ref, a_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("plan", [dict(path=1, split_k=3), dict(path=2, m_tile=16, dequant_warps=8, split_k=2),
                                  dict(path=2, m_tile=64, split_k=3), dict(path=2, m_tile=256, split_k=2)],
                         ids=lambda p: "-".join(f"{k}{v}" for k, v in p.items()))
def test_debug_bounds_build_runs_clean(W, plan):
    D = W.load_debug_bounds()
    assert D.w4a16_debug_bounds() == 1
    M = 5 if plan["path"] == 1 else 37
    K, N = 1280, 352
    qw, s8, g, x = _case(M, K, N, seed=70 + M)
    y_ref, a_ref = oracle.gemm_nvfp4(x, qw, s8, g)
    s = torch.cuda.current_stream().cuda_stream
    q = torch.from_numpy(qw).cuda()
    sc = torch.from_numpy(s8).cuda()
    qw_r = torch.empty(N * K // 8, dtype=torch.int32, device="cuda")
    sc_r = torch.empty((K // 16) * N, dtype=torch.int16, device="cuda")
    assert D.w4a16_repack_nvfp4(q.data_ptr(), sc.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), N, K, s) == 0
    xd = x_to_dev(x)
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    p = W.Plan(**plan)
    assert D.w4a16_gemm_nvfp4_ex(xd.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), ctypes.c_float(g), y.data_ptr(), M,
                                 N, K, ctypes.byref(p), s) == 0
    torch.cuda.synchronize()
    assert D.w4a16_device_status(s) == 0
    assert_parity(y_f64(y), y_ref, a_ref, "debug-bounds build")


@pytest.mark.parametrize("M", [1, 2])
def test_gemv_batch_depth(W, M):
    """NVFP4 through the GEMV with 8 blocks in flight per warp (a one-wave grid at M <= 2)."""
    K, N = 5120, 5120
    qw, s8, g, x = _case(M, K, N, seed=950 + M)
    r = _dev_weights(W, qw, s8)
    y = _run(W, x, r, g, N, K)
    what = W.w4a16_last_dispatch()
    assert what.startswith("path=gemv") and "unroll=8" in what, what
    y_ref, a_ref = oracle.gemm_nvfp4(x, qw, s8, g)
    assert_parity(y_f64(y), y_ref, a_ref, what)
