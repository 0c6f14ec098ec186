"""W4A8 (int8 activations) on the GPU against the CPU oracle.

"Qwen3.8-27B at 764, 1,035 and 1,623 tok/s" (ai.satyajit.si), section "Where the line bends", runs
the MLP GEMMs with int8 activations; the reading is per-token symmetric int8 with exact integer
group sums. Checked:
  * the quantisation (w4a16_quantize_x_int8) bit for bit against the oracle's binary32 statement:
    every xq, every sx, the fp16 copy, ties, zero rows, heavy tails, rows longer than the
    register-cached length;
  * y on every element at the acceptance bound for the integer GEMV (M <= 8, split-K, ragged
    column tiles, several group sizes) and the tensor-core tiles (M > 8, split-K), fed the oracle's
    own xq and sx, and the full chain quantise -> GEMM;
  * the full-size decode and verify workloads on every element, the batched one sampled;
  * a quantisation that reads the previous GEMM's output (programmatic dependent launch);
  * every W4A8 kernel through the debug-bounds build."""
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


def _weights(W, K, N, G, seed):
    qw, sc = inputs.generate_weights(K, N, G, seed=seed)
    r = W.repack(torch.from_numpy(qw).cuda(), torch.from_numpy(sc.view(np.int16)).cuda(), G)
    return qw, sc, r


def _act(xq, sx):
    """Device copies of oracle activations: (xq int8, xq as fp16, sx fp32)."""
    xq_d = torch.from_numpy(np.ascontiguousarray(xq)).cuda()
    return xq_d, xq_d.to(torch.float16), torch.from_numpy(np.ascontiguousarray(sx)).cuda()


def _run(W, act, r, N, K, G, plan=None):
    y = W.gemm_w4a8(*act, r[0], r[1], N, K, G, plan=plan)
    torch.cuda.synchronize()
    st = W.w4a16_device_status()
    assert st == W.OK, W.status_string(st)
    assert "activations=int8" in W.w4a16_last_dispatch()
    return y


def _quant_rows(M, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float16)
    if M > 1:
        x[1] = np.clip(rng.standard_cauchy(K) * 3, -60000, 60000).astype(np.float16)  # heavy tails
    if M > 2:
        x[2] = 0  # a zero row
    if M > 3:  # amax 127 with ties at .5: rounding to even
        x[3] = np.resize(np.array([127, 2.5, 3.5, -2.5, 0.5, -0.5, 1.5, -126.5], np.float16), K)
    if M > 4:
        x[4] *= np.float16(2.0 ** -12)  # small magnitudes
    return x


@pytest.mark.parametrize("M,K", [(5, 1000), (6, 5120), (3, 17408), (2, 40960), (1, 17408), (70, 5120)])
def test_quantize_matches_oracle_bit_for_bit(W, M, K):
    x = _quant_rows(M, K, seed=K)
    xq_ref, sx_ref = oracle.quantize_x_int8(x.view(np.uint16))
    xq, xh, sx = W.quantize_x_int8(x_to_dev(x.view(np.uint16)))
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(xh.cpu().numpy(), xq_ref.astype(np.float16))
    # without the fp16 copy
    xq2, xh2, sx2 = W.quantize_x_int8(x_to_dev(x.view(np.uint16)), with_f16=False)
    torch.cuda.synchronize()
    assert xh2 is None and np.array_equal(xq2.cpu().numpy(), xq_ref)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("G", [128, 64])
def test_gemv_rows(W, M, G):
    K, N = 1024, 352  # ragged last column tile
    qw, sc, r = _weights(W, K, N, G, seed=100 + M + G)
    x = inputs.generate_x(M, K, seed=200 + M)
    xq, sx = oracle.quantize_x_int8(x)
    y_ref, a_ref = oracle.gemm_w4a8(xq, sx, qw, sc, G)
    act = _act(xq, sx)
    for split in (1, 3, 16):
        y = _run(W, act, r, N, K, G, plan=dict(path=1, split_k=split))
        assert "path=gemv" in W.w4a16_last_dispatch()
        assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


def test_gemv_group_32_and_256(W):
    for G in (32, 256):
        K, N, M = 1024, 160, 4
        qw, sc, r = _weights(W, K, N, G, seed=300 + G)
        x = inputs.generate_x(M, K, seed=301)
        xq, sx = oracle.quantize_x_int8(x)
        y_ref, a_ref = oracle.gemm_w4a8(xq, sx, qw, sc, G)
        y = _run(W, _act(xq, sx), r, N, K, G, plan=dict(path=1, split_k=2))
        assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


TILES = [(16, 128, 4, 16), (64, 256, 2, 16), (128, 128, 2, 16), (256, 128, 1, 16), (16, 128, 4, 8),
         (64, 128, 2, 8)]


@pytest.mark.parametrize("mt,kc,ni,dw", TILES)
def test_tiles(W, mt, kc, ni, dw):
    M, K, N, G = mt + 5 if mt < 256 else 300, 1280 if kc == 128 else 1024, 352, 128
    qw, sc, r = _weights(W, K, N, G, seed=400 + mt + dw)
    x = inputs.generate_x(M, K, seed=401 + mt)
    xq, sx = oracle.quantize_x_int8(x)
    y_ref, a_ref = oracle.gemm_w4a8(xq, sx, qw, sc, G)
    act = _act(xq, sx)
    for split in (1, 3):
        plan = dict(path=2, m_tile=mt, k_chunk=kc, mma_issuers=ni, dequant_warps=dw, split_k=split)
        if dw == 8:
            plan["tmem_stages"] = 2
        y = _run(W, act, r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("M", [1, 4, 8, 9, 16, 37, 130])
def test_quantize_then_gemm_automatic(W, M):
    # the whole W4A8 call sequence on automatic plans against the oracle's own sequence
    K, N, G = 2048, 1056, 128
    qw, sc, r = _weights(W, K, N, G, seed=500 + M)
    x = inputs.generate_x(M, K, seed=501 + M)
    xq_ref, sx_ref = oracle.quantize_x_int8(x)
    y_ref, a_ref = oracle.gemm_w4a8(xq_ref, sx_ref, qw, sc, G)
    act = W.quantize_x_int8(x_to_dev(x))
    y = _run(W, act, r, N, K, G)
    assert ("path=gemv" in W.w4a16_last_dispatch()) == (W.w4a16_plan_for_w4a8(M, N, K, G).path == W.PATH_GEMV)
    assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


def test_zero_rows_and_scales(W):
    K, N, G, M = 512, 128, 128, 4
    qw, sc, r = _weights(W, K, N, G, seed=600)
    x = inputs.generate_x(M, K, seed=601)
    x.view(np.float16)[1] = 0
    xq, sx = oracle.quantize_x_int8(x)
    act = _act(xq, sx)
    for path in (1, 2):
        y = _run(W, act, r, N, K, G, plan=dict(path=path)).float().cpu().numpy()
        assert np.all(y[1] == 0.0)
    r0 = W.repack(torch.from_numpy(qw).cuda(), torch.zeros((K // G, N), dtype=torch.int16, device="cuda"), G)
    for path in (1, 2):
        assert np.all(_run(W, act, r0, N, K, G, plan=dict(path=path)).float().cpu().numpy() == 0.0)


def test_tiles_need_the_fp16_copy(W):
    K, N, G, M = 512, 128, 128, 16
    _, _, r = _weights(W, K, N, G, seed=700)
    xq, xh, sx = W.quantize_x_int8(torch.randn(M, K, device="cuda").half(), with_f16=False)
    with pytest.raises(W.W4A16Error):
        W.gemm_w4a8(xq, None, sx, r[0], r[1], N, K, G)
    y = W.gemm_w4a8(xq[:8], None, sx[:8], r[0], r[1], N, K, G, plan=dict(path=1))  # the GEMV reads int8 only
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK and torch.isfinite(y.float()).all()


@pytest.mark.parametrize("M,K,N", [(1, 5120, 5120), (1, 17408, 5120), (1, 5120, 34816), (8, 5120, 7168),
                                   (16, 5120, 34816)])
def test_full_size_every_element(W, M, K, N):
    G = 128
    qw, sc, r = _weights(W, K, N, G, seed=800 + M)
    x = inputs.generate_x(M, K, seed=801 + M)
    xq, sx = oracle.quantize_x_int8(x)
    y_ref, a_ref = oracle.gemm_w4a8(xq, sx, qw, sc, G)
    act = W.quantize_x_int8(x_to_dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(act[0].cpu().numpy(), xq)
    y = _run(W, act, r, N, K, G)
    assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


def test_batched_sampled(W):
    M, K, N, G = 256, 5120, 34816, 128
    qw, sc, r = _weights(W, K, N, G, seed=900)
    x = inputs.generate_x(M, K, seed=901)
    act = W.quantize_x_int8(x_to_dev(x))
    y = _run(W, act, r, N, K, G)
    xq, sx = oracle.quantize_x_int8(x)
    rng = np.random.default_rng(902)
    ms = np.concatenate([rng.integers(0, M, 1500), [0, M - 1, M - 1]])
    ns = np.concatenate([rng.integers(0, N, 1500), [N - 1, 0, N - 1]])
    y_ref, a_ref = oracle.gemm_w4a8_sampled(xq, sx, qw, sc, G, ms, ns)
    assert_parity(y_f64(y)[ms, ns], y_ref, a_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("M", [1, 16])
def test_quantize_reads_previous_gemm_output(W, M):
    # y1 = W4A16 GEMM -> quantise y1 -> W4A8 GEMM on one stream, the intermediate buffers NaN-filled
    # first: the quantisation (launched with programmatic dependent launch) must see y1 complete
    K1, N1, N2, G = 1024, 2048, 512, 128
    qw1, sc1, r1 = _weights(W, K1, N1, G, seed=1000)
    qw2, sc2, r2 = _weights(W, N1, N2, G, seed=1001)
    x = inputs.generate_x(M, K1, seed=1002)
    y1 = torch.full((M, N1), float("nan"), dtype=torch.float16, device="cuda")
    xq = torch.full((M, N1), 77, dtype=torch.int8, device="cuda")
    xh = torch.full((M, N1), float("nan"), dtype=torch.float16, device="cuda")
    sx = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    y2 = torch.full((M, N2), float("nan"), dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    W.gemm(x_to_dev(x), *r1, N1, K1, G, y=y1)
    W.quantize_x_int8(y1, out=(xq, xh, sx))
    W.gemm_w4a8(xq, xh, sx, *r2, N2, N1, G, y=y2)
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    y1_bits = y1.cpu().numpy().view(np.uint16)
    xq_ref, sx_ref = oracle.quantize_x_int8(y1_bits)
    assert np.array_equal(xq.cpu().numpy(), xq_ref) and np.array_equal(sx.cpu().numpy(), sx_ref)
    y_ref, a_ref = oracle.gemm_w4a8(xq_ref, sx_ref, qw2, sc2, G)
    assert_parity(y_f64(y2), y_ref, a_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("plan", [dict(path=1, split_k=3), dict(path=2, m_tile=16, dequant_warps=8, split_k=2),
                                  dict(path=2, m_tile=256, split_k=2)],
                         ids=lambda p: "-".join(f"{k}{v}" for k, v in p.items()))
def test_debug_bounds_build_runs_clean(W, plan):
    D = W.load_debug_bounds()
    assert D.w4a16_debug_bounds() == 1
    M = 5 if plan["path"] == 1 else 37
    K, N, G = 1280, 352, 128
    qw, sc, r = _weights(W, K, N, G, seed=1100 + M)
    x = inputs.generate_x(M, K, seed=1101)
    xq_ref, sx_ref = oracle.quantize_x_int8(x)
    y_ref, a_ref = oracle.gemm_w4a8(xq_ref, sx_ref, qw, sc, G)
    s = torch.cuda.current_stream().cuda_stream
    xd = x_to_dev(x)
    xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    xh = torch.empty((M, K), dtype=torch.float16, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    assert D.w4a16_quantize_x_int8(xd.data_ptr(), xq.data_ptr(), xh.data_ptr(), sx.data_ptr(), M, K, s) == 0
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    p = W.Plan(**plan)
    assert D.w4a16_gemm_w4a8_ex(xq.data_ptr(), xh.data_ptr(), sx.data_ptr(), r[0].data_ptr(), r[1].data_ptr(),
                                y.data_ptr(), M, N, K, G, ctypes.byref(p), s) == 0
    torch.cuda.synchronize()
    assert D.w4a16_device_status(s) == 0
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert_parity(y_f64(y), y_ref, a_ref, "debug-bounds build")


@pytest.mark.parametrize("M", [1, 2, 3, 16])
@pytest.mark.parametrize("split", [0, 1, 3, 16])
def test_quantize_gemm_in_one_call(W, M, split):
    # w4a16_quantize_gemm_w4a8: quantisation kernel + GEMM in one call; xq / sx bit-exact
    K, N, G = 2048, 352, 128
    if split and M > 8:
        pytest.skip("explicit GEMV splits apply to M <= 8")
    qw, sc, r = _weights(W, K, N, G, seed=1200 + M)
    x = inputs.generate_x(M, K, seed=1201 + M)
    x.view(np.float16)[0, :7] = np.array([0.5, 1.5, -2.5, 3.5, 0, 0, 0], np.float16) * (np.abs(
        x.view(np.float16)[0]).max() / np.float16(127))
    xq_ref, sx_ref = oracle.quantize_x_int8(x)
    y_ref, a_ref = oracle.gemm_w4a8(xq_ref, sx_ref, qw, sc, G)
    plan = dict(path=1, split_k=split) if split else None
    y, (xq, xh, sx) = W.quantize_gemm_w4a8(x_to_dev(x), r[0], r[1], N, K, G, plan=plan)
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    desc = W.w4a16_last_dispatch()
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(xh.cpu().numpy(), xq_ref.astype(np.float16))
    assert_parity(y_f64(y), y_ref, a_ref, desc)


@pytest.mark.parametrize("K", [5120, 17408])
def test_quantize_gemm_in_one_call_full_size_and_zero_row(W, K):
    # (the GEMV path needs no fp16 copy of the codes)
    N, G, M = 5120, 128, 2
    qw, sc, r = _weights(W, K, N, G, seed=1300 + K)
    x = inputs.generate_x(M, K, seed=1301)
    x.view(np.float16)[1] = 0
    xq_ref, sx_ref = oracle.quantize_x_int8(x)
    y_ref, a_ref = oracle.gemm_w4a8(xq_ref, sx_ref, qw, sc, G)
    y, (xq, xh, sx) = W.quantize_gemm_w4a8(x_to_dev(x), r[0], r[1], N, K, G, with_f16=False)
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK and xh is None
    assert "path=gemv" in W.w4a16_last_dispatch()
    assert np.array_equal(xq.cpu().numpy(), xq_ref) and sx.cpu().numpy()[1] == 0.0
    assert np.all(y.float().cpu().numpy()[1] == 0.0)
    assert_parity(y_f64(y), y_ref, a_ref, W.w4a16_last_dispatch())


def test_quantize_gemm_reads_previous_gemm_output(W):
    # W4A16 GEMM -> quantise-and-multiply -> W4A8 GEMM of the same codes, NaN-filled first
    M, K1, N1, N2, N3, G = 2, 1024, 2048, 512, 256, 128
    qw1, sc1, r1 = _weights(W, K1, N1, G, seed=1400)
    qw2, sc2, r2 = _weights(W, N1, N2, G, seed=1401)
    qw3, sc3, r3 = _weights(W, N1, N3, G, seed=1402)
    x = inputs.generate_x(M, K1, seed=1403)
    y1 = torch.full((M, N1), float("nan"), dtype=torch.float16, device="cuda")
    out = (torch.full((M, N1), 55, dtype=torch.int8, device="cuda"), None,
           torch.full((M,), float("nan"), dtype=torch.float32, device="cuda"))
    y2 = torch.full((M, N2), float("nan"), dtype=torch.float16, device="cuda")
    y3 = torch.full((M, N3), float("nan"), dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    W.gemm(x_to_dev(x), *r1, N1, K1, G, y=y1)
    W.quantize_gemm_w4a8(y1, *r2, N2, N1, G, out=out, y=y2)
    W.gemm_w4a8(*out, *r3, N3, N1, G, y=y3)
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    xq_ref, sx_ref = oracle.quantize_x_int8(y1.cpu().numpy().view(np.uint16))
    assert np.array_equal(out[0].cpu().numpy(), xq_ref) and np.array_equal(out[2].cpu().numpy(), sx_ref)
    for yk, qwk, sck in ((y2, qw2, sc2), (y3, qw3, sc3)):
        y_ref, a_ref = oracle.gemm_w4a8(xq_ref, sx_ref, qwk, sck, G)
        assert_parity(y_f64(yk), y_ref, a_ref, "chain")


def test_quantize_gemm_debug_bounds(W):
    D = W.load_debug_bounds()
    M, K, N, G = 2, 1280, 352, 128
    qw, sc, r = _weights(W, K, N, G, seed=1500)
    x = inputs.generate_x(M, K, seed=1501)
    xq_ref, sx_ref = oracle.quantize_x_int8(x)
    y_ref, a_ref = oracle.gemm_w4a8(xq_ref, sx_ref, qw, sc, G)
    s = torch.cuda.current_stream().cuda_stream
    xd = x_to_dev(x)
    xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    xh = torch.empty((M, K), dtype=torch.float16, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    p = W.Plan(path=1, split_k=3)
    assert D.w4a16_quantize_gemm_w4a8(xd.data_ptr(), xq.data_ptr(), xh.data_ptr(), sx.data_ptr(), r[0].data_ptr(),
                                      r[1].data_ptr(), y.data_ptr(), M, N, K, G, ctypes.byref(p), s) == 0
    torch.cuda.synchronize()
    assert D.w4a16_device_status(s) == 0
    assert np.array_equal(xq.cpu().numpy(), xq_ref) and np.array_equal(xh.cpu().numpy(), xq_ref.astype(np.float16))
    assert_parity(y_f64(y), y_ref, a_ref, "debug-bounds build")


def test_quantize_near_half_integers(W):
    # activations at and beside every (k + 1/2) * sx, for several row scales: the codes must equal the
    # oracle's rne(fl32(x / sx)) wherever the quotient lies within rounding of a half-integer
    rng = np.random.default_rng(1600)
    rows = []
    for amax in np.concatenate([[127.0, 1.0, 0.1], rng.uniform(0.01, 3000.0, 13)]).astype(np.float16):
        sx = np.float32(np.float32(amax) / np.float32(127))
        vals = [amax]
        for k in range(-127, 127):
            c = np.float16((k + 0.5) * float(sx))
            vals += [c, np.nextafter(c, np.float16(np.inf)), np.nextafter(c, np.float16(-np.inf))]
        v = np.array(vals, np.float16)
        v = v[np.abs(v.astype(np.float32)) <= np.float32(amax)]
        rows.append(v)
    K = ((max(len(r) for r in rows) + 7) // 8) * 8
    x = np.zeros((len(rows), K), np.float16)
    for i, r in enumerate(rows):
        x[i, :len(r)] = r
    xq_ref, sx_ref = oracle.quantize_x_int8(x.view(np.uint16))
    xq, xh, sx = W.quantize_x_int8(x_to_dev(x.view(np.uint16)))
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))
    bad = np.argwhere(xq.cpu().numpy() != xq_ref)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"
