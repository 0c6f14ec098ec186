"""The persistent stream-K kernel (w4a16_gemm_ws, M <= 64) against the CPU oracle, element by element.

Bound (every element): |y - y_ref| <= 2^-10 |y_ref| + 2^-10 sum_k |x w|, y finite. The CTA counts
below cut the (tile, chunk) units so that tiles are whole in one CTA, shared by two, or spread over
many CTAs (the partial tiles summed through the workspace by the last CTA to finish); ragged last
tiles, group sizes, one-hot exactness, determinism, workspace reuse and guard bands are covered."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import assert_parity, lib, to_dev, y_f64

pytestmark = pytest.mark.gpu

WS_BYTES = 64 << 20


@pytest.fixture(scope="module")
def W():
    return lib()


@pytest.fixture(scope="module")
def ws(W):
    return W.new_workspace(WS_BYTES)


def _case(M, K, N, G, seed):
    d = inputs.generate(M, K, N, G, seed=seed)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    return d, y_ref, abs_ref


def _repacked(W, d, G):
    x, qw, sc = to_dev(d)
    qw_r, sc_r = W.repack(qw, sc, G)
    return x, qw_r, sc_r


def _run(W, x, qw_r, sc_r, N, K, G, ws, plan=None, y=None):
    y = W.gemm(x, qw_r, sc_r, N, K, G, plan=plan, workspace=ws, y=y)
    torch.cuda.synchronize()
    st = W.w4a16_device_status()
    assert st == W.OK, W.status_string(st)
    return y


SK_TILES = [(16, 128), (16, 256), (32, 128), (32, 256), (64, 128), (64, 256)]


@pytest.mark.parametrize("mt,kc", SK_TILES)
def test_every_streamk_tile(W, ws, mt, kc):
    # 3 column tiles (the last one 96 wide) x 1280/kc chunks: CTA counts from one CTA for everything
    # to one unit per CTA
    K, N, G = 1280, 352, 128
    for M in sorted({1, mt - 3, mt}):
        d, y_ref, abs_ref = _case(M, K, N, G, seed=mt + kc + M)
        x, qw_r, sc_r = _repacked(W, d, G)
        units = 3 * (K // kc)
        for ctas in sorted({1, 2, 3, 4, 7, units - 1, units}):
            plan = dict(path=3, m_tile=mt, k_chunk=kc, ctas=ctas)
            y = _run(W, x, qw_r, sc_r, N, K, G, ws, plan)
            assert "path=streamk" in W.w4a16_last_dispatch()
            assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("stages", [2, 3, 5, 16])
def test_ring_depths(W, ws, stages):
    M, K, N, G = 16, 2560, 256, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=40 + stages)
    x, qw_r, sc_r = _repacked(W, d, G)
    for kc in (128, 256):
        plan = dict(path=3, m_tile=16, k_chunk=kc, stages=stages, ctas=5)
        y = _run(W, x, qw_r, sc_r, N, K, G, ws, plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("G", [32, 64, 256, 512])
def test_group_sizes(W, ws, G):
    M, K, N = 7, 2048, 160
    d, y_ref, abs_ref = _case(M, K, N, G, seed=G + 1)
    x, qw_r, sc_r = _repacked(W, d, G)
    for kc in (128, 256):
        for ctas in (1, 3, 11):
            y = _run(W, x, qw_r, sc_r, N, K, G, ws, dict(path=3, k_chunk=kc, ctas=ctas))
            assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 15, 16, 17, 31, 33, 48, 63, 64])
def test_automatic_plan_rows(W, ws, M):
    K, N, G = 1536, 480, 128  # 4 tiles, the last 96 wide; 6 or 12 chunks per tile
    d, y_ref, abs_ref = _case(M, K, N, G, seed=200 + M)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = _run(W, x, qw_r, sc_r, N, K, G, ws)
    assert "path=streamk" in W.w4a16_last_dispatch()
    assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_one_hot_rows_are_exact(W, ws):
    K, N, G = 1024, 256, 128
    d = inputs.generate(1, K, N, G, seed=21)
    ks = [0, 7, 8, 127, 128, 255, 256, 511, 512, K - 1]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    d["x"] = x.view(np.uint16)
    w = oracle.dequant(d["qweight"], d["scales"], G)
    expect = np.stack([w[k] for k in ks]).astype(np.float16)
    xd, qw_r, sc_r = _repacked(W, d, G)
    for plan in (dict(path=3, ctas=1), dict(path=3, ctas=3), dict(path=3, k_chunk=128, ctas=16)):
        y = _run(W, xd, qw_r, sc_r, N, K, G, ws, plan).cpu().numpy()
        assert np.array_equal(y.view(np.uint16), expect.view(np.uint16)), W.w4a16_last_dispatch()


def test_zero_scales_give_zero(W, ws):
    M, K, N, G = 9, 1024, 128, 128
    d = inputs.generate(M, K, N, G, seed=22)
    d["scales"] = np.zeros_like(d["scales"])
    x, qw_r, sc_r = _repacked(W, d, G)
    for ctas in (1, 5):
        y = _run(W, x, qw_r, sc_r, N, K, G, ws, dict(path=3, ctas=ctas))
        assert torch.count_nonzero(y.float()).item() == 0


@pytest.mark.parametrize("qv", [0, 15])
def test_extreme_nibbles_and_large_x(W, ws, qv):
    M, K, N, G = 6, 1024, 128, 128
    d = inputs.generate(M, K, N, G, seed=23)
    d["qweight"] = inputs.pack_nibbles(np.full((K, N), qv, np.uint8))
    rng = np.random.default_rng(qv)
    d["x"] = rng.choice([-8.0, 8.0], size=(M, K)).astype(np.float16).view(np.uint16)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    x, qw_r, sc_r = _repacked(W, d, G)
    for ctas in (1, 6):
        y = _run(W, x, qw_r, sc_r, N, K, G, ws, dict(path=3, ctas=ctas))
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_deterministic_repeats_and_workspace_reuse(W, ws):
    # the same workspace through many calls in stream order (the tile counters must come back to
    # zero after every call), bit-identical results, also on another stream
    M, K, N, G = 16, 5120, 1024, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=24)
    x, qw_r, sc_r = _repacked(W, d, G)
    plan = dict(path=3, ctas=37)  # 8 tiles x 20 chunks over 37 CTAs: every tile split
    y0 = _run(W, x, qw_r, sc_r, N, K, G, ws, plan)
    assert_parity(y_f64(y0), y_ref, abs_ref, W.w4a16_last_dispatch())
    ys = [W.gemm(x, qw_r, sc_r, N, K, G, plan=plan, workspace=ws) for _ in range(50)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ys.append(W.gemm(x, qw_r, sc_r, N, K, G, plan=plan, workspace=ws, stream=s))
    s.synchronize()
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    for y in ys:
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


def test_one_workspace_for_every_shape(W):
    # one workspace through calls of different row tiles and widths in stream order: a call's
    # partial tiles never land on another call's counters
    ws = W.new_workspace(WS_BYTES)
    cases = []
    for (M, K, N, seed) in [(64, 2048, 640, 60), (3, 2048, 4096, 61), (33, 4096, 256, 62), (16, 4096, 1536, 63)]:
        d, y_ref, abs_ref = _case(M, K, N, 128, seed)
        cases.append((d, y_ref, abs_ref, _repacked(W, d, 128), K, N))
    for _ in range(3):
        for (d, y_ref, abs_ref, (x, qw_r, sc_r), K, N) in cases:
            y = _run(W, x, qw_r, sc_r, N, K, 128, ws, dict(path=3, ctas=29))
            assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_counters_clean_after_calls(W):
    M, K, N, G = 5, 2048, 384, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=25)
    x, qw_r, sc_r = _repacked(W, d, G)
    need = W.w4a16_workspace_bytes(M, N, K, G)
    assert need > 0
    ws = W.new_workspace(need)
    for ctas in (2, 5, 7, 24):
        y = _run(W, x, qw_r, sc_r, N, K, G, ws, dict(path=3, ctas=ctas))
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())
        cnt = ws[:256 * 1024].cpu().numpy().view(np.uint32)  # the counter zone
        assert not cnt.any(), f"tile counters left non-zero after ctas={ctas}"


@pytest.mark.parametrize("ctas", [1, 3, 10])
def test_no_writes_outside_y_and_workspace(W, ctas):
    M, K, N, G = 13, 1024, 352, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=52 + ctas)
    x, qw_r, sc_r = _repacked(W, d, G)
    pad = 4096
    canary = 0x7BAD
    buf = torch.full((M * N + 2 * pad,), canary, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + M * N].view(torch.float16).view(M, N)
    plan = W.Plan(path=3, ctas=ctas)
    # the workspace this plan needs (256 KiB of counters, then ctas x 2 x 16 x 128 fp32), between guard bands
    need = 256 * 1024 + ctas * 2 * 16 * 128 * 4
    wbuf = torch.zeros(need + 2 * 8192, dtype=torch.uint8, device="cuda")
    wbuf[:8192] = 0xA5
    wbuf[8192 + need:] = 0xA5
    ws = wbuf[8192:8192 + need]
    rc = W.w4a16_gemm_ws(x.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), y.data_ptr(), M, N, K, G, plan,
                         ws.data_ptr(), need, torch.cuda.current_stream().cuda_stream)
    assert rc == W.OK
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    host = buf.cpu().numpy().view(np.uint16)
    assert (host[:pad] == canary).all() and (host[pad + M * N:] == canary).all()
    wh = wbuf.cpu().numpy()
    assert (wh[:8192] == 0xA5).all() and (wh[8192 + need:] == 0xA5).all()
    assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_workspace_checks(W):
    M, K, N, G = 4, 1024, 256, 128
    d, _, _ = _case(M, K, N, G, seed=26)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    need = W.w4a16_workspace_bytes(M, N, K, G)
    ws = W.new_workspace(need)
    s = torch.cuda.current_stream().cuda_stream
    args = (x.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), y.data_ptr(), M, N, K, G)
    assert W.w4a16_gemm_ws(*args, None, ws.data_ptr(), need - 16, s) == W.ERR_INVALID_ARG  # too small
    assert W.w4a16_gemm_ws(*args, None, ws.data_ptr() + 8, need, s) == W.ERR_MISALIGNED
    assert W.w4a16_gemm_ws(*args, None, y.data_ptr(), need, s) == W.ERR_INVALID_ARG  # overlaps y
    assert W.w4a16_gemm_ex(*args, W.Plan(path=3), s) == W.ERR_INVALID_ARG  # stream-K needs a workspace
    assert W.w4a16_gemm_ws(*args, W.Plan(path=3, m_tile=16, ctas=10 ** 5), ws.data_ptr(), need, s) != W.OK
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
