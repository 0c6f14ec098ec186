"""W4A16 GEMM on the GPU against the CPU oracle, element by element.

Bound (every element): |y - y_ref| <= 2^-10 |y_ref| + 2^-10 sum_k |x w|, y finite. One-hot rows
and zero scales are bit-exact. Small shapes span several column tiles, K chunks, cluster splits
and a ragged last tile; the single-configuration workloads run at full size on every element, the
layer sweep on every element up to M = 64 and on samples above."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import assert_parity, lib, run_gemm, to_dev, x_to_dev, y_f64

pytestmark = pytest.mark.gpu


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


# ------------------------------------------------------------------------------ oracle-scale workload
ORACLE_SCALE_PLANS = [
    None,
    dict(path=1), dict(path=1, split_k=1), dict(path=1, split_k=2), dict(path=1, split_k=5), dict(path=1, split_k=16),
    dict(path=2), dict(path=2, m_tile=16, k_chunk=128, stages=3, split_k=1),
    dict(path=2, m_tile=16, k_chunk=256, stages=4, split_k=2), dict(path=2, m_tile=16, k_chunk=128, stages=2, split_k=3),
    dict(path=2, m_tile=16, k_chunk=128, stages=3, split_k=8), dict(path=2, m_tile=32, k_chunk=128, stages=6, split_k=8),
]


def plan_id(p):
    if p is None:
        return "auto"
    name = {1: "gemv", 2: "tc"}.get(p.get("path", 0), "auto")
    return name + "".join(f"-{k[0]}{v}" for k, v in p.items() if k != "path")


@pytest.mark.parametrize("plan", ORACLE_SCALE_PLANS, ids=plan_id)
def test_oracle_scale_workload(W, plan):
    M, K, N, G = 4, 1024, 1024, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=0)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
    assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


# ------------------------------------------------------------------------------ ragged / edge shapes
EDGE_M = [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 63, 65, 127, 129, 200, 257, 513]


@pytest.fixture(scope="module")
def edge_matrix(W):
    K, N, G = 640, 352, 128  # 5 chunks of 128 (uneven splits), 3 column tiles, the last one 96 wide
    d = inputs.generate(max(EDGE_M), K, N, G, seed=11)
    x_all, qw_r, sc_r = _repacked(W, d, G)
    return d, x_all, qw_r, sc_r, K, N, G


@pytest.mark.parametrize("M", EDGE_M)
def test_edge_rows_tc(W, edge_matrix, M):
    d, x_all, qw_r, sc_r, K, N, G = edge_matrix
    y_ref, abs_ref = oracle.gemm(d["x"][:M], d["qweight"], d["scales"], G)
    x = x_all[:M].contiguous()
    for plan in (None, dict(path=2, split_k=1), dict(path=2, split_k=5)):
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("M", [m for m in EDGE_M if m <= 8])
def test_edge_rows_gemv(W, edge_matrix, M):
    d, x_all, qw_r, sc_r, K, N, G = edge_matrix
    y_ref, abs_ref = oracle.gemm(d["x"][:M], d["qweight"], d["scales"], G)
    x = x_all[:M].contiguous()
    for split in (1, 3, 16):
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=dict(path=1, split_k=split))
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


# every instantiated (m_tile, k_chunk, mma_issuers) kernel
TC_TILES = [(16, 128, 4), (16, 256, 4), (32, 128, 4), (32, 256, 4), (64, 128, 4), (64, 256, 4), (64, 256, 2),
            (128, 128, 2), (128, 128, 1), (256, 128, 1)]


@pytest.mark.parametrize("mt,kc,ni", TC_TILES)
def test_every_tc_tile(W, mt, kc, ni):
    M, K, N, G = mt - 3, 1024, 352, 128  # ragged last column tile (96 wide)
    d, y_ref, abs_ref = _case(M, K, N, G, seed=mt + kc + ni)
    x, qw_r, sc_r = _repacked(W, d, G)
    for split in (1, 3):
        for ts in (2, 3):
            if ts * kc // 2 + ni * mt > 512:
                continue
            plan = dict(path=2, m_tile=mt, k_chunk=kc, split_k=split, tmem_stages=ts, mma_issuers=ni)
            y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
            assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_shallow_and_deep_rings(W):
    M, K, N, G = 16, 2048, 256, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=31)
    x, qw_r, sc_r = _repacked(W, d, G)
    for (kc, st, ts) in [(128, 2, 2), (128, 16, 6), (128, 7, 3), (256, 2, 2), (256, 5, 3)]:
        plan = dict(path=2, m_tile=16, k_chunk=kc, stages=st, tmem_stages=ts, split_k=1)
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("G", [32, 64, 256])
def test_group_sizes(W, G):
    M, K, N = 5, 1024, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=G)
    x, qw_r, sc_r = _repacked(W, d, G)
    plans = [dict(path=1), dict(path=2, k_chunk=128, stages=4), dict(path=2, k_chunk=128, stages=3, split_k=2),
             dict(path=2, k_chunk=256, split_k=2)]
    for plan in plans:
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("G,K", [(96, 1920), (160, 1920), (64, 1216)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_shapes_the_tiles_cannot_stage(W, G, K, M):
    # group sizes that do not fit a 128-k stage, and K = 64 mod 128: automatic plans send these to
    # the GEMV, which works in 32-k rows with one scale each
    N = 160
    d, y_ref, abs_ref = _case(M, K, N, G, seed=G + M)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = run_gemm(W, x, qw_r, sc_r, N, K, G)
    assert "path=gemv" in W.w4a16_last_dispatch()
    assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_host_buffer_entry_point(W):
    M, K, N, G = 3, 1280, 352, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=90)
    x_dev, qw, sc = to_dev(d)
    qw_r, sc_r = W.repack(qw, sc, G)
    x_host = x_dev.cpu().pin_memory()
    y_host = torch.zeros((M, N), dtype=torch.float16).pin_memory()
    x_buf = torch.empty_like(x_dev)
    y_buf = torch.empty((M, N), dtype=torch.float16, device="cuda")
    W.gemm_host(x_host, x_buf, qw_r, sc_r, y_buf, y_host, N, K, G)
    torch.cuda.synchronize()
    assert_parity(y_f64(y_host), y_ref, abs_ref, W.w4a16_last_dispatch())
    y_dev = W.gemm(x_dev, qw_r, sc_r, N, K, G)  # the same plan on device buffers: the same bits
    assert torch.equal(y_dev.cpu().view(torch.int16), y_host.view(torch.int16))
    both = torch.zeros(M * K + M * N, dtype=torch.float16).pin_memory()
    with pytest.raises(W.W4A16Error):  # host buffers overlapping
        W.gemm_host(both[: M * K].view(M, K), x_buf, qw_r, sc_r, y_buf, both[: M * N].view(M, N), N, K, G)
    with pytest.raises(W.W4A16Error):  # a device buffer as x_host
        W.gemm_host(x_dev, x_buf, qw_r, sc_r, y_buf, y_host, N, K, G)


@pytest.fixture(scope="module")
def output_head(W):
    # the output-head matrix K x N = 5120 x 248320 (636 MB packed), generated once for both row counts
    (_, K, N, seed), = inputs.WORKLOADS["output_head"]
    qweight, scales = inputs.generate_weights(K, N, 128, seed=seed)
    qw_r, sc_r = W.repack(torch.from_numpy(qweight).cuda(), torch.from_numpy(scales.view(np.int16)).cuda(), 128)
    return K, N, seed, qweight, scales, qw_r, sc_r


@pytest.mark.parametrize("M", [1, 16])
def test_output_head_sampled(W, output_head, M):
    K, N, seed, qweight, scales, qw_r, sc_r = output_head
    x = inputs.generate_x(M, K, seed + M)
    y = y_f64(run_gemm(W, x_to_dev(x), qw_r, sc_r, N, K, 128))
    rng = np.random.default_rng(M)
    ns = np.concatenate([rng.integers(0, N, 240), np.arange(N - 8, N)])  # the last tile too
    ms = rng.integers(0, M, ns.size)
    y_ref, abs_ref = oracle.gemm_sampled(x, qweight, scales, 128, ms, ns)
    assert_parity(y[ms, ns], y_ref, abs_ref, W.w4a16_last_dispatch())


# ------------------------------------------------------------------------------ exact cases
def test_one_hot_rows_are_exact(W):
    K, N, G = 512, 256, 128
    d = inputs.generate(1, K, N, G, seed=21)
    ks = [0, 7, 8, 127, 128, 255, 256, K - 1]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    d["x"] = x.view(np.uint16)
    w = oracle.dequant(d["qweight"], d["scales"], G)
    expect = np.stack([w[k] for k in ks]).astype(np.float16)  # every w is an fp16 value
    xd, qw_r, sc_r = _repacked(W, d, G)
    plans = [dict(path=1, split_k=1), dict(path=1, split_k=4), dict(path=2, split_k=1), dict(path=2, split_k=4),
             dict(path=2, m_tile=16, k_chunk=128, stages=4, split_k=4)]
    for plan in plans:
        y = run_gemm(W, xd, qw_r, sc_r, N, K, G, plan=plan).cpu().numpy()
        assert np.array_equal(y.view(np.uint16), expect.view(np.uint16)), W.w4a16_last_dispatch()


def test_zero_scales_give_zero(W):
    M, K, N, G = 9, 512, 128, 128
    d = inputs.generate(M, K, N, G, seed=22)
    d["scales"] = np.zeros_like(d["scales"])
    x, qw_r, sc_r = _repacked(W, d, G)
    for plan in (dict(path=1), dict(path=2), dict(path=2, split_k=4)):
        if plan["path"] == 1:
            y = run_gemm(W, x[:8].contiguous(), qw_r, sc_r, N, K, G, plan=plan)
        else:
            y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert torch.count_nonzero(y.float()).item() == 0


@pytest.mark.parametrize("qv", [0, 15])
def test_extreme_nibbles_and_large_x(W, qv):
    M, K, N, G = 6, 512, 128, 128
    d = inputs.generate(M, K, N, G, seed=23)
    q = np.full((K, N), qv, np.uint8)
    d["qweight"] = inputs.pack_nibbles(q)
    rng = np.random.default_rng(qv)
    d["x"] = (rng.choice([-8.0, 8.0], size=(M, K))).astype(np.float16).view(np.uint16)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    x, qw_r, sc_r = _repacked(W, d, G)
    for plan in (dict(path=1), dict(path=2), dict(path=2, split_k=4)):
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


def test_deterministic_and_stream_ordered(W):
    M, K, N, G = 16, 2048, 512, 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=24)
    x, qw_r, sc_r = _repacked(W, d, G)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y1 = W.gemm(x, qw_r, sc_r, N, K, G, plan=dict(path=2, split_k=4), stream=s)
        y2 = W.gemm(x, qw_r, sc_r, N, K, G, plan=dict(path=2, split_k=4), stream=s)
    s.synchronize()
    assert W.w4a16_device_status(s.cuda_stream) == W.OK
    assert torch.equal(y1, y2)
    assert_parity(y_f64(y1), y_ref, abs_ref, "non-default stream")


# ------------------------------------------------------------------------------ full-size workloads
FULL = [(M, K, N, seed) for name in ("decode_gemv", "spec_verify", "batched_verify")
        for (M, K, N, seed) in inputs.WORKLOADS[name]]


@pytest.mark.parametrize("M,K,N,seed", FULL)
def test_full_size_workloads(W, M, K, N, seed):
    """The bench's single-configuration workloads at full size, in the automatic launch plan the
    bench times, compared with the oracle on EVERY element (the verify output 16 x 34816, the
    batched ones 256 x 34816 and 256 x 5120)."""
    G = inputs.GROUP
    d = inputs.generate(M, K, N, G, seed=seed)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = y_f64(run_gemm(W, x, qw_r, sc_r, N, K, G))
    assert np.all(np.isfinite(y))
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    assert_parity(y, y_ref, abs_ref, W.w4a16_last_dispatch())


def test_layer_sweep_all_rows(W):
    """Every matrix of the dense-layer sweep at every M, automatic plan: every element up to
    M = 64, 2000 sampled elements (and the four corners) above."""
    G = inputs.GROUP
    rng = np.random.default_rng(4)
    for name, K, N in inputs.SWEEP_MATRICES:
        qweight, scales = inputs.generate_weights(K, N, G, seed=inputs.SWEEP_SEED)
        qw = torch.from_numpy(qweight).cuda()
        sc = torch.from_numpy(scales.view(np.int16)).cuda()
        qw_r, sc_r = W.repack(qw, sc, G)
        for M in inputs.SWEEP_M:
            xb = inputs.generate_x(M, K, seed=1000 + M)
            y = y_f64(run_gemm(W, x_to_dev(xb), qw_r, sc_r, N, K, G))
            what = f"{name} M={M}: {W.w4a16_last_dispatch()}"
            assert np.all(np.isfinite(y)), what
            if M <= 64:
                y_ref, abs_ref = oracle.gemm(xb, qweight, scales, G)
                assert_parity(y, y_ref, abs_ref, what)
                continue
            ms = np.concatenate([[0, 0, M - 1, M - 1], rng.integers(0, M, 2000)])
            ns = np.concatenate([[0, N - 1, 0, N - 1], rng.integers(0, N, 2000)])
            y_ref, abs_ref = oracle.gemm_sampled(xb, qweight, scales, G, ms, ns)
            assert_parity(y[ms, ns], y_ref, abs_ref, what)


def test_status_word_clean(W):
    assert W.w4a16_device_status() == W.OK


# the half-size tile kernels (8 dequant warps, two CTAs per SM)
@pytest.mark.parametrize("mt,ni", [(16, 4), (32, 4), (64, 2)])
def test_half_size_tiles(W, mt, ni):
    M, K, N, G = mt - 3, 1280, 352, 128  # ragged last column tile (96 wide), 10 chunks of 128
    d, y_ref, abs_ref = _case(M, K, N, G, seed=70 + mt)
    x, qw_r, sc_r = _repacked(W, d, G)
    for split in (1, 3):
        for ts in (2, 3):
            if ts * 64 + ni * mt > 256:
                continue
            plan = dict(path=2, m_tile=mt, k_chunk=128, split_k=split, tmem_stages=ts, mma_issuers=ni,
                        dequant_warps=8)
            y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
            assert "dequant_warps=8" in W.w4a16_last_dispatch()
            assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


# ------------------------------------------------------------------------------ partial last wave
# Work items of 128 columns x 256 rows that overfill whole waves of one CTA per SM: the items of the
# last, partial wave run as a second launch whose clusters split each of them along K.
TAIL_SAMPLED = [(1024, 5120, 5120), (1000, 5120, 5088), (1024, 17408, 5120), (1024, 5120, 7168), (1024, 5120, 34816)]


def _tail_samples(M, N, rng):
    """Every column of the last two column tiles on rows of every row tile, plus random elements."""
    cols = np.arange(max(0, N - 256), N)
    rows = np.array(sorted({0, 1, 255, 256, 511, 512, 767, 768, min(M - 1, 900), M - 1} & set(range(M))))
    ms = np.concatenate([np.repeat(rows, len(cols)), rng.integers(0, M, 2000)])
    ns = np.concatenate([np.tile(cols, len(rows)), rng.integers(0, N, 2000)])
    return ms, ns


@pytest.mark.parametrize("M,K,N", TAIL_SAMPLED)
def test_partial_wave_tail_sampled(W, M, K, N):
    """Automatic plans of the layer shapes at M = 1000-1024 (a tail in each; the first with ragged
    rows and a 96-column last tile)."""
    G = inputs.GROUP
    d = inputs.generate(M, K, N, G, seed=M + K + N)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = y_f64(run_gemm(W, x, qw_r, sc_r, N, K, G))
    what = W.w4a16_last_dispatch()
    assert "tail_items=" in what, what
    assert np.all(np.isfinite(y))
    ms, ns = _tail_samples(M, N, np.random.default_rng(M + N))
    y_ref, abs_ref = oracle.gemm_sampled(d["x"], d["qweight"], d["scales"], G, ms, ns)
    assert_parity(y[ms, ns], y_ref, abs_ref, what)


@pytest.mark.parametrize("M,K,N,split,tails", [(200, 256, 19552, 1, (2,)), (300, 1024, 10112, 1, (2, 3, 8)),
                                               (129, 512, 19584, 1, (4,)), (200, 512, 19552, 2, (4,))])
def test_partial_wave_tail_every_element(W, M, K, N, split, tails):
    """Explicit tail plans on shapes the oracle multiplies in full: 153 or 158 work items (one or
    six in the tail), ragged rows, a 96-column last tile, tail splits 2-8 up to K's stage count, the
    whole waves unsplit or split 2 ways."""
    G = inputs.GROUP
    d, y_ref, abs_ref = _case(M, K, N, G, seed=M + N)
    x, qw_r, sc_r = _repacked(W, d, G)
    for t in tails:
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=dict(path=2, m_tile=256, split_k=split, tail_split=t))
        what = W.w4a16_last_dispatch()
        assert f"split_k={split} " in what and f"tail_split={t}" in what, what
        assert_parity(y_f64(y), y_ref, abs_ref, what)
        # the same product in one launch: bit-identical on the column tiles before the tail
        y1 = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=dict(path=2, m_tile=256, split_k=split))
        mtiles, items = -(-M // 256), -(-N // 128) * -(-M // 256)
        first_tail_col = 128 * ((items - int(what.split("tail_items=")[1].split()[0])) // mtiles)
        assert torch.equal(y[:, :first_tail_col], y1[:, :first_tail_col]), what


def test_partial_wave_tail_nvfp4_and_int8_activations(W):
    """The other weight and activation formats through the same two-launch plan (M = 1024,
    5120 x 5120), sampled on the tail's columns and at random."""
    M, K, N = 1024, 5120, 5120
    rng = np.random.default_rng(77)
    ms, ns = _tail_samples(M, N, rng)
    qw, s8, g = inputs.generate_nvfp4_weights(K, N, seed=78)
    x = inputs.generate_x(M, K, seed=79)
    r = W.repack_nvfp4(torch.from_numpy(qw).cuda(), torch.from_numpy(s8).cuda())
    y = W.gemm_nvfp4(x_to_dev(x), r[0], r[1], g, N, K)
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    what = W.w4a16_last_dispatch()
    assert "tail_items=" in what and "weights=nvfp4" in what, what
    y_ref, abs_ref = oracle.gemm_nvfp4_sampled(x, qw, s8, g, ms, ns)
    assert_parity(y_f64(y)[ms, ns], y_ref, abs_ref, what)

    G = inputs.GROUP
    qw, sc = inputs.generate_weights(K, N, G, seed=80)
    r = W.repack(torch.from_numpy(qw).cuda(), torch.from_numpy(sc.view(np.int16)).cuda(), G)
    act = W.quantize_x_int8(x_to_dev(x))
    y = W.gemm_w4a8(*act, r[0], r[1], N, K, G)
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    what = W.w4a16_last_dispatch()
    assert "tail_items=" in what and "activations=int8" in what, what
    xq, sx = oracle.quantize_x_int8(x)
    y_ref, abs_ref = oracle.gemm_w4a8_sampled(xq, sx, qw, sc, G, ms, ns)
    assert_parity(y_f64(y)[ms, ns], y_ref, abs_ref, what)


# ------------------------------------------------------------------------------ persistent grids
# An unsplit launch of the 128- or 256-row tile with more work items than resident CTAs (one per
# SM) runs one CTA per slot, each taking every slots-th item, its ring and barrier phases running on
# from one item to the next.
PERSISTENT = [
    (256, 256, 20480, dict(path=2, m_tile=256, split_k=1)),                 # 160 items: 8 CTAs take two
    (130, 512, 40960, dict(path=2, m_tile=256, split_k=1)),                 # 320 items, ragged rows
    (200, 256, 19552, dict(path=2, m_tile=256, split_k=1)),                 # 153 items, the last 96 wide
    (128, 256, 20480, dict(path=2, m_tile=128, split_k=1)),                 # the 128-row tile
    (256, 512, 39680, dict(path=2, m_tile=256, split_k=1, tail_split=4)),   # 2 persistent waves + a tail
]


@pytest.mark.parametrize("M,K,N,plan", PERSISTENT, ids=lambda v: str(v) if not isinstance(v, dict) else "")
def test_persistent_grid_every_element(W, M, K, N, plan):
    G = inputs.GROUP
    d, y_ref, abs_ref = _case(M, K, N, G, seed=M + 3 * N)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
    what = W.w4a16_last_dispatch()
    assert " persistent" in what, what
    assert_parity(y_f64(y), y_ref, abs_ref, what)
    # deterministic: the same plan again gives the same bits
    y2 = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), what


# ------------------------------------------------------------------------------ GEMV batch depth
# At one and two rows the GEMV keeps 8 blocks of 32 k in flight per warp (instead of 4) when its
# grid fits in one wave of that larger-register kernel.
@pytest.mark.parametrize("M,K,N,G,plan,deep", [
    (1, 5120, 5120, 128, None, True), (2, 5120, 5120, 128, None, True), (1, 17408, 5120, 128, None, True),
    (1, 5120, 7168, 128, None, True),                                  # split 4 -> 3: 672 CTAs, one wave
    (2, 5120, 7168, 128, None, False),                                 # 896 CTAs: two waves, stays at 4
    (1, 5120, 34816, 128, None, False),                                # 2176 CTAs
    (1, 1088, 5120, 64, dict(path=1, split_k=1), True), (2, 1088, 5120, 32, dict(path=1, split_k=3), True),
    (1, 5120, 5120, 128, dict(path=1, split_k=16), False),             # 2560 CTAs
])
def test_gemv_batch_depth_every_element(W, M, K, N, G, plan, deep):
    d, y_ref, abs_ref = _case(M, K, N, G, seed=M + K + N)
    x, qw_r, sc_r = _repacked(W, d, G)
    y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
    what = W.w4a16_last_dispatch()
    assert what.startswith("path=gemv") and ("unroll=8" in what) == deep, what
    if plan is None and (M, N) == (1, 7168):
        assert "split_k=3" in what, what
    assert_parity(y_f64(y), y_ref, abs_ref, what)
    if deep:  # one-hot rows stay exact through the deeper batches
        xb = np.zeros((M, K), np.uint16)
        for m in range(M):
            xb[m, (37 * m + 5) % K] = 0x3C00
        y1 = run_gemm(W, x_to_dev(xb), qw_r, sc_r, N, K, G, plan=plan)
        yo, _ = oracle.gemm(xb, d["qweight"], d["scales"], G)
        assert np.array_equal(y1.cpu().numpy().view(np.uint16), yo.astype(np.float16).view(np.uint16)), what
