"""The C-ABI library loads, exports every entry point include/w4a16.h declares, and rejects bad
arguments on the host before any launch (no GPU needed: these calls return before touching CUDA)."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def W():
    import __graft_entry__

    __graft_entry__.build_library()
    import w4a16_weight_streaming_gb300 as W

    return W


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(w4a16_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_gemm_and_repack_calls():
    names = declared_functions()
    for n in ("w4a16_repack", "w4a16_unrepack", "w4a16_gemm", "w4a16_gemm_ex", "w4a16_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(W):
    lib = ctypes.CDLL(W.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in w4a16.h but not exported"
    assert sorted(W.EXPORTED) == declared_functions()


def test_debug_bounds_build_exports_the_same_symbols(W):
    dbg = W.load_debug_bounds()
    for name in declared_functions():
        assert hasattr(dbg, name), f"{name} missing from the debug-bounds build"
    assert dbg.w4a16_debug_bounds() == 1 and W.lib.w4a16_debug_bounds() == 0
    assert dbg.w4a16_status_string(6).decode().startswith("W4A16_ERR_BOUNDS")


def test_version_and_status_strings(W):
    assert W.w4a16_version() >= 100
    for code in range(7):
        assert W.status_string(code).startswith("W4A16_")
    assert W.status_string(99) == "W4A16_ERR_UNKNOWN"


def test_repacked_sizes_equal_canonical_sizes(W):
    for (N, K, G) in [(1024, 1024, 128), (5120, 17408, 128), (34816, 5120, 128), (96, 256, 32)]:
        assert W.w4a16_repacked_qweight_bytes(N, K, G) == K * N // 2
        assert W.w4a16_repacked_scales_bytes(N, K, G) == (K // G) * N * 2
    assert W.w4a16_repacked_qweight_bytes(100, 1024, 128) == 0  # N % 32
    assert W.w4a16_repacked_scales_bytes(1024, 1000, 128) == 0  # K % 64


FAKE = 1 << 40  # never dereferenced: every call below is rejected before any launch


@pytest.mark.parametrize("args,code", [
    ((0, FAKE, FAKE, FAKE, 4, 1024, 1024, 128), 1),          # null x
    ((FAKE, 0, FAKE, FAKE, 4, 1024, 1024, 128), 1),          # null qweight
    ((FAKE, FAKE, FAKE, 0, 4, 1024, 1024, 128), 1),          # null y
    ((FAKE, FAKE, FAKE, FAKE * 2, 0, 1024, 1024, 128), 1),   # M = 0
    ((FAKE, FAKE, FAKE, FAKE * 2, -3, 1024, 1024, 128), 1),  # M < 0
    ((FAKE, FAKE, FAKE, FAKE * 2, 4, 1000, 1024, 128), 2),   # N % 32
    ((FAKE, FAKE, FAKE, FAKE * 2, 4, 1024, 1000, 128), 2),   # K % 64
    ((FAKE, FAKE, FAKE, FAKE * 2, 4, 1024, 1024, 48), 2),    # group % 32
    ((FAKE, FAKE, FAKE, FAKE * 2, 4, 1024, 640, 256), 2),    # K % group
    ((FAKE, FAKE, FAKE, FAKE * 2, (1 << 20) + 1, 1024, 1024, 128), 2),  # M too large
    ((FAKE + 8, FAKE, FAKE, FAKE * 2, 4, 1024, 1024, 128), 3),          # misaligned x
    ((FAKE, FAKE, FAKE + 4, FAKE * 2, 4, 1024, 1024, 128), 3),          # misaligned scales
    ((FAKE, FAKE * 4, FAKE * 4, FAKE + 1024, 4, 1024, 1024, 128), 1),   # y overlaps x
])
def test_gemm_rejects_bad_arguments_on_host(W, args, code):
    assert W.w4a16_gemm(*args, None) == code


def test_gemm_host_rejects_bad_arguments_on_host(W):
    ok = [FAKE * 8, FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 9]  # x_host x_dev qw sc y_dev y_host
    shape = (4, 1024, 1024, 128)

    def call(i, v, *sh):
        a = list(ok)
        if i is not None:
            a[i] = v
        return W.w4a16_gemm_host(*a, *(sh or shape), None)

    assert call(0, 0) == 1                     # null x_host
    assert call(5, 0) == 1                     # null y_host
    assert call(1, 0) == 1                     # null x_dev
    assert call(4, 0) == 1                     # null y_dev
    assert call(None, 0, 4, 1000, 1024, 128) == 2   # N % 32
    assert call(1, FAKE + 8) == 3              # misaligned x_dev
    assert call(4, FAKE + 1024) == 1           # y_dev overlaps x_dev


def test_repack_rejects_bad_arguments_on_host(W):
    assert W.w4a16_repack(0, FAKE, FAKE * 2, FAKE * 3, 1024, 1024, 128, None) == 1
    assert W.w4a16_repack(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, 1000, 1024, 128, None) == 2
    assert W.w4a16_repack(FAKE + 2, FAKE * 2, FAKE * 3, FAKE * 4, 1024, 1024, 128, None) == 3
    # output overlapping the input
    assert W.w4a16_repack(FAKE, FAKE * 2, FAKE + 64, FAKE * 4, 1024, 1024, 128, None) == 1
    assert W.w4a16_unrepack(FAKE, FAKE * 2, FAKE * 3, 0, 1024, 1024, 128, None) == 1


def test_plan_for_host_only(W):
    p = W.w4a16_plan_for(1, 5120, 5120, 128)
    assert p.path in (W.PATH_GEMV, W.PATH_TC)
    for M in (1, 16, 256, 1024):
        p = W.w4a16_plan_for(M, 34816, 5120, 128)
        if p.path == W.PATH_TC:
            assert p.m_tile in (16, 32, 64, 128, 256) and p.m_tile >= min(M, 16)
            assert p.k_chunk in (64, 128, 256) and 2 <= p.stages <= 16 and 1 <= p.split_k <= 16
            assert 2 <= p.tmem_stages <= 8
    with pytest.raises(W.W4A16Error):
        W.w4a16_plan_for(0, 5120, 5120, 128)


def test_plan_for_group_sizes(W):
    # groups that divide 128 or are multiples of it run on the tiles; others on the GEMV (M <= 8)
    for G in (32, 64, 128, 256, 384):
        assert W.w4a16_plan_for(16, 256, 1536, G).path == W.PATH_TC
    for G in (96, 160):
        for M in (1, 3, 8):
            assert W.w4a16_plan_for(M, 256, 1920, G).path == W.PATH_GEMV
        with pytest.raises(W.W4A16Error):
            W.w4a16_plan_for(9, 256, 1920, G)


def test_every_supported_shape_gets_a_plan(W):
    # host-only property of the dispatcher: inside the supported set every automatic plan resolves,
    # except, at more than 8 rows, shapes the tiles cannot stage (K % 128, odd group sizes)
    rng = np.random.default_rng(5)
    for _ in range(400):
        G = int(rng.choice([32, 64, 96, 128, 160, 256, 384, 512]))
        K = G * int(rng.integers(1, 40))
        K = K if K % 64 == 0 else 2 * K
        N = 32 * int(rng.integers(1, 1200))
        M = int(rng.choice([1, 2, 3, 5, 8, 9, 16, 31, 64, 65, 128, 200, 256, 511, 1024, 4096]))
        fits = (128 % G == 0 or G % 128 == 0) and K % 128 == 0
        if M > 8 and not fits:
            with pytest.raises(W.W4A16Error):
                W.w4a16_plan_for(M, N, K, G)
            continue
        p = W.w4a16_plan_for(M, N, K, G)
        assert p.path in (W.PATH_GEMV, W.PATH_TC)
        assert p.split_k >= 1
        if p.path == W.PATH_TC:
            assert p.k_chunk in (128, 256) and K % p.k_chunk == 0
            assert p.split_k <= K // p.k_chunk
            assert 2 <= p.stages <= 16 and p.m_tile in (16, 32, 64, 128, 256)
            # a K-split tail only behind unsplit whole waves of the 128- and 256-row tiles, and only
            # when the work items overfill whole waves (152 one-CTA-per-SM slots without a device)
            if p.tail_split:
                items = -(-N // 128) * -(-M // p.m_tile)
                assert p.m_tile >= 128 and p.split_k == 1 and 2 <= p.tail_split <= min(16, K // p.k_chunk)
                assert items > 152 and items % 152, (M, N, K, G, items)
        else:
            assert p.tail_split == 0


def test_boundary_shapes_get_plans(W):
    # the corners of the advertised set: widest N, longest K, most rows, and the GEMV-only shapes
    # (K % 128 != 0) at the documented M * K <= 1,500,000
    for (M, N, K, G) in [(1, 1 << 23, 5120, 128), (1, 5120, 1 << 22, 128), (8, 5120, 1 << 22, 128),
                         (1 << 20, 1 << 23, 1 << 22, 128), (1 << 20, 32, 128, 128), (1, 1 << 23, 1 << 22, 128),
                         (1, 256, 1_499_968, 64), (8, 256, 187_456, 64), (3, 1 << 23, 1216, 64)]:
        p = W.w4a16_plan_for(M, N, K, G)
        assert p.path in (W.PATH_GEMV, W.PATH_TC), (M, N, K, G)
        if p.path == W.PATH_GEMV:
            assert M <= 8 and 1 <= p.split_k <= 16
        else:
            assert K % p.k_chunk == 0 and p.split_k * -(-N // 128) * -(-M // p.m_tile) < 2 ** 31
    with pytest.raises(W.W4A16Error):
        W.w4a16_plan_for(1, (1 << 23) + 32, 5120, 128)
    with pytest.raises(W.W4A16Error):
        W.w4a16_plan_for(1, 5120, (1 << 22) + 128, 128)


def _plan_in_subprocess(env_value, shape=(1, 5120, 5120, 128), fields=("path", "split_k", "m_tile")):
    import subprocess
    import sys

    code = ("import w4a16_weight_streaming_gb300 as W\n"
            "try:\n"
            f"    p = W.w4a16_plan_for{tuple(shape)}; print(*[getattr(p, f) for f in {tuple(fields)}])\n"
            "except W.W4A16Error as e:\n"
            "    print('error', e.code)\n")
    env = dict(os.environ)
    env.pop("W4A16_PLAN", None)
    if env_value is not None:
        env["W4A16_PLAN"] = env_value
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    return out.stdout.split()


def test_plan_override_from_environment(W):
    assert _plan_in_subprocess(None)[0] == str(W.PATH_GEMV)           # automatic: the GEMV at M = 1
    assert _plan_in_subprocess("path=2,m_tile=16,split_k=2") == ["2", "2", "16"]
    assert _plan_in_subprocess("path=2,bogus=1") == ["error", "1"]    # malformed: refused loudly
    assert _plan_in_subprocess("path=2,split_k=x") == ["error", "1"]
    assert _plan_in_subprocess("path=1,split_k=40") == ["error", "2"]  # valid syntax, invalid plan


def test_partial_wave_tail_plans(W):
    # Work items of 128 columns x 256 rows that overfill whole waves (one CTA per SM, 152 SMs
    # without a device): the automatic plan runs the last, partial wave's items as a second launch,
    # each split along K, when the cost model rates it cheaper than one launch.
    for N, K in ((5120, 5120), (7168, 5120), (34816, 5120), (5120, 17408)):
        p = W.w4a16_plan_for(1024, N, K, 128)
        assert p.path == W.PATH_TC and p.m_tile == 256 and p.split_k == 1 and 2 <= p.tail_split <= 16, (N, K)
        assert p.tail_split <= K // p.k_chunk
    assert W.w4a16_plan_for(1000, 5088, 5120, 128).tail_split > 0  # ragged rows and last column tile
    p = W.w4a16_plan_for(512, 5120, 17408, 128)  # 80 items: split whole waves are for explicit plans only
    assert (p.split_k, p.tail_split) == (3, 0), (p.split_k, p.tail_split)
    assert W.w4a16_plan_for(512, 34816, 5120, 128).tail_split == 0  # 88 left over: no one-wave tail
    assert W.w4a16_plan_for(256, 5120, 5120, 128).tail_split == 0  # 40 items: one partial wave, split_k
    assert W.w4a16_plan_for(16, 34816, 5120, 128).tail_split == 0  # small tiles: not this rule
    assert W.w4a16_plan_for(1, 34816, 5120, 128).tail_split == 0  # the GEMV
    assert W.w4a16_plan_for_nvfp4(1024, 5120, 5120).tail_split > 0
    assert W.w4a16_plan_for_w4a8(1024, 5120, 5120).tail_split > 0


def test_tail_split_in_explicit_plans(W):
    shape, f = (1024, 5120, 5120, 128), ("path", "split_k", "tail_split")
    assert _plan_in_subprocess("path=2,m_tile=256,split_k=1,tail_split=3", shape, f) == ["2", "1", "3"]
    assert _plan_in_subprocess("path=2,tail_split=8", shape, f) == ["2", "1", "8"]
    assert _plan_in_subprocess("path=2,m_tile=256,split_k=2", shape, f) == ["2", "2", "0"]  # explicit: none unless asked
    assert _plan_in_subprocess("path=2,tail_split=1", shape, f) == ["error", "1"]
    assert _plan_in_subprocess("path=2,tail_split=17", shape, f) == ["error", "1"]
    assert _plan_in_subprocess("path=2,tail_split=-2", shape, f) == ["error", "1"]
    assert _plan_in_subprocess("path=2,split_k=2,tail_split=4", shape, f) == ["2", "2", "4"]  # 76 items a wave
    # one partial wave only (40 items): nothing to split off, the plan stays one unsplit launch
    assert _plan_in_subprocess("path=2,m_tile=256,tail_split=4", (256, 5120, 5120, 128), f) == ["2", "1", "0"]
    # a tail split above the stage count of K
    assert _plan_in_subprocess("path=2,tail_split=16", (1024, 5120, 1024, 128), f) == ["error", "2"]


def test_wait_timeout_setting(W):
    assert W.w4a16_set_wait_timeout_ns(10) == 1
    assert W.w4a16_set_wait_timeout_ns(2_000_000_000) == 0


def test_selftest_rejects_bad_mode(W):
    # host-side check before any launch
    assert W.w4a16_selftest_wait_timeout(2) == 1
    assert W.w4a16_selftest_wait_timeout(-1) == 1


def test_nvfp4_host_checks(W):
    # argument checks of the NVFP4 entry points, before any device work
    assert W.w4a16_repacked_nvfp4_scales_bytes(256, 1024) == (1024 // 16) * 256 * 2
    assert W.w4a16_repacked_nvfp4_scales_bytes(250, 1024) == 0
    assert W.w4a16_repack_nvfp4(0, FAKE, FAKE * 2, FAKE * 3, 1024, 1024, None) == 1
    assert W.w4a16_repack_nvfp4(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, 1000, 1024, None) == 2
    assert W.w4a16_repack_nvfp4(FAKE + 2, FAKE * 2, FAKE * 3, FAKE * 4, 1024, 1024, None) == 3
    assert W.w4a16_unrepack_nvfp4(FAKE, FAKE * 2, FAKE * 3, 0, 1024, 1024, None) == 1
    assert W.w4a16_gemm_nvfp4(FAKE, FAKE * 2, FAKE * 3, float("nan"), FAKE * 4, 1, 1024, 1024, None) == 1
    assert W.w4a16_gemm_nvfp4(FAKE, FAKE * 2, FAKE * 3, float("inf"), FAKE * 4, 1, 1024, 1024, None) == 1
    assert W.w4a16_gemm_nvfp4(FAKE, FAKE * 2, FAKE * 3, 1.0, FAKE * 4, 1, 1024, 1000, None) == 2
    p = W.w4a16_plan_for_nvfp4(16, 34816, 5120)
    assert p.path == W.PATH_TC and p.m_tile == 16
    assert W.w4a16_plan_for_nvfp4(1, 5120, 5120).path == W.PATH_GEMV
    with pytest.raises(W.W4A16Error):
        W.w4a16_plan_for_nvfp4(9, 5120, 5120 + 64)  # K % 128 != 0 needs the GEMV, which takes M <= 8


def test_w4a8_host_checks(W):
    # argument checks of the int8-activation entry points, before any device work
    q = W.w4a16_quantize_x_int8
    assert q(0, FAKE, None, FAKE * 2, 4, 1024, None) == 1            # null x
    assert q(FAKE, FAKE * 2, None, 0, 4, 1024, None) == 1            # null sx
    assert q(FAKE, FAKE * 2, None, FAKE * 3, 0, 1024, None) == 1     # M = 0
    assert q(FAKE, FAKE * 2, None, FAKE * 3, 4, 1001, None) == 2     # K % 8
    assert q(FAKE + 2, FAKE * 2, None, FAKE * 3, 4, 1024, None) == 3  # x misaligned
    assert q(FAKE, FAKE * 2, FAKE * 4 + 8, FAKE * 3, 4, 1024, None) == 3  # xq_f16 misaligned
    assert q(FAKE, FAKE * 2, None, FAKE * 3 + 2, 4, 1024, None) == 3  # sx not 4-byte aligned
    assert q(FAKE, FAKE + 4096, None, FAKE * 3, 4, 1024, None) == 1   # xq overlaps x (8 KB)
    g = W.w4a16_gemm_w4a8
    assert g(0, None, FAKE, FAKE * 2, FAKE * 3, FAKE * 4, 1, 1024, 1024, 128, None) == 1
    assert g(FAKE, None, FAKE * 5, FAKE * 2, FAKE * 3, FAKE * 4, 0, 1024, 1024, 128, None) == 1
    assert g(FAKE, None, FAKE * 5, FAKE * 2, FAKE * 3, FAKE * 4, 1, 1000, 1024, 128, None) == 2
    assert g(FAKE + 8, None, FAKE * 5, FAKE * 2, FAKE * 3, FAKE * 4, 1, 1024, 1024, 128, None) == 3
    assert g(FAKE, None, FAKE * 5 + 1, FAKE * 2, FAKE * 3, FAKE * 4, 1, 1024, 1024, 128, None) == 3
    assert g(FAKE, None, FAKE * 5, FAKE * 2, FAKE * 3, FAKE + 64, 1, 1024, 1024, 128, None) == 1  # y overlaps xq
    # the automatic plan: the integer GEMV at M <= 2, at M = 3 while its grid fits in one wave
    for M in (1, 2):
        for (N, K) in ((5120, 5120), (7168, 5120), (34816, 5120), (5120, 17408)):
            assert W.w4a16_plan_for_w4a8(M, N, K).path == W.PATH_GEMV
    assert W.w4a16_plan_for_w4a8(3, 5120, 17408).path == W.PATH_GEMV   # 40 tiles x split 16 = 640 CTAs
    assert W.w4a16_plan_for_w4a8(3, 7168, 5120).path == W.PATH_TC      # 56 tiles x split 16 = 896 CTAs
    for (N, K) in ((5120, 5120), (34816, 5120)):
        assert W.w4a16_plan_for_w4a8(4, N, K).path == W.PATH_TC
    # one wave: the split is the largest power of two whose grid fits (8 CTAs per SM at M <= 2)
    assert W.w4a16_plan_for_w4a8(1, 34816, 5120).split_k == 4       # 272 tiles x 4 = 1088 <= 1216
    assert W.w4a16_plan_for_w4a8(1, 5120, 17408).split_k == 16
    assert W.w4a16_plan_for_w4a8(5, 5120, 5120).path == W.PATH_TC
    assert W.w4a16_plan_for_w4a8(8, 5120, 5120 + 64, 64).path == W.PATH_GEMV  # K % 128 != 0: only the GEMV can
    p = W.w4a16_plan_for_w4a8(9, 5120, 5120)
    assert p.path == W.PATH_TC and p.m_tile == 16
    assert W.w4a16_plan_for_w4a8(256, 34816, 5120).m_tile == 256
    with pytest.raises(W.W4A16Error):
        W.w4a16_plan_for_w4a8(9, 5120, 5120 + 64)  # K % 128 != 0: the tiles cannot, the GEMV takes M <= 8


def test_quantize_gemm_w4a8_host_checks(W):
    f = W.w4a16_quantize_gemm_w4a8
    A = [FAKE, FAKE * 2, None, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6]  # x, xq, xq_f16, sx, qw_r, sc_r, y
    def call(args, M=1, N=1024, K=1024, G=128):
        return f(*args, M, N, K, G, None, None)
    assert call([0] + A[1:]) == 1                        # null x
    assert call(A, M=0) == 1
    assert call(A, N=1000) == 2
    assert call([FAKE + 2] + A[1:]) == 3                  # x misaligned
    assert call(A[:3] + [FAKE * 3 + 1] + A[4:]) == 3      # sx misaligned
    assert call(A[:1] + [FAKE + 256] + A[2:]) == 1        # xq overlaps x
    assert call(A[:6] + [FAKE * 2 + 64]) == 1             # y overlaps xq
    assert call(A[:2] + [FAKE * 3 - 64] + A[3:]) == 1     # xq_f16 overlaps sx
