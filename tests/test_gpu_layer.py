"""The dense layer's activation and a two-layer GEMM chain on the GPU against the CPU oracle.

* w4a16_silu_mul against the oracle's fp64 silu(gate) * up on every element: the GPU evaluates in
  fp32 and rounds once to fp16, so |act - act_ref| <= (2^-11 + 2^-20) |act_ref| + 2^-25.
* Two dense layers chained on one stream as a decode step runs them (qkv and o from the layer
  input, gate+up from o, silu * up, down -> the next layer's input), every kernel with
  programmatic dependent launch, against the oracle's own chain (fp64 GEMMs, fp64 activation, fp16
  rounding between the stages, like the GPU). Each stage is held to the per-GEMM acceptance bound
  2^-10 (|y| + sum_k |x w|), plus the oracle's own rounding of its intermediate, plus the
  difference of the stage's inputs carried through the stage as independent errors (6 sigma, with
  the previous stage's bound as sigma). The layer is the dense-layer shape scaled down (hidden 2048,
  qkv 2560, MLP 4096) so that the oracle holds |w|^2 in memory.
* The same two layers with int8 activations (W4A8), every stage against the oracle applied to the
  stage's own GPU inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import lib, x_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def W():
    return lib()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(bits: np.ndarray) -> np.ndarray:
    return bits.view(np.float16).astype(np.float64)


@pytest.mark.parametrize("M,I", [(1, 8), (3, 1000 * 8), (16, 17408), (64, 4096)])
def test_silu_mul_matches_oracle(W, M, I):
    rng = np.random.default_rng(M * 7 + I)
    gu = rng.normal(0.0, 3.0, size=(M, 2 * I)).astype(np.float16)
    # special values: zeros of both signs, large |g|, subnormal g and u
    flat = gu.reshape(-1)
    flat[:8] = np.array([0.0, -0.0, 30.0, -30.0, 6e-5, -6e-8, 1000.0, -1000.0], np.float16)[: flat.size]
    bits = gu.view(np.uint16)
    act_ref, _ = oracle.silu_mul(bits)
    act = W.silu_mul(x_to_dev(bits))
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    got = _f64(_bits(act))
    assert np.all(np.isfinite(got))
    bound = (2.0 ** -11 + 2.0 ** -20) * np.abs(act_ref) + 2.0 ** -25
    err = np.abs(got - act_ref)
    assert (err <= bound).all(), f"{int((err > bound).sum())} elements outside, worst {float((err / bound).max()):.3f}"


def test_silu_mul_rejects_bad_arguments(W):
    gu = torch.zeros((2, 16), dtype=torch.float16, device="cuda")
    act = torch.zeros((2, 8), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert W.w4a16_silu_mul(gu.data_ptr(), act.data_ptr(), 2, 6, s) == W.ERR_UNSUPPORTED_SHAPE  # I % 8
    assert W.w4a16_silu_mul(gu.data_ptr(), act.data_ptr(), 0, 8, s) == W.ERR_INVALID_ARG
    assert W.w4a16_silu_mul(gu.data_ptr() + 2, act.data_ptr(), 2, 8, s) == W.ERR_MISALIGNED
    assert W.w4a16_silu_mul(gu.data_ptr(), gu.data_ptr() + 16, 1, 8, s) == W.ERR_INVALID_ARG  # overlap


# ------------------------------------------------------------------------------ two-layer chain
H, QKV, INTER, G = 2048, 2560, 4096, 128


@pytest.fixture(scope="module")
def layers(W):
    out = []
    for layer in range(2):
        mats = {}
        for name, (K, N) in (("qkv", (H, QKV)), ("o", (H, H)), ("gu", (H, 2 * INTER)), ("down", (INTER, H))):
            qw, sc = inputs.generate_weights(K, N, G, seed=500 + 10 * layer + len(mats))
            r = W.repack(torch.from_numpy(qw).cuda(), torch.from_numpy(sc.view(np.int16)).cuda(), G)
            w2 = oracle.dequant(qw, sc, G) ** 2  # |w|^2 for the carried input differences
            mats[name] = dict(K=K, N=N, qw=qw, sc=sc, r=r, w2=w2)
        out.append(mats)
    return out


def _oracle_gemm_stage(x_bits, e_in, m):
    """(y fp16 bits, bound) of one GEMM stage of the oracle chain."""
    y, a = oracle.gemm(x_bits, m["qw"], m["sc"], G)
    carried = 6.0 * np.sqrt(e_in ** 2 @ m["w2"]) if e_in is not None else 0.0
    bound = 2.0 ** -10 * (np.abs(y) + a) + 2.0 ** -11 * np.abs(y) + 2.0 ** -25 + carried
    return oracle.double_to_half(y), bound


def _oracle_act_stage(gu_bits, e_gu):
    act, act_bits = oracle.silu_mul(gu_bits)
    ones = np.full((gu_bits.shape[0], gu_bits.shape[1] // 2), np.float16(1.0)).view(np.uint16)
    silu, _ = oracle.silu_mul(np.concatenate([gu_bits[:, : gu_bits.shape[1] // 2], ones], axis=1))
    u = _f64(gu_bits[:, gu_bits.shape[1] // 2:])
    e_g, e_u = e_gu[:, : e_gu.shape[1] // 2], e_gu[:, e_gu.shape[1] // 2:]
    carried = 6.0 * np.sqrt((1.1 * e_g * (np.abs(u) + e_u)) ** 2 + (np.abs(silu) * e_u) ** 2)
    return act_bits, (2.0 ** -10 + 2.0 ** -20) * np.abs(act) + 2.0 ** -24 + carried


@pytest.mark.parametrize("M", [1, 4, 16])
def test_two_layer_chain(W, layers, M):
    x0 = inputs.generate_x(M, H, seed=600 + M)
    # ---- the GPU chain, one stream, no synchronisation between the kernels
    h = x_to_dev(x0)
    outs = []
    for mats in layers:
        qkv = W.gemm(h, *mats["qkv"]["r"], QKV, H, G)
        o = W.gemm(h, *mats["o"]["r"], H, H, G)
        gu = W.gemm(o, *mats["gu"]["r"], 2 * INTER, H, G)
        act = W.silu_mul(gu)
        h = W.gemm(act, *mats["down"]["r"], H, INTER, G)
        outs.append(dict(qkv=qkv, o=o, gu=gu, act=act, down=h))
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    # ---- the oracle's chain and the stage bounds
    hb, e_h = x0, None
    for layer, mats in enumerate(layers):
        ref = {}
        ref["qkv"] = _oracle_gemm_stage(hb, e_h, mats["qkv"])
        ref["o"] = _oracle_gemm_stage(hb, e_h, mats["o"])
        ref["gu"] = _oracle_gemm_stage(ref["o"][0], ref["o"][1], mats["gu"])
        ref["act"] = _oracle_act_stage(ref["gu"][0], ref["gu"][1])
        ref["down"] = _oracle_gemm_stage(ref["act"][0], ref["act"][1], mats["down"])
        for stage in ("qkv", "o", "gu", "act", "down"):
            got = _f64(_bits(outs[layer][stage]))
            want_bits, bound = ref[stage]
            err = np.abs(got - _f64(want_bits))
            assert np.all(np.isfinite(got)), f"layer {layer} {stage}"
            bad = ~(err <= bound)
            assert not bad.any(), (f"layer {layer} {stage}: {int(bad.sum())} of {err.size} outside, "
                                   f"worst err/bound {float(np.max(err / bound)):.3f}")
        hb, e_h = ref["down"]


@pytest.mark.parametrize("M", [1, 2, 16])
def test_two_layer_chain_int8_activations(W, layers, M):
    # The same two layers with int8 activations (W4A8): every GEMM input quantised per token in the
    # call of its first GEMM, all on one stream with programmatic dependent launch. Each stage is
    # checked against the oracle applied to that stage's own GPU inputs: the codes and scales bit
    # for bit, every GEMM output at the per-GEMM bound, the activation at its bound.
    x0 = inputs.generate_x(M, H, seed=700 + M)
    h = x_to_dev(x0)
    outs = []
    for mats in layers:
        qkv, qh = W.quantize_gemm_w4a8(h, *mats["qkv"]["r"], QKV, H, G)
        o = W.gemm_w4a8(*qh, *mats["o"]["r"], H, H, G)
        gu, qo = W.quantize_gemm_w4a8(o, *mats["gu"]["r"], 2 * INTER, H, G)
        act = W.silu_mul(gu)
        h_next, qa = W.quantize_gemm_w4a8(act, *mats["down"]["r"], H, INTER, G)
        outs.append(dict(h=h, qh=qh, qkv=qkv, o=o, qo=qo, gu=gu, act=act, qa=qa, down=h_next))
        h = h_next
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    for layer, (mats, st) in enumerate(zip(layers, outs)):
        for (src, q, gemms) in (("h", "qh", (("qkv", "qkv"), ("o", "o"))), ("o", "qo", (("gu", "gu"),)),
                                ("act", "qa", (("down", "down"),))):
            xq_ref, sx_ref = oracle.quantize_x_int8(_bits(st[src]))
            xq, _, sx = st[q]
            assert np.array_equal(xq.cpu().numpy(), xq_ref), f"layer {layer}: codes of {src}"
            assert np.array_equal(sx.cpu().numpy(), sx_ref), f"layer {layer}: scales of {src}"
            for (mname, out) in gemms:
                y_ref, a_ref = oracle.gemm_w4a8(xq_ref, sx_ref, mats[mname]["qw"], mats[mname]["sc"], G)
                got = _f64(_bits(st[out]))
                bound = 2.0 ** -10 * (np.abs(y_ref) + a_ref)
                bad = ~(np.abs(got - y_ref) <= bound)
                assert not bad.any(), f"layer {layer} {out}: {int(bad.sum())} outside"
        act_ref, _ = oracle.silu_mul(_bits(st["gu"]))
        got = _f64(_bits(st["act"]))
        assert np.all(np.abs(got - act_ref) <= (2.0 ** -11 + 2.0 ** -20) * np.abs(act_ref) + 2.0 ** -25)
