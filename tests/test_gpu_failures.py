"""Failure reporting without a GPU fault, and output guard bands.

* A kernel whose bounded wait can never complete (an mbarrier phase that nothing arrives on) must
  give up after the wait limit, report W4A16_ERR_DEVICE_TIMEOUT through w4a16_device_status and
  leave the context usable: a GEMM right after it runs and matches the oracle.
* No kernel writes outside y: canary regions before and after y stay untouched on every path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import assert_parity, lib, run_gemm, to_dev, y_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def W():
    return lib()


def _small_case(W, M=4, K=1024, N=352, G=128, seed=51):
    d = inputs.generate(M, K, N, G, seed=seed)
    y_ref, abs_ref = oracle.gemm(d["x"], d["qweight"], d["scales"], G)
    x, qw, sc = to_dev(d)
    qw_r, sc_r = W.repack(qw, sc, G)
    return x, qw_r, sc_r, y_ref, abs_ref, K, N, G


@pytest.mark.parametrize("mode", [0, 1])
def test_bounded_wait_reports_timeout_and_context_survives(W, mode):
    assert W.w4a16_device_status() == W.OK
    assert W.w4a16_set_wait_timeout_ns(1_000_000) == W.OK  # 1 ms
    try:
        assert W.w4a16_selftest_wait_timeout(mode) == W.OK
        assert W.w4a16_device_status() == 5  # W4A16_ERR_DEVICE_TIMEOUT
        assert W.w4a16_device_status() == W.OK  # read clears it
    finally:
        assert W.w4a16_set_wait_timeout_ns(2_000_000_000) == W.OK
    x, qw_r, sc_r, y_ref, abs_ref, K, N, G = _small_case(W)
    for plan in (dict(path=1), dict(path=2)):
        y = run_gemm(W, x, qw_r, sc_r, N, K, G, plan=plan)
        assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())


@pytest.mark.parametrize("plan", [dict(path=1), dict(path=1, split_k=3), dict(path=2), dict(path=2, split_k=3),
                                  dict(path=2, m_tile=128)],
                         ids=lambda p: "-".join(f"{k}{v}" for k, v in p.items()))
def test_no_writes_outside_y(W, plan):
    M = 3 if plan["path"] == 1 else 17
    x, qw_r, sc_r, y_ref, abs_ref, K, N, G = _small_case(W, M=M, seed=52 + M)
    pad = 4096  # fp16 elements (8 KB) of canary on each side
    canary = 0x7BAD  # a finite fp16 bit pattern no kernel produces here
    buf = torch.full((M * N + 2 * pad,), canary, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + M * N].view(torch.float16).view(M, N)
    W.gemm(x, qw_r, sc_r, N, K, G, y=y, plan=plan)
    torch.cuda.synchronize()
    assert W.w4a16_device_status() == W.OK
    host = buf.cpu().numpy().view(np.uint16)
    assert (host[:pad] == canary).all() and (host[pad + M * N:] == canary).all(), W.w4a16_last_dispatch()
    assert_parity(y_f64(y), y_ref, abs_ref, W.w4a16_last_dispatch())
