"""GEMMs chained on one stream, as in a decode step: the second reads the first's output as x.

Every kernel is launched with programmatic dependent launch, so the second may start (and stream
its weights) while the first is still running; it must read x only after the first completed. The
first GEMM's x is made of one-hot rows, so its output is exactly rows of dequant(W1) (one product
per element, exact in fp32 and in fp16): the second GEMM's expected result is the oracle applied to
those rows, computed on the CPU without any GPU value. The intermediate buffer is filled with NaN
before each chain, so a read that came too early shows up as NaN or a wrong value."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import assert_parity, lib, to_dev, x_to_dev, y_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def W():
    return lib()


@pytest.fixture(scope="module")
def chain(W):
    M, K1, N1, N2, G = 6, 1024, 2048, 640, 128
    d1 = inputs.generate(M, K1, N1, G, seed=301)
    d2 = inputs.generate(M, N1, N2, G, seed=302)
    ks = [0, 129, 500, 511, 777, K1 - 1]
    x0 = np.zeros((M, K1), np.float16)
    for i, k in enumerate(ks):
        x0[i, k] = 1.0
    w1 = oracle.dequant(d1["qweight"], d1["scales"], G)
    y1_exp = np.stack([w1[k] for k in ks]).astype(np.float16)  # exact: one product per element
    y2_ref, abs2 = oracle.gemm(y1_exp.view(np.uint16), d2["qweight"], d2["scales"], G)
    _, qw1, sc1 = to_dev(d1)
    _, qw2, sc2 = to_dev(d2)
    r1 = W.repack(qw1, sc1, G)
    r2 = W.repack(qw2, sc2, G)
    return dict(M=M, K1=K1, N1=N1, N2=N2, G=G, x0=x_to_dev(x0.view(np.uint16)), r1=r1, r2=r2, y1_exp=y1_exp,
                y2_ref=y2_ref, abs2=abs2)


PLANS = [(None, None), (dict(path=1), dict(path=1)), (dict(path=2), dict(path=2)), (dict(path=1), dict(path=2)),
         (dict(path=2, split_k=3), dict(path=1, split_k=4)), (dict(path=2, m_tile=128), dict(path=2, split_k=2))]


def _run_chain(W, c, p1, p2, y1, y2, stream=None):
    y1.fill_(float("nan"))
    W.gemm(c["x0"], *c["r1"], c["N1"], c["K1"], c["G"], y=y1, plan=p1, stream=stream)
    W.gemm(y1, *c["r2"], c["N2"], c["N1"], c["G"], y=y2, plan=p2, stream=stream)


@pytest.mark.parametrize("p1,p2", PLANS, ids=lambda p: "auto" if p is None else "-".join(f"{k}{v}" for k, v in p.items()))
def test_chain_reads_the_previous_output(W, chain, p1, p2):
    c = chain
    y1 = torch.empty((c["M"], c["N1"]), dtype=torch.float16, device="cuda")
    y2 = torch.empty((c["M"], c["N2"]), dtype=torch.float16, device="cuda")
    for _ in range(5):
        _run_chain(W, c, p1, p2, y1, y2)
        torch.cuda.synchronize()
        assert W.w4a16_device_status() == W.OK
        assert np.array_equal(y1.cpu().numpy().view(np.uint16), c["y1_exp"].view(np.uint16))
        assert_parity(y_f64(y2), c["y2_ref"], c["abs2"], "second GEMM of the chain")


def test_chain_in_a_cuda_graph(W, chain):
    c = chain
    y1 = torch.empty((c["M"], c["N1"]), dtype=torch.float16, device="cuda")
    y2 = torch.empty((c["M"], c["N2"]), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    for p1, p2 in PLANS:  # warm the plan cache outside capture
        _run_chain(W, c, p1, p2, y1, y2)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for p1, p2 in PLANS:
            _run_chain(W, c, p1, p2, y1, y2, stream=s)
    for _ in range(10):
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert W.w4a16_device_status() == W.OK
        assert np.array_equal(y1.cpu().numpy().view(np.uint16), c["y1_exp"].view(np.uint16))
        assert_parity(y_f64(y2), c["y2_ref"], c["abs2"], "second GEMM of the chain, CUDA graph")
