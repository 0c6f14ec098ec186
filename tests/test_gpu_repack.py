"""w4a16_repack / w4a16_unrepack on the GPU: bit-exact against the oracle's statement of the
device layout, and an exact round trip back to the canonical format."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs
from gpu_util import lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K,N,G", [(1024, 1024, 128), (256, 96, 32), (640, 352, 64), (5120, 5120, 128),
                                   (17408, 5120, 128)])
def test_repack_bit_exact_and_round_trip(K, N, G):
    W = lib()
    rng = np.random.default_rng(K * 7 + N)
    words = rng.integers(0, 2 ** 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    scales = rng.integers(0, 2 ** 16, size=(K // G, N), dtype=np.uint32).astype(np.uint16)
    qw = torch.from_numpy(words).cuda()
    sc = torch.from_numpy(scales.view(np.int16)).cuda()
    qw_r, sc_r = W.repack(qw, sc, G)
    torch.cuda.synchronize()
    wr_ref, sr_ref = oracle.repack(words, scales, G)
    assert np.array_equal(qw_r.cpu().numpy().view(np.uint32), wr_ref.reshape(-1))
    assert np.array_equal(sc_r.cpu().numpy().view(np.uint16), sr_ref.reshape(-1))
    qw2, sc2 = W.unrepack(qw_r, sc_r, N, K, G)
    torch.cuda.synchronize()
    assert np.array_equal(qw2.cpu().numpy(), words)
    assert np.array_equal(sc2.cpu().numpy().view(np.uint16), scales)


def test_repack_of_workload_matrix():
    W = lib()
    d = inputs.generate(1, 1024, 1024, 128, seed=0)
    qw = torch.from_numpy(d["qweight"]).cuda()
    sc = torch.from_numpy(d["scales"].view(np.int16)).cuda()
    qw_r, sc_r = W.repack(qw, sc, 128)
    torch.cuda.synchronize()
    wr_ref, sr_ref = oracle.repack(d["qweight"], d["scales"], 128)
    assert np.array_equal(qw_r.cpu().numpy().view(np.uint32), wr_ref.reshape(-1))
    assert np.array_equal(sc_r.cpu().numpy().view(np.uint16), sr_ref.reshape(-1))
