"""Pins of the oracle's dense W4A16 GEMM (qmm: bf16 x [M, K] against 4-bit W
[N, K]), each against a route that does not go through it."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth

GROUP = {0: 64, 1: 32, 2: 16}


def weights(mode, N, K, seed, group=None):
    wb = synth.to_u16(synth.bf16_normal((N, K), 0.02, seed=seed))
    g = group or GROUP[mode]
    if mode == 0:
        q, s, b = oracle.affine_quantize(wb, g)
        return q, s, b, None, g
    gs = oracle.global_scale(wb) if mode == 2 else None
    q, s = oracle.quantize(wb, mode, gs)
    return q, s, None, gs, g


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_qmm_rows_are_qmv(mode):
    """Row m of the GEMM is the GEMV of x[m] (the pinned oracle qmv), exactly."""
    q, s, b, gs, g = weights(mode, 24, 256, seed=1)
    x = synth.to_u16(synth.bf16_normal((5, 256), 1.0, seed=2))
    out = oracle.qmm(x, q, s, b, mode, g, gs)
    for m in range(5):
        assert np.array_equal(out[m], oracle.qmv(x[m], q, s, b, mode, g, gs))
    sub = oracle.qmm(x, q, s, b, mode, g, gs, rows=[4, 1])
    assert np.array_equal(sub, out[[4, 1]])


@pytest.mark.parametrize("mode", [0, 1])
def test_qmm_is_gather_with_identity_routing(mode):
    q, s, b, gs, g = weights(mode, 32, 128, seed=3)
    x = synth.to_u16(synth.bf16_normal((7, 128), 1.0, seed=4))
    out = oracle.qmm(x, q, s, b, mode, g, gs)
    ref = oracle.gather_qmm(x, np.arange(7, dtype=np.int32), np.zeros(7, np.int32), q[None], s[None],
                            None if b is None else b[None], mode, g)
    assert np.array_equal(out, ref)


def test_qmm_integer_weights_and_activations_are_exact():
    """MXFP4 codes under scale byte 127 (2^0) are the e2m1 values; with small
    integer x every product and sum is exact, so the GEMM equals an integer
    matmul of the decoded codes (orientation out[m, n] = x[m] . W[n])."""
    rng = np.random.default_rng(5)
    M, N, K = 6, 10, 64
    codes = rng.integers(0, 16, (N, K))
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])[codes]
    q = np.zeros((N, K // 8), np.uint32)
    for k in range(K):
        q[:, k // 8] |= (codes[:, k].astype(np.uint32) << np.uint32(4 * (k % 8)))
    s = np.full((N, K // 32), 127, np.uint8)
    xi = rng.integers(-8, 9, (M, K)).astype(np.float32)
    xb = synth.to_u16(torch.from_numpy(xi).to(torch.bfloat16))
    out = oracle.qmm(xb, q, s, None, 1, 32)
    assert np.array_equal(out, xi.astype(np.float64) @ vals.T)
