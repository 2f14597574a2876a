"""Pins of the oracle's one-row quantized-activation route (quantize x,
dequantize it to bf16, GEMV against 4-bit W), "mlx 0.30.7.3 -> 0.30.7.6",
qqmm.cpp, QQMatmul::eval_gpu (one row, quantized W: fp_quantize_dequantize then
fp_qmv).  Each pin is a property the definition fixes, checked against an
independent route through the oracle."""
import numpy as np
import pytest

import oracle
from block_scaled_fp4_fp_gb300 import synth


def weights(mode, N, K, seed):
    wb = synth.to_u16(synth.bf16_normal((N, K), 0.02, seed=seed))
    gs = oracle.global_scale(wb) if mode == oracle.MODE_NVFP4 else None
    q, s = oracle.quantize(wb, mode, gs)
    return q, s, gs


@pytest.mark.parametrize("mode,use_gs", [(2, True), (2, False), (1, False)])
def test_quantize_dequantize_is_idempotent(mode, use_gs):
    """x_hat quantizes to exactly the codes and scales x did: every block's
    largest element lands on code +-6 and the bf16 rounding of x_hat (only with
    a global scale) stays far inside the e2m1 and E4M3 steps."""
    x = synth.to_u16(synth.activations_with_outliers(64, 1024, seed=2, outlier_seed=3))
    gs = oracle.global_scale(x) if use_gs else None
    q0, s0 = oracle.quantize(x, mode, gs)
    xh = oracle.quantize_dequantize(x, mode, gs)
    q1, s1 = oracle.quantize(xh, mode, gs)
    assert np.array_equal(q0, q1) and np.array_equal(s0, s1)
    # and x_hat is the dequantized value, not x
    assert not np.array_equal(xh, x)


@pytest.mark.parametrize("mode", [2, 1])
def test_one_hot_x_returns_the_weight_column(mode):
    """A one-hot x of value 1 quantizes to code 6 under the largest scale and
    dequantizes back to exactly 1 (NVFP4: 6 * 448 * fl(1/2688) rounds to 1 in
    bf16), so y is column k of deq(W), exactly."""
    N, K = 48, 256
    q, s, gs = weights(mode, N, K, seed=5)
    deq = oracle.dequantize_f64(q, s, None, mode, oracle.GROUP_OF[mode], gs)
    for k in (0, 17, 128, 255):
        x = np.zeros(K, np.uint16)
        x[k] = 0x3F80  # bf16 1.0
        gx = oracle.global_scale(x) if mode == 2 else None
        xh = oracle.quantize_dequantize(x.reshape(1, -1), mode, gx)
        assert xh[0, k] == 0x3F80 and np.count_nonzero(xh) == 1
        y = oracle.qqmv(x, q, s, mode, gx, gs)
        assert np.array_equal(y, deq[:, k]), k


@pytest.mark.parametrize("mode", [2, 1])
def test_without_global_scale_it_is_the_one_row_qqmm(mode):
    """With no activation global scale (MXFP4 has none) x_hat is exactly
    code * block scale, so the route equals the FP4 x FP4 product qqmm computes
    for one row (a different oracle function: code-times-scale products, alpha
    epilogue), up to fp64 summation order."""
    N, K = 40, 512
    q, s, gs = weights(mode, N, K, seed=7)
    x = synth.to_u16(synth.bf16_normal((1, K), 1.0, seed=8))
    xq, xs = oracle.quantize(x, mode, None)
    y = oracle.qqmv(x, q, s, mode, None, gs)
    ref = oracle.qqmm(xq, xs, q, s, mode, alpha=gs if gs is not None else 1.0)[0]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_nvfp4_global_scale_rounds_x_hat_to_bf16():
    """With an activation global scale x_hat = bf16(code * s8 * gs): the route
    differs from the unrounded W4A4 product by at most the bf16 half-ulp of each
    x_hat element (relative 2^-9) times |W|, and it does differ."""
    N, K = 40, 512
    q, s, gs = weights(2, N, K, seed=9)
    x = synth.to_u16(synth.bf16_normal((1, K), 1.0, seed=10))
    gx = oracle.global_scale(x)
    xq, xs = oracle.quantize(x, 2, gx)
    y = oracle.qqmv(x, q, s, 2, gx, gs)
    xe = oracle.dequantize_f64(xq, xs, None, 2, 16, gx)[0]
    wd = oracle.dequantize_f64(q, s, None, 2, 16, gs)
    exact = wd @ xe
    bound = (np.abs(xe)[None, :] * 2.0 ** -9 * np.abs(wd)).sum(axis=1) + 1e-12 * np.abs(exact).max()
    assert np.all(np.abs(y - exact) <= bound)
    assert np.any(y != exact)
