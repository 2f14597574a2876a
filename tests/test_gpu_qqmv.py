"""GPU parity of qqmv, the one-row quantized-activation GEMV ("mlx 0.30.7.3 ->
0.30.7.6", qqmm.cpp, QQMatmul::eval_gpu, one row with quantized W:
fp_quantize_dequantize of x, then the GEMV), against the oracle's composition
of its quantizer, bf16 dequantizer and fp64 GEMV."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import assert_close_to_oracle, bf16_u16

pytestmark = pytest.mark.gpu
GROUP = {1: 32, 2: 16}


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


def weights(mode, N, K, seed):
    wb = synth.to_u16(synth.bf16_normal((N, K), 0.02, seed=seed))
    gs = oracle.global_scale(wb) if mode == 2 else None
    q, s = oracle.quantize(wb, mode, gs)
    dev = (torch.from_numpy(q.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
           torch.tensor(gs, dtype=torch.float32, device="cuda") if gs is not None else None)
    return q, s, gs, dev


def run(B, mode, N, K, seed, use_gs_x, x=None, rows=None):
    q, s, gs, (qd, sd, gsd) = weights(mode, N, K, seed)
    if x is None:
        x = synth.activations_with_outliers(1, K, seed=seed + 1, outlier_seed=seed + 2).view(-1)
    xb = synth.to_u16(x)
    gx = oracle.global_scale(xb) if use_gs_x else None
    gxd = torch.tensor(gx, dtype=torch.float32, device="cuda") if gx is not None else None
    y = B.qqmv(x.cuda(), qd, sd, gxd, gsd, mode=mode)
    ref = oracle.qqmv(xb, q, s, mode, gx, gs, rows=rows)
    return (y if rows is None else y[torch.from_numpy(rows).cuda()]), ref, (x, qd, sd, gxd, gsd)


@pytest.mark.parametrize("mode,use_gs_x", [(2, True), (2, False), (1, False)])
@pytest.mark.parametrize("N,K", [(256, 512), (300, 1024), (33, 4096), (1000, 96), (7, 256), (20000, 512)])
def test_qqmv_shapes(B, mode, use_gs_x, N, K):
    """Tensor-core shapes (K a multiple of the stage, up to 256 rows per SM) and
    the mma.sync shapes (K = 96, MXFP4 K = 256), ragged row counts."""
    y, ref, _ = run(B, mode, N, K, seed=N + K, use_gs_x=use_gs_x)
    assert_close_to_oracle(y, ref, f"qqmv mode {mode} gs_x {use_gs_x} {N}x{K}")


@pytest.mark.parametrize("mode,use_gs_x", [(2, True), (1, False)])
def test_qqmv_is_qmv_of_the_dequantized_activation(B, mode, use_gs_x):
    """The fused route gives bit for bit what qmv gives on fp4_dequantize(
    fp4_quantize(x)) computed by the separate kernels: the in-kernel x_hat is the
    same bf16 vector and the GEMV arithmetic is the same."""
    for N, K in [(5120, 5120), (1000, 96)]:
        y, _, (x, qd, sd, gxd, gsd) = run(B, mode, N, K, seed=3, use_gs_x=use_gs_x)
        xd = x.cuda().view(1, -1)
        xq, xs = B.fp4_quantize(xd, mode, global_scale=gxd)
        xh = B.fp4_dequantize(xq, xs, mode=mode, global_scale=gxd).view(-1)
        y2 = B.qmv(xh, qd, sd, None, gsd, mode=mode)
        assert np.array_equal(bf16_u16(y), bf16_u16(y2)), (N, K)


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("N", [3 * synth.HIDDEN, synth.HIDDEN, 2 * synth.MLP])
def test_qqmv_fused_decode_shapes_sampled(B, mode, N):
    """The fused decode projections (q|k|v [15360, 5120], o [5120, 5120] with
    K split over clusters, gate|up [34816, 5120]) with an activation global
    scale for NVFP4; sampled rows."""
    rows = np.unique(np.concatenate([np.arange(8), N - 1 - np.arange(8),
                                     np.random.default_rng(N).integers(0, N, 240)]))
    y, ref, _ = run(B, mode, N, synth.HIDDEN, seed=N + mode, use_gs_x=(mode == 2), rows=rows)
    assert_close_to_oracle(y, ref, f"qqmv fused {N} mode {mode}")


@pytest.mark.parametrize("mode", [2, 1])
def test_qqmv_down_projection_split_k(B, mode):
    """K = 17408 (the down projection): the x blocks are quantized per CTA slice
    of a split-K cluster."""
    N, K = synth.HIDDEN, synth.MLP
    rows = np.unique(np.concatenate([np.arange(8), N - 1 - np.arange(8),
                                     np.random.default_rng(5).integers(0, N, 240)]))
    y, ref, _ = run(B, mode, N, K, seed=17, use_gs_x=(mode == 2), rows=rows)
    assert_close_to_oracle(y, ref, f"qqmv down mode {mode}")
