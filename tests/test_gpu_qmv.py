"""GPU parity of qmv (decode GEMV, W4A16) against the oracle's fp64 GEMV."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import assert_close_to_oracle

pytestmark = pytest.mark.gpu
GROUP = {0: 64, 1: 32, 2: 16}


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


def make_weights(mode, N, K, seed, group=None):
    """Quantized weights made by the oracle from seeded bf16 N(0, 0.02)."""
    w = synth.bf16_normal((N, K), 0.02, seed=seed)
    wb = synth.to_u16(w)
    g = group or GROUP[mode]
    gs = None
    b = None
    if mode == 0:
        q, s, b = oracle.affine_quantize(wb, g)
    elif mode == 2:
        gs = oracle.global_scale(wb)
        q, s = oracle.nvfp4_quantize(wb, gs)
    else:
        q, s = oracle.mxfp4_quantize(wb)
    return q, s, b, gs, g


def to_dev(mode, q, s, b, gs):
    qd = torch.from_numpy(q.view(np.int32)).cuda()
    sd = synth.from_u16(s, "cuda") if mode == 0 else torch.from_numpy(s).cuda()
    bd = synth.from_u16(b, "cuda") if b is not None else None
    gsd = torch.tensor(gs, dtype=torch.float32, device="cuda") if gs is not None else None
    return qd, sd, bd, gsd


@pytest.mark.parametrize("mode", [2, 1, 0])
@pytest.mark.parametrize("N,K", [(256, 512), (300, 1024), (33, 4096), (1, 64), (1000, 96)])
def test_qmv_small(B, mode, N, K):
    if K % GROUP[mode]:
        pytest.skip("K not a multiple of the group")
    q, s, b, gs, g = make_weights(mode, N, K, seed=N + K)
    x = synth.bf16_normal((K,), 1.0, seed=7)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    y = B.qmv(x.cuda(), qd, sd, bd, gsd, mode=mode, group_size=g)
    ref = oracle.qmv(synth.to_u16(x), q, s, b, mode, g, gs)
    assert_close_to_oracle(y, ref, f"qmv mode {mode} {N}x{K}")


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (9, 256), (129, 768), (1000, 2048), (20000, 512),
                                 (333, 1536), (40000, 256)])
def test_qmv_fp4_tensor_core_ragged_rows(B, mode, N, K):
    """Row counts that leave partial 8-row atoms per CTA, row blocks above 128
    rows (20000 rows: the B rows past 128 take the second scale group), and N
    above 256 rows per SM or K off the stage size (which take the mma.sync
    kernel)."""
    q, s, b, gs, g = make_weights(mode, N, K, seed=N)
    x = synth.activations_with_outliers(1, K, seed=3).view(-1)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=mode)
    assert_close_to_oracle(y, oracle.qmv(synth.to_u16(x), q, s, None, mode, g, gs), f"mode {mode} {N}x{K}")


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("N,K", [(64, 65536), (1024, 5120), (5000, 34816)])
def test_qmv_fp4_split_k_clusters(B, mode, N, K):
    """Shapes whose K is sliced across the CTAs of a cluster (partials summed
    through distributed shared memory), including K beyond one CTA's x slice."""
    q, s, b, gs, g = make_weights(mode, N, K, seed=N + 1)
    x = synth.activations_with_outliers(1, K, seed=11).view(-1)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=mode)
    rows = np.unique(np.concatenate([np.arange(min(N, 8)), N - 1 - np.arange(min(N, 8)),
                                     np.random.default_rng(N).integers(0, N, 120)]))
    ref = oracle.qmv(synth.to_u16(x), q, s, None, mode, g, gs, rows=rows)
    assert_close_to_oracle(y[torch.from_numpy(rows).cuda()], ref, f"mode {mode} {N}x{K}")


@pytest.mark.parametrize("mode", [2, 1, 0])
def test_qmv_nonfinite_activation_gives_nonfinite_rows(B, mode):
    """An infinity in x makes every row of the exact product non-finite (inf, or
    NaN where the weight is zero); the kernels return non-finite rows too."""
    N, K = 160, 512
    q, s, b, gs, g = make_weights(mode, N, K, seed=12)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    x = synth.bf16_normal((K,), 1.0, seed=13)
    x[300] = float("inf")
    ref = oracle.qmv(synth.to_u16(x), q, s, b, mode, g, gs)
    assert not np.isfinite(ref).any()
    y = B.qmv(x.cuda(), qd, sd, bd, gsd, mode=mode, group_size=g).float().cpu()
    assert not torch.isfinite(y).any()


@pytest.mark.parametrize("mode", [2, 1])
def test_qmv_fp4_tiny_and_huge_activations(B, mode):
    """x scaled far from 1 (the residual expansion's per-slice exponent)."""
    N, K = 256, 1024
    q, s, b, gs, g = make_weights(mode, N, K, seed=4)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    for scale in (2.0 ** -60, 2.0 ** -20, 1.0, 2.0 ** 30, 2.0 ** 100):
        x = (synth.bf16_normal((K,), 1.0, seed=5).float() * scale).to(torch.bfloat16)
        y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=mode)
        assert_close_to_oracle(y, oracle.qmv(synth.to_u16(x), q, s, None, mode, g, gs), f"scale {scale}")


@pytest.mark.parametrize("group", [32, 128])
def test_qmv_affine_other_groups(B, group):
    q, s, b, gs, g = make_weights(0, 96, 1024, seed=3, group=group)
    x = synth.bf16_normal((1024,), 1.0, seed=8)
    qd, sd, bd, gsd = to_dev(0, q, s, b, gs)
    y = B.qmv(x.cuda(), qd, sd, bd, None, mode=0, group_size=group)
    assert_close_to_oracle(y, oracle.qmv(synth.to_u16(x), q, s, b, 0, group), f"affine g{group}")


@pytest.mark.parametrize("mode", [2, 1, 0])
def test_qmv_one_hot_returns_dequantized_column(B, mode):
    N, K = 64, 512  # K = 512 runs both FP4 formats on the tensor-core path
    q, s, b, gs, g = make_weights(mode, N, K, seed=1)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    deq = oracle.dequantize_f64(q, s, b, mode, g, gs)
    for k in [0, 1, 8, 15, 31, 32, 255, 300, 511]:
        x = torch.zeros(K, dtype=torch.bfloat16)
        x[k] = 1.0
        y = B.qmv(x.cuda(), qd, sd, bd, gsd, mode=mode, group_size=g).float().cpu().double().numpy()
        ref = oracle.bf16_bits_to_f64(oracle.bf16_round_array(deq[:, k]))
        if mode == 2:
            # the tensor-core NVFP4 path expands x into NVFP4 residual terms (relative
            # error ~1e-5), so a bf16 rounding may land one ulp away
            assert np.all(np.abs(y - deq[:, k]) <= np.abs(deq[:, k]) * 2.0 ** -8 + 1e-30), k
        else:
            assert np.array_equal(y, ref), k


@pytest.mark.parametrize("mode", [2, 1, 0])
@pytest.mark.parametrize("proj", [0, 4, 6])
def test_qmv_decode_layer_shapes_sampled(B, mode, proj):
    """Full-size decode projections (q 5120x5120, gate 17408x5120, down
    5120x17408) in the launch configuration the bench uses; the oracle checks a
    seeded sample of rows."""
    name, N, K = synth.LAYER_PROJECTIONS[proj]
    q, s, b, gs, g = make_weights(mode, N, K, seed=synth.layer_seed(0, proj))
    x = synth.bf16_normal((K,), 1.0, seed=99)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    y = B.qmv(x.cuda(), qd, sd, bd, gsd, mode=mode, group_size=g)
    rows = np.unique(np.concatenate([np.arange(8), N - 1 - np.arange(8),
                                     np.random.default_rng(proj).integers(0, N, 240)]))
    ref = oracle.qmv(synth.to_u16(x), q, s, b, mode, g, gs, rows=rows)
    assert_close_to_oracle(y[torch.from_numpy(rows).cuda()], ref, f"{name} mode {mode}")


@pytest.mark.parametrize("mode", [2, 1])
def test_qmv_fp4_wide_row_blocks_every_row(B, mode):
    """Row blocks above 128 rows (W rows are the MMA's N, up to 256 per CTA):
    [34816, 2048] puts 230 rows in each of 152 blocks.  For MXFP4 a weight slot
    is then ~62 KB, the ring holds two, and the MMA commits free them (the
    path where the ring holds fewer slots than there are prep groups)."""
    N, K = 34816, 2048
    q, s, b, gs, g = make_weights(mode, N, K, seed=31 + mode)
    x = synth.activations_with_outliers(1, K, seed=5).view(-1)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=mode)
    assert_close_to_oracle(y, oracle.qmv(synth.to_u16(x), q, s, None, mode, g, gs), f"mode {mode} {N}x{K}")


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("N", [3 * synth.HIDDEN, 2 * 17408])
def test_qmv_fused_decode_shapes_sampled(B, mode, N):
    """The fused decode projections (q|k|v [15360, 5120], gate|up [34816, 5120])
    in the launch configuration the bench uses; the oracle checks a seeded
    sample of rows, including the first and last of the matrix."""
    K = synth.HIDDEN
    q, s, b, gs, g = make_weights(mode, N, K, seed=N + mode)
    x = synth.bf16_normal((K,), 1.0, seed=98)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=mode)
    rows = np.unique(np.concatenate([np.arange(8), N - 1 - np.arange(8),
                                     np.random.default_rng(N).integers(0, N, 240)]))
    ref = oracle.qmv(synth.to_u16(x), q, s, None, mode, g, gs, rows=rows)
    assert_close_to_oracle(y[torch.from_numpy(rows).cuda()], ref, f"fused {N}x{K} mode {mode}")


def test_weight_stream_ceiling_runs_clean(B):
    """The stream-only measurement kernel reads the decode shapes' weights as the
    tensor-core path does and leaves no device error behind."""
    for N, K in [(5120, 5120), (17408, 5120), (5120, 17408), (7, 256)]:
        w = synth.bf16_normal((N, K), 0.02, seed=N + K, device="cuda")
        gs = B.fp4_amax_global_scale(w)
        q, s = B.fp4_quantize(w, B.MODE_NVFP4, global_scale=gs)
        B.fp4_debug_stream_weights(q, s)
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK


@pytest.mark.parametrize("mode", [2, 1])
def test_qmv_timeout_injection_reports_and_recovers(B, mode):
    """The tensor-core GEMV's MMA thread first waits 1 ms on a barrier nothing
    arrives at: the kernel reports FP4_ERR_TIMEOUT and still returns the right y."""
    N, K = 512, 2048
    q, s, b, gs, g = make_weights(mode, N, K, seed=21)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    x = synth.bf16_normal((K,), 1.0, seed=22)
    ref = oracle.qmv(synth.to_u16(x), q, s, None, mode, g, gs)
    B.fp4_check_device_error()
    B.fp4_debug_inject_wait_timeout(True)
    try:
        y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=mode)
        torch.cuda.synchronize()
        assert B.fp4_check_device_error() == B.FP4_ERR_TIMEOUT
    finally:
        B.fp4_debug_inject_wait_timeout(False)
    assert_close_to_oracle(y, ref, f"qmv mode {mode} after injected timeout")
    y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=mode)
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    assert_close_to_oracle(y, ref, f"qmv mode {mode} after recovery")


def test_qmv_nvfp4_extreme_outlier_in_x(B):
    """One element of x 10^4 times the others: the term expansion's error is
    bounded by 2^-17 of its slice's max|x| per element, far inside the bar."""
    N, K = 1024, 5120
    q, s, b, gs, g = make_weights(2, N, K, seed=23)
    qd, sd, bd, gsd = to_dev(2, q, s, b, gs)
    x = synth.bf16_normal((K,), 1.0, seed=24)
    x[1234] = 1.0e4
    y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=2)
    assert_close_to_oracle(y, oracle.qmv(synth.to_u16(x), q, s, None, 2, 16, gs), "nvfp4 x outlier 1e4")


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("outlier", [1.0e3, 1.0e4])
def test_qmv_fp4_outlier_bound_per_row(B, mode, outlier):
    """The tensor-core GEMV's x expansion, checked row by row: one element of x
    is ``outlier`` times the N(0, 1) rest, and the rows whose weight code is 0
    at that column (their exact result does not see the outlier, y ~ 1) must
    still meet the expansion's stated bound, |y - y_exact| <= 2^-17 max|x|
    sum_k |deq(W)[n, k]| (the truncated radix-8 remainder of every element)
    plus half a bf16 ulp of the output and an fp32 accumulation allowance."""
    N, K, col = 1024, 5120, 1234
    q, s, b, gs, g = make_weights(mode, N, K, seed=40 + mode)
    qd, sd, bd, gsd = to_dev(mode, q, s, b, gs)
    x = synth.bf16_normal((K,), 1.0, seed=41)
    x[col] = outlier
    y = B.qmv(x.cuda(), qd, sd, None, gsd, mode=mode).float().cpu().double().numpy()
    xb = synth.to_u16(x)
    exact = oracle.qmv(xb, q, s, None, mode, g, gs)
    deq = oracle.dequantize_f64(q, s, None, mode, g, gs)
    code = (q[:, col // 8] >> np.uint32(4 * (col % 8))) & np.uint32(0x7)
    rows = np.nonzero(code == 0)[0]
    assert len(rows) >= 16, "too few rows with a zero code at the outlier's column"
    xf = oracle.bf16_bits_to_f64(xb)
    xmax = np.max(np.abs(xf))
    absw = np.abs(deq[rows]).sum(axis=1)
    absprod = np.abs(deq[rows] * xf[None, :]).sum(axis=1)
    mag = np.maximum(np.abs(exact[rows]), np.abs(y[rows]))
    half_ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.maximum(mag, 1e-300))) - 8), 0.0)
    bound = 2.0 ** -17 * xmax * absw + half_ulp + 2.0 ** -20 * absprod
    err = np.abs(y[rows] - exact[rows])
    worst = int(np.argmax(err / bound))
    assert np.all(err <= bound), (f"row {rows[worst]}: |y - exact| = {err[worst]:.3e} > bound {bound[worst]:.3e} "
                                  f"(exact {exact[rows[worst]]:.4f})")
