"""GPU parity of qqmm_quantize_x: the activation's global scale, quantization
and the FP4 x FP4 GEMM in one cooperative launch.  It must give bit for bit what
the separate entry points give (fp4_amax_global_scale, fp4_quantize with tiled
scales, qqmm), and match the oracle's GEMM of the oracle-quantized operands."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import assert_close_to_oracle, bf16_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


def separate(B, mode, x, wq, sw, gw, gx=None):
    if mode == 2 and gx is None:
        gx = B.fp4_amax_global_scale(x)
    xq, xs = B.fp4_quantize(x, mode, global_scale=gx, layout=B.SCALES_TILED)
    return B.qqmm(xq, xs, wq, sw, gx, gw, mode=mode), gx, xq, xs


@pytest.mark.parametrize("mode,static_gs", [(2, False), (2, True), (1, False)])
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (200, 264, 768), (1024, 17408, 5120), (300, 4096, 2048),
                                   (4096, 512, 5120), (2048, 17408, 5120), (8192, 17408, 5120)])
def test_fused_equals_separate_launches(B, mode, static_gs, M, N, K):
    """(4096, 512, 5120): each CTA's share of x is larger than the shared-memory
    ring, so the quantize pass streams part of it a second time.  M = 1024, 2048
    and 8192 x 17408 x 5120 are the shapes the bench times."""
    x = synth.activations_with_outliers(M, K, seed=M + K, outlier_seed=5).cuda()
    w = synth.bf16_normal((N, K), 0.02, seed=N, device="cuda")
    gw = B.fp4_amax_global_scale(w) if mode == 2 else None
    wq, sw = B.fp4_quantize(w, mode, global_scale=gw, layout=B.SCALES_TILED)
    gx_in = None
    if static_gs:  # a calibrated activation scale, deliberately not this x's amax / 2688
        gx_in = torch.tensor(float(x.abs().max().float()) / 2000.0, dtype=torch.float32, device="cuda")
    ref, gx, xq, xs = separate(B, mode, x, wq, sw, gw, gx_in)
    ws = B.qqmm_quantize_x_workspace(M, K, mode)
    gout = torch.empty((), dtype=torch.float32, device="cuda") if mode == 2 else None
    for call in range(2):  # the workspace's barrier words are reused by the second call
        out = B.qqmm_quantize_x(x, wq, sw, ws, gx_in, gw, mode=mode, global_scale_x_out=gout)
        torch.cuda.synchronize()
        assert B.fp4_check_device_error() == B.FP4_OK
        assert np.array_equal(bf16_u16(out), bf16_u16(ref)), f"call {call}"
        if mode == 2:
            assert gout.item() == gx.item()
    # the quantized x sits at the start of the workspace
    nq = M * K // 2
    assert torch.equal(ws[:nq], xq.view(torch.uint8).flatten())


def test_fused_matches_oracle(B):
    M, N, K = 130, 272, 1024
    x = synth.bf16_normal((M, K), 1.0, seed=1)
    w = synth.bf16_normal((N, K), 0.02, seed=2)
    xb, wb = synth.to_u16(x), synth.to_u16(w)
    gx, gw = oracle.global_scale(xb), oracle.global_scale(wb)
    oq, os_ = oracle.nvfp4_quantize(wb, gw)
    xq, xs = oracle.nvfp4_quantize(xb, gx)
    ref = oracle.qqmm(xq, xs, oq, os_, 2, alpha=np.float32(gx) * np.float32(gw))
    ws = B.qqmm_quantize_x_workspace(M, K, 2)
    out = B.qqmm_quantize_x(x.cuda(), torch.from_numpy(oq.view(np.int32)).cuda(),
                            torch.from_numpy(oracle.tile_scales(os_)).cuda(), ws, None,
                            torch.tensor(gw, dtype=torch.float32, device="cuda"), mode=2)
    assert_close_to_oracle(out, ref, "fused qqmm")


def test_fused_timeout_injection_reports_and_recovers(B):
    """A bounded wait made to expire inside the fused launch (the MMA thread's
    first wait, after the quantize prologue and both grid barriers): the call
    reports FP4_ERR_TIMEOUT, still writes the right product (the expiry is on a
    separate flag, so the protocol continues), and the same workspace serves the
    next call -- its grid-barrier word was left at a zero count."""
    M, N, K = 256, 512, 1024
    x = synth.bf16_normal((M, K), 1.0, seed=21, device="cuda")
    w = synth.bf16_normal((N, K), 0.02, seed=22, device="cuda")
    gw = B.fp4_amax_global_scale(w)
    wq, sw = B.fp4_quantize(w, 2, global_scale=gw, layout=B.SCALES_TILED)
    ref, _, _, _ = separate(B, 2, x, wq, sw, gw)
    ws = B.qqmm_quantize_x_workspace(M, K, 2)
    B.fp4_debug_inject_wait_timeout(True)
    try:
        out = B.qqmm_quantize_x(x, wq, sw, ws, None, gw, mode=2)
        torch.cuda.synchronize()
        assert B.fp4_check_device_error() == B.FP4_ERR_TIMEOUT
    finally:
        B.fp4_debug_inject_wait_timeout(False)
    assert np.array_equal(bf16_u16(out), bf16_u16(ref))
    out = B.qqmm_quantize_x(x, wq, sw, ws, None, gw, mode=2)
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    assert np.array_equal(bf16_u16(out), bf16_u16(ref))
