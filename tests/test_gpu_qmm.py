"""GPU parity of qmm, the dense W4A16 prefill GEMM (bf16 x [M, K] against
NVFP4, MXFP4 or affine-4 W [N, K]), and of gather_qmm's NVFP4 and affine
experts, against the oracle's fp64 GEMMs."""
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


def weights(mode, N, K, seed, group=None, use_gs=True):
    wb = synth.to_u16(synth.bf16_normal((N, K), 0.02, seed=seed))
    g = group or GROUP[mode]
    b = gs = None
    if mode == 0:
        q, s, b = oracle.affine_quantize(wb, g)
    else:
        gs = oracle.global_scale(wb) if (mode == 2 and use_gs) else None
        q, s = oracle.quantize(wb, mode, gs)
    dev = (torch.from_numpy(q.view(np.int32)).cuda(),
           synth.from_u16(s, "cuda") if mode == 0 else torch.from_numpy(s).cuda(),
           synth.from_u16(b, "cuda") if b is not None else None,
           torch.tensor(gs, dtype=torch.float32, device="cuda") if gs is not None else None)
    return (q, s, b, gs, g), dev


@pytest.mark.parametrize("mode,group", [(2, 16), (1, 32), (0, 64), (0, 32), (0, 128)])
@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (100, 272, 512), (256, 256, 256), (300, 48, 1024), (129, 512, 64),
                                   (1000, 272, 512)])
def test_qmm_small(B, mode, group, M, N, K):
    """Ragged shapes: one row, rows ending inside the first or second 256-row
    half of a 512-row tile (and a second tile ending inside its last quarter),
    columns ending inside a 256-column slice, K of one 64-code stage."""
    if K % group:
        pytest.skip("K not a multiple of the group")
    (q, s, b, gs, g), (qd, sd, bd, gsd) = weights(mode, N, K, seed=M + N + K, group=group)
    x = synth.bf16_normal((M, K), 1.0, seed=M)
    out = B.qmm(x.cuda(), qd, sd, bd, gsd, mode=mode, group_size=g)
    ref = oracle.qmm(synth.to_u16(x), q, s, b, mode, g, gs)
    assert_close_to_oracle(out, ref, f"qmm mode {mode} g{g} {M}x{N}x{K}")


def test_qmm_nvfp4_without_global_scale(B):
    (q, s, b, gs, g), (qd, sd, bd, gsd) = weights(2, 272, 512, seed=9, use_gs=False)
    x = synth.bf16_normal((300, 512), 1.0, seed=10)
    out = B.qmm(x.cuda(), qd, sd, None, None, mode=2)
    assert_close_to_oracle(out, oracle.qmm(synth.to_u16(x), q, s, None, 2, 16, None), "qmm nvfp4 no gs")


@pytest.mark.parametrize("mode", [2, 1, 0])
@pytest.mark.parametrize("M", [1024, 2048, 8192])
def test_qmm_prefill_full_size_sampled(B, mode, M):
    """The prefill shapes M x 17408 x 5120 in the bench's launch configuration;
    sampled rows (first and last of the matrix, the 128-row blocks of both CTAs
    of a pair and both 256-row halves of a 512-row tile, random), every column."""
    N, K = 17408, 5120
    (q, s, b, gs, g), (qd, sd, bd, gsd) = weights(mode, N, K, seed=1)
    x = synth.bf16_normal((M, K), 1.0, seed=2)
    out = B.qmm(x.cuda(), qd, sd, bd, gsd, mode=mode)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, 383, 384, 511, 512, M - 1],
                                     np.random.default_rng(M).integers(0, M, 18)]))
    ref = oracle.qmm(synth.to_u16(x), q, s, b, mode, g, gs, rows=rows)
    assert_close_to_oracle(out[torch.from_numpy(rows).cuda()], ref, f"qmm mode {mode} M={M}")


@pytest.mark.parametrize("mode", [2, 0])
def test_gather_qmm_nvfp4_and_affine_experts(B, mode):
    tokens, E, topk, N, K = 300, 8, 4, 272, 256
    lhs, rhs = synth.moe_routing(tokens, E, topk, seed=3)
    x = synth.bf16_normal((tokens, K), 1.0, seed=4)
    wb = synth.to_u16(synth.bf16_normal((E * N, K), 0.02, seed=5))
    g = GROUP[mode]
    if mode == 0:
        q, s, b = oracle.affine_quantize(wb, g)
        sd, bd = synth.from_u16(s.reshape(E, N, K // g), "cuda"), synth.from_u16(b.reshape(E, N, K // g), "cuda")
        b3 = b.reshape(E, N, K // g)
    else:
        q, s = oracle.quantize(wb, mode, None)
        sd, bd, b3 = torch.from_numpy(s.reshape(E, N, K // g)).cuda(), None, None
    q3, s3 = q.reshape(E, N, K // 8), s.reshape(E, N, K // g)
    out = B.gather_qmm(x.cuda(), torch.from_numpy(lhs).cuda(), torch.from_numpy(rhs).cuda(),
                       torch.from_numpy(q3.view(np.int32)).cuda(), sd, bd, mode=mode, group_size=g)
    ref = oracle.gather_qmm(synth.to_u16(x), lhs, rhs, q3, s3, b3, mode, g)
    assert_close_to_oracle(out, ref, f"gather mode {mode}")


def test_qmm_timeout_injection_reports_and_recovers(B):
    """The MMA thread waits 1 ms on a barrier nothing arrives at: the call still
    gives the right product and reports FP4_ERR_TIMEOUT; the next call reports
    nothing."""
    (q, s, b, gs, g), (qd, sd, bd, gsd) = weights(2, 272, 512, seed=5)
    x = synth.bf16_normal((600, 512), 1.0, seed=6)
    ref = oracle.qmm(synth.to_u16(x), q, s, b, 2, g, gs)
    B.fp4_debug_inject_wait_timeout(True)
    try:
        out = B.qmm(x.cuda(), qd, sd, bd, gsd, mode=2)
        torch.cuda.synchronize()
        assert B.fp4_check_device_error() == B.FP4_ERR_TIMEOUT
    finally:
        B.fp4_debug_inject_wait_timeout(False)
    assert_close_to_oracle(out, ref, "qmm after injected timeout")
    out = B.qmm(x.cuda(), qd, sd, bd, gsd, mode=2)
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    assert_close_to_oracle(out, ref, "qmm after recovery")
