"""GPU parity of qqmm (tcgen05 block-scaled FP4 GEMM) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import assert_close_to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


def quantized(mode, t):
    tb = synth.to_u16(t)
    gs = oracle.global_scale(tb) if mode == 2 else None
    q, s = oracle.quantize(tb, mode, gs)
    return q, s, gs


def run(B, mode, M, N, K, seed=0, mrows=None, ncols=None):
    x = synth.bf16_normal((M, K), 1.0, seed=seed)
    w = synth.bf16_normal((N, K), 0.02, seed=seed + 1)
    xq, xs, gx = quantized(mode, x)
    wq, ws, gw = quantized(mode, w)
    dev = lambda a: torch.from_numpy(a).cuda()
    gxd = torch.tensor(gx, dtype=torch.float32, device="cuda") if gx is not None else None
    gwd = torch.tensor(gw, dtype=torch.float32, device="cuda") if gw is not None else None
    out = B.qqmm(dev(xq.view(np.int32)), dev(oracle.tile_scales(xs)), dev(wq.view(np.int32)),
                 dev(oracle.tile_scales(ws)), gxd, gwd, mode=mode)
    alpha = np.float32(gx) * np.float32(gw) if mode == 2 else 1.0
    ref = oracle.qqmm(xq, xs, wq, ws, mode, alpha=alpha, mrows=mrows, ncols=ncols)
    if mrows is not None:
        out = out[torch.as_tensor(mrows).cuda()][:, torch.as_tensor(ncols).cuda()]
    return out, ref


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (128, 256, 256), (200, 264, 768), (300, 520, 1024),
                                   (64, 8, 256), (129, 512, 2048)])
def test_qqmm_small(B, mode, M, N, K):
    out, ref = run(B, mode, M, N, K, seed=M + N)
    assert_close_to_oracle(out, ref, f"qqmm mode {mode} {M}x{N}x{K}")


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("M", [1024, 2048])
def test_qqmm_prefill_full_size_sampled(B, mode, M):
    """The prefill GEMM M x 17408 x 5120 in the bench's launch configuration;
    the oracle computes a seeded sample of outputs across tiles and tails."""
    rng = np.random.default_rng(M)
    mrows = np.unique(np.concatenate([[0, 127, 128, M - 1], rng.integers(0, M, 28)]))
    ncols = np.unique(np.concatenate([[0, 255, 256, 17407], rng.integers(0, 17408, 60)]))
    out, ref = run(B, mode, M, 17408, 5120, seed=0, mrows=mrows, ncols=ncols)
    assert_close_to_oracle(out, ref, f"qqmm mode {mode} M={M}")


@pytest.mark.parametrize("mode", [2, 1])
def test_qqmm_prefill_m8192_sampled(B, mode):
    """The largest prefill GEMM, 8192 x 17408 x 5120, in the bench's launch
    configuration: more than 256 output rows (the first and last 128-row tiles
    in part, a tile boundary and random rows) against columns of the first and
    last 256-column tiles, a tile boundary and random columns."""
    M, N = 8192, 17408
    rng = np.random.default_rng(8192 + mode)
    mrows = np.unique(np.concatenate([np.arange(64), np.arange(120, 136), np.arange(M - 64, M),
                                      rng.integers(0, M, 128)]))
    assert len(mrows) >= 256
    ncols = np.unique(np.concatenate([np.arange(32), np.arange(250, 262), np.arange(N - 32, N),
                                      rng.integers(0, N, 40)]))
    out, ref = run(B, mode, M, N, 5120, seed=0, mrows=mrows, ncols=ncols)
    assert_close_to_oracle(out, ref, f"qqmm mode {mode} M={M}")


def test_qqmm_timeout_injection_reports_and_recovers(B):
    B.fp4_debug_inject_wait_timeout(True)
    try:
        out, ref = run(B, 2, 128, 256, 256, seed=9)
        assert B.fp4_check_device_error() == B.FP4_ERR_TIMEOUT
    finally:
        B.fp4_debug_inject_wait_timeout(False)
    assert_close_to_oracle(out, ref, "qqmm after injected timeout")
    out, ref = run(B, 2, 128, 256, 256, seed=9)
    assert B.fp4_check_device_error() == B.FP4_OK
    assert_close_to_oracle(out, ref, "qqmm after recovery")


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("shared_w", [False, True])
def test_qqmm_batched_matches_each_gemm(B, mode, shared_w):
    """qqmm_batched: every batch's output is the single FP4 x FP4 GEMM of its own
    operands and global scales (per-batch x, W either per batch or shared)."""
    Bt, M, N, K = 3, 200, 264, 512
    g = 16 if mode == 2 else 32
    xs, ws = [], []
    for b in range(Bt):
        xs.append(quantized(mode, synth.bf16_normal((M, K), 1.0 + b, seed=60 + b)))
        if b == 0 or not shared_w:
            ws.append(quantized(mode, synth.bf16_normal((N, K), 0.02, seed=70 + b)))
    dev = lambda a: torch.from_numpy(a).cuda()
    xq = dev(np.stack([x[0] for x in xs]).view(np.int32))
    sx = dev(np.stack([oracle.tile_scales(x[1]) for x in xs]))
    wq = dev(np.stack([w[0] for w in ws]).view(np.int32))
    sw = dev(np.stack([oracle.tile_scales(w[1]) for w in ws]))
    if shared_w:
        wq, sw = wq[0], sw[0]
    gx = gw = None
    if mode == 2:
        gx = torch.tensor([x[2] for x in xs], dtype=torch.float32, device="cuda")
        gw = torch.tensor([ws[0 if shared_w else b][2] for b in range(Bt)], dtype=torch.float32, device="cuda")
    out = B.qqmm_batched(xq, sx, wq, sw, gx, gw, mode=mode)
    for b in range(Bt):
        xq_b, xs_b, gx_b = xs[b]
        wq_b, ws_b, gw_b = ws[0 if shared_w else b]
        alpha = np.float32(gx_b) * np.float32(gw_b) if mode == 2 else 1.0
        ref = oracle.qqmm(xq_b, xs_b, wq_b, ws_b, mode, alpha=alpha)
        assert_close_to_oracle(out[b], ref, f"batched qqmm mode {mode} batch {b}")
