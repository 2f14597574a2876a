"""GPU parity of gather_qmm (MoE grouped W4A16 GEMM, MXFP4 experts)."""
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


def run(B, tokens, E, topk, N, K, seed=0, rows=None):
    lhs, rhs = synth.moe_routing(tokens, E, topk, seed=seed)
    x = synth.bf16_normal((tokens, K), 1.0, seed=seed + 1)
    w = synth.bf16_normal((E * N, K), 0.02, seed=seed + 2)
    q, s = oracle.mxfp4_quantize(synth.to_u16(w))
    q3, s3 = q.reshape(E, N, K // 8), s.reshape(E, N, K // 32)
    out = B.gather_qmm(x.cuda(), torch.from_numpy(lhs).cuda(), torch.from_numpy(rhs).cuda(),
                       torch.from_numpy(q3.view(np.int32)).cuda(), torch.from_numpy(s3).cuda())
    ref = oracle.gather_qmm(synth.to_u16(x), lhs, rhs, q3, s3, None, oracle.MODE_MXFP4, 32, rows=rows)
    if rows is not None:
        out = out[torch.as_tensor(rows).cuda()]
    return out, ref


@pytest.mark.parametrize("tokens,E,topk,N,K", [(16, 4, 2, 64, 128), (300, 8, 4, 272, 256), (64, 32, 4, 512, 192)])
def test_gather_small(B, tokens, E, topk, N, K):
    out, ref = run(B, tokens, E, topk, N, K, seed=tokens)
    assert_close_to_oracle(out, ref, f"gather {tokens}x{E}x{N}x{K}")


def test_gather_moe_full_size_sampled(B):
    """2048 tokens, 32 experts, top-4, gate/up 5760 x 2880; sampled routed rows
    (first/last of several expert segments and random ones)."""
    lhs, rhs = synth.moe_routing(2048, 32, 4, seed=0)
    starts = np.searchsorted(rhs, np.arange(32))
    rows = np.unique(np.concatenate([starts[:6], starts[1:7] - 1, [len(rhs) - 1],
                                     np.random.default_rng(0).integers(0, len(rhs), 8)]))
    out, ref = run(B, 2048, 32, 4, 5760, 2880, seed=0, rows=rows)
    assert_close_to_oracle(out, ref, "gather gate/up full size")


def test_gather_moe_down_full_size_sampled(B):
    """The MoE down projection as the bench runs it: 8192 routed rows already in
    expert order (lhs is the identity), 32 experts of 2880 x 2880 MXFP4 weights;
    sampled rows: the first and last rows of expert segments and random ones."""
    _, rhs = synth.moe_routing(2048, 32, 4, seed=0)
    R, E, N, K = len(rhs), 32, 2880, 2880
    lhs = np.arange(R, dtype=np.int32)
    x = synth.bf16_normal((R, K), 1.0, seed=3)
    w = synth.bf16_normal((E * N, K), 0.02, seed=4)
    q, s = oracle.mxfp4_quantize(synth.to_u16(w))
    q3, s3 = q.reshape(E, N, K // 8), s.reshape(E, N, K // 32)
    out = B.gather_qmm(x.cuda(), torch.from_numpy(lhs).cuda(), torch.from_numpy(rhs).cuda(),
                       torch.from_numpy(q3.view(np.int32)).cuda(), torch.from_numpy(s3).cuda())
    starts = np.searchsorted(rhs, np.arange(E))
    rows = np.unique(np.concatenate([starts[::4], starts[1::4] - 1, [0, R - 1],
                                     np.random.default_rng(3).integers(0, R, 16)]))
    ref = oracle.gather_qmm(synth.to_u16(x), lhs, rhs, q3, s3, None, oracle.MODE_MXFP4, 32, rows=rows)
    assert_close_to_oracle(out[torch.as_tensor(rows).cuda()], ref, "gather down full size")


def test_gather_segments_on_tile_boundaries(B):
    """Hand-built routing whose expert segments are empty, one row, and 127 /
    128 / 129 / 255 / 256 / 257 / 383 / 384 / 385 / 513 / 769 rows long, so the
    tiles of up to 256 rows (two 128-row MMA halves) start, end and straddle
    every boundary case: one half, both halves, a one-row tail; activation rows
    repeat and come in any order (the 16-byte gather path)."""
    E, N, K = 14, 96, 128
    sizes = [0, 1, 127, 128, 0, 129, 255, 256, 257, 383, 384, 385, 513, 769]
    rhs = np.repeat(np.arange(E, dtype=np.int32), sizes)
    R = len(rhs)
    tokens = 200
    lhs = np.random.default_rng(5).integers(0, tokens, R).astype(np.int32)
    x = synth.bf16_normal((tokens, K), 1.0, seed=6)
    w = synth.bf16_normal((E * N, K), 0.02, seed=7)
    q, s = oracle.mxfp4_quantize(synth.to_u16(w))
    q3, s3 = q.reshape(E, N, K // 8), s.reshape(E, N, K // 32)
    out = B.gather_qmm(x.cuda(), torch.from_numpy(lhs).cuda(), torch.from_numpy(rhs).cuda(),
                       torch.from_numpy(q3.view(np.int32)).cuda(), torch.from_numpy(s3).cuda())
    ref = oracle.gather_qmm(synth.to_u16(x), lhs, rhs, q3, s3, None, oracle.MODE_MXFP4, 32)
    assert_close_to_oracle(out, ref, "gather tile-boundary segments")


def test_gather_timeout_injection_reports_and_recovers(B):
    B.fp4_check_device_error()
    B.fp4_debug_inject_wait_timeout(True)
    try:
        out, ref = run(B, 16, 4, 2, 64, 128, seed=31)
        torch.cuda.synchronize()
        assert B.fp4_check_device_error() == B.FP4_ERR_TIMEOUT
    finally:
        B.fp4_debug_inject_wait_timeout(False)
    assert_close_to_oracle(out, ref, "gather after injected timeout")
    out, ref = run(B, 16, 4, 2, 64, 128, seed=31)
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    assert_close_to_oracle(out, ref, "gather after recovery")


@pytest.mark.parametrize("bad", ["out_of_range", "negative", "unsorted"])
def test_gather_routing_contract_violation_is_reported(B, bad):
    """Expert ids live in device memory, so the kernel checks them: an id outside
    [0, E) or a decreasing pair is reported by fp4_check_device_error as an
    invalid argument (the rows it affects get no tile; every access stays inside
    the buffers), and the next valid call reports nothing."""
    tokens, E, N, K = 32, 4, 64, 128
    lhs = np.arange(tokens, dtype=np.int32)
    rhs = np.repeat(np.arange(E, dtype=np.int32), tokens // E)
    if bad == "out_of_range":
        rhs[-1] = E
    elif bad == "negative":
        rhs[0] = -1
    else:
        rhs[3], rhs[20] = rhs[20], rhs[3]
    x = synth.bf16_normal((tokens, K), 1.0, seed=51).cuda()
    w = synth.bf16_normal((E * N, K), 0.02, seed=52)
    q, s = oracle.mxfp4_quantize(synth.to_u16(w))
    q3 = torch.from_numpy(q.reshape(E, N, K // 8).view(np.int32)).cuda()
    s3 = torch.from_numpy(s.reshape(E, N, K // 32)).cuda()
    B.fp4_check_device_error()
    B.gather_qmm(x, torch.from_numpy(lhs).cuda(), torch.from_numpy(rhs).cuda(), q3, s3)
    assert B.fp4_check_device_error() == B.FP4_ERR_INVALID_ARG
    good = np.repeat(np.arange(E, dtype=np.int32), tokens // E)
    B.gather_qmm(x, torch.from_numpy(lhs).cuda(), torch.from_numpy(good).cuda(), q3, s3)
    assert B.fp4_check_device_error() == B.FP4_OK


@pytest.mark.parametrize("scatter", [False, True])
def test_gather_contiguous_rows_tma_path(B, scatter):
    """Activations already in routed order: every tile's rows are consecutive rows
    of x (starting 7 rows in, x longer than the routing), so the full 128-row
    halves arrive by TMA boxes and a partial last half by the 16-byte gather.
    With `scatter`, one expert's segment has two rows swapped, so that tile
    falls back to the gather while the others keep the TMA path."""
    E, N, K = 12, 160 + 48, 192
    sizes = [1, 127, 128, 129, 256, 257, 383, 384, 385, 0, 513, 200]
    rhs = np.repeat(np.arange(E, dtype=np.int32), sizes)
    R = len(rhs)
    lhs = (np.arange(R) + 7).astype(np.int32)
    if scatter:
        a = sum(sizes[:6]) + 10
        lhs[a], lhs[a + 100] = lhs[a + 100], lhs[a]
    x = synth.bf16_normal((R + 20, K), 1.0, seed=61)
    w = synth.bf16_normal((E * N, K), 0.02, seed=62)
    q, s = oracle.mxfp4_quantize(synth.to_u16(w))
    q3, s3 = q.reshape(E, N, K // 8), s.reshape(E, N, K // 32)
    out = B.gather_qmm(x.cuda(), torch.from_numpy(lhs).cuda(), torch.from_numpy(rhs).cuda(),
                       torch.from_numpy(q3.view(np.int32)).cuda(), torch.from_numpy(s3).cuda())
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    ref = oracle.gather_qmm(synth.to_u16(x), lhs, rhs, q3, s3, None, oracle.MODE_MXFP4, 32)
    assert_close_to_oracle(out, ref, f"gather contiguous rows (scatter={scatter})")


@pytest.mark.parametrize("T,R,K", [(1, 1, 8), (37, 300, 2880), (2048, 8192, 2880), (5, 64, 4104)])
def test_gather_rows_bit_exact(B, T, R, K):
    """gather_rows moves bf16 rows into routing order: bit-exact against the
    oracle's indexing (ragged K, repeated and arbitrary indices)."""
    x = synth.bf16_normal((T, K), 1.0, seed=T + K)
    idx = np.random.default_rng(R).integers(0, T, R).astype(np.int32)
    out = B.gather_rows(x.cuda(), torch.from_numpy(idx).cuda())
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    ref = oracle.gather_rows(synth.to_u16(x), idx)
    assert np.array_equal(synth.to_u16(out.cpu()), ref)


def test_gather_rows_bad_index_is_reported(B):
    """An index outside [0, x_rows) leaves its row unwritten and is reported;
    the other rows are still moved, and the next valid call reports nothing."""
    T, R, K = 10, 6, 64
    x = synth.bf16_normal((T, K), 1.0, seed=71).cuda()
    idx = torch.tensor([0, 9, -1, 3, 10, 4], dtype=torch.int32).cuda()
    out = torch.full((R, K), 7.0, dtype=torch.bfloat16).cuda()
    B.fp4_check_device_error()
    B.gather_rows(x, idx, out=out)
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_ERR_INVALID_ARG
    for i, j in enumerate([0, 9, None, 3, None, 4]):
        if j is None:
            assert bool((out[i] == 7.0).all())
        else:
            assert torch.equal(out[i], x[j])
    B.gather_rows(x, idx.clamp(0, T - 1), out=out)
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
