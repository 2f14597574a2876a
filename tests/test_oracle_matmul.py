"""Pins for the oracle's matmuls (CPU only): one-hot probes, exact small-integer
products, brute force in exact rationals, dequantize-then-matmul equivalence
with the alpha epilogue, and gather routing."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth

E2M1 = [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def pack(codes):
    codes = np.asarray(codes, np.uint32)
    rows, cols = codes.shape
    q = np.zeros((rows, cols // 8), np.uint32)
    for j in range(8):
        q |= codes[:, j::8] << np.uint32(4 * j)
    return q


@pytest.mark.parametrize("mode,group", [(oracle.MODE_NVFP4, 16), (oracle.MODE_MXFP4, 32),
                                        (oracle.MODE_AFFINE, 64)])
def test_qmv_one_hot_returns_dequantized_column(mode, group):
    N, K = 48, 128
    w = synth.bf16_normal((N, K), 0.02, seed=1)
    wb = synth.to_u16(w)
    gs = None
    if mode == oracle.MODE_NVFP4:
        gs = oracle.global_scale(wb)
        q, s = oracle.nvfp4_quantize(wb, gs)
        b = None
    elif mode == oracle.MODE_MXFP4:
        q, s = oracle.mxfp4_quantize(wb)
        b = None
    else:
        q, s, b = oracle.affine_quantize(wb, group)
    deq = oracle.dequantize_f64(q, s, b, mode, group, gs)
    for k in [0, 1, 7, 8, 15, 16, 31, 63, 64, 127]:
        x = np.zeros(K)
        x[k] = 1.0
        y = oracle.qmv(synth.to_u16(torch.tensor(x).to(torch.bfloat16)), q, s, b, mode, group, gs)
        assert np.array_equal(y, deq[:, k]), k


def test_qmv_integer_weights_are_exact():
    # unit scales (E4M3 0x38 = 1.0) and gs = 1: deq(W) = e2m1 codes, x small integers.
    rng = np.random.default_rng(0)
    N, K = 64, 256
    codes = rng.integers(0, 16, size=(N, K))
    q = pack(codes)
    s = np.full((N, K // 16), 0x38, np.uint8)
    xi = rng.integers(-8, 9, size=K).astype(np.float64)
    xb = synth.to_u16(torch.tensor(xi).to(torch.bfloat16))
    vals = np.array([(-1 if c & 8 else 1) * E2M1[c & 7] for c in codes.ravel()]).reshape(N, K)
    want = vals @ xi  # every partial sum is a multiple of 0.5 below 2^20: exact in fp64
    got = oracle.qmv(xb, q, s, None, oracle.MODE_NVFP4, 16, None)
    assert np.array_equal(got, want)


def test_qmv_row_subset_and_transpose_orientation():
    N, K = 40, 64
    w = synth.bf16_normal((N, K), 0.02, seed=9)
    x = synth.bf16_normal((1, K), 1.0, seed=10)
    wb, xb = synth.to_u16(w), synth.to_u16(x)
    q, s = oracle.mxfp4_quantize(wb)
    deq = oracle.dequantize_f64(q, s, None, oracle.MODE_MXFP4, 32)
    full = oracle.qmv(xb, q, s, None, oracle.MODE_MXFP4, 32)
    ref = deq @ x.double().numpy().ravel()  # W stored [N, K]: y = W x
    np.testing.assert_allclose(full, ref, rtol=1e-12, atol=1e-15)
    rows = [39, 0, 17]
    assert np.array_equal(oracle.qmv(xb, q, s, None, oracle.MODE_MXFP4, 32, rows=rows), full[rows])


def _exact_qqmm(cx, sx, cw, sw, group, scale_dec):
    M, K = cx.shape
    N = cw.shape[0]
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = Fraction((-1 if cx[m, k] & 8 else 1) * E2M1[cx[m, k] & 7]) * scale_dec(sx[m, k // group])
                b = Fraction((-1 if cw[n, k] & 8 else 1) * E2M1[cw[n, k] & 7]) * scale_dec(sw[n, k // group])
                acc += a * b
            out[m][n] = acc
    return out


@pytest.mark.parametrize("K", [16, 32, 64])
@pytest.mark.parametrize("mode", [oracle.MODE_NVFP4, oracle.MODE_MXFP4])
def test_qqmm_brute_force_exact_rationals(K, mode):
    group = 16 if mode == oracle.MODE_NVFP4 else 32
    if K % group:
        pytest.skip("K must be a multiple of the group")
    rng = np.random.default_rng(K + mode)
    M, N = 3, 5
    cx = rng.integers(0, 16, size=(M, K))
    cw = rng.integers(0, 16, size=(N, K))
    if mode == oracle.MODE_NVFP4:
        sx = rng.integers(0x20, 0x50, size=(M, K // group)).astype(np.uint8)
        sw = rng.integers(0x20, 0x50, size=(N, K // group)).astype(np.uint8)
        dec = lambda b: Fraction(oracle.e4m3_decode(int(b)))
    else:
        sx = rng.integers(110, 140, size=(M, K // group)).astype(np.uint8)
        sw = rng.integers(110, 140, size=(N, K // group)).astype(np.uint8)
        dec = lambda b: Fraction(2) ** (int(b) - 127)
    got = oracle.qqmm(pack(cx), sx, pack(cw), sw, mode, alpha=1.0)
    want = _exact_qqmm(cx, sx, cw, sw, group, dec)
    for m in range(M):
        for n in range(N):
            assert Fraction(got[m, n]) == want[m][n]


def test_qqmm_alpha_epilogue_equals_dequantize_then_matmul():
    M, N, K = 20, 36, 128
    x = synth.bf16_normal((M, K), 1.0, seed=0)
    w = synth.bf16_normal((N, K), 0.02, seed=1)
    xb, wb = synth.to_u16(x), synth.to_u16(w)
    gx, gw = oracle.global_scale(xb), oracle.global_scale(wb)
    qx, sx = oracle.nvfp4_quantize(xb, gx)
    qw, sw = oracle.nvfp4_quantize(wb, gw)
    alpha = oracle.alpha_from_amax(oracle.amax(xb), oracle.amax(wb))
    out = oracle.qqmm(qx, sx, qw, sw, oracle.MODE_NVFP4, alpha=np.float32(gx) * np.float32(gw))
    ref = oracle.dequantize_f64(qx, sx, None, 2, 16, gx) @ oracle.dequantize_f64(qw, sw, None, 2, 16, gw).T
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-9 * np.abs(ref).max())
    # the alpha of the pages' formula agrees with gs_x * gs_w to a few fp32 ulps
    assert alpha == pytest.approx(float(np.float32(gx)) * float(np.float32(gw)), rel=4 * 2 ** -23)
    # sub-block selection
    sub = oracle.qqmm(qx, sx, qw, sw, 2, alpha=1.0, mrows=[19, 2], ncols=[35, 0, 7])
    fullu = oracle.qqmm(qx, sx, qw, sw, 2, alpha=1.0)
    assert np.array_equal(sub, fullu[np.ix_([19, 2], [35, 0, 7])])


def test_gather_qmm_routes_rows_to_experts():
    E, N, K, T = 4, 24, 64, 6
    w = synth.bf16_normal((E * N, K), 0.02, seed=2)
    q, s = oracle.mxfp4_quantize(synth.to_u16(w))
    q3 = q.reshape(E, N, K // 8)
    s3 = s.reshape(E, N, K // 32)
    x = synth.bf16_normal((T, K), 1.0, seed=3)
    xb = synth.to_u16(x)
    lhs = np.array([0, 3, 5, 1, 0, 2], np.int32)
    rhs = np.array([0, 0, 1, 2, 3, 3], np.int32)
    out = oracle.gather_qmm(xb, lhs, rhs, q3, s3, None, oracle.MODE_MXFP4, 32)
    for r in range(len(lhs)):
        y = oracle.qmv(xb[lhs[r]], q3[rhs[r]], s3[rhs[r]], None, oracle.MODE_MXFP4, 32)
        assert np.array_equal(out[r], y)
    sub = oracle.gather_qmm(xb, lhs, rhs, q3, s3, None, oracle.MODE_MXFP4, 32, rows=[5, 1])
    assert np.array_equal(sub, out[[5, 1]])


def test_gather_rows_is_row_indexing_and_commutes_with_gather_qmm():
    """gather_rows against a plain loop over the index list, and the identity the
    routed-order path relies on: gather_qmm over x with routing lhs equals
    gather_qmm over gather_rows(x, lhs) with the identity routing."""
    T, K = 7, 16
    x = synth.to_u16(synth.bf16_normal((T, K), 1.0, seed=11))
    idx = np.array([6, 0, 0, 3, 6, 2, 5], np.int32)
    g = oracle.gather_rows(x, idx)
    assert g.dtype == np.uint16 and g.shape == (len(idx), K)
    for i, j in enumerate(idx):
        for k in range(K):
            assert g[i, k] == x[j, k]
    E, N, K2 = 3, 16, 64
    w = synth.bf16_normal((E * N, K2), 0.02, seed=12)
    q, s = oracle.mxfp4_quantize(synth.to_u16(w))
    q3, s3 = q.reshape(E, N, K2 // 8), s.reshape(E, N, K2 // 32)
    xb = synth.to_u16(synth.bf16_normal((T, K2), 1.0, seed=13))
    lhs = np.array([4, 1, 1, 6, 0, 2, 3, 5], np.int32)
    rhs = np.array([0, 0, 0, 1, 1, 2, 2, 2], np.int32)
    a = oracle.gather_qmm(xb, lhs, rhs, q3, s3, None, oracle.MODE_MXFP4, 32)
    b = oracle.gather_qmm(oracle.gather_rows(xb, lhs), np.arange(len(lhs), dtype=np.int32), rhs, q3, s3, None,
                          oracle.MODE_MXFP4, 32)
    assert np.array_equal(a, b)


def test_moe_routing_is_sorted_topk_without_repeats():
    lhs, rhs = synth.moe_routing(tokens=64, experts=8, topk=4, seed=0)
    assert len(lhs) == 256 and np.all(np.diff(rhs) >= 0)
    for t in range(64):
        ex = rhs[lhs == t]
        assert len(ex) == 4 and len(set(ex.tolist())) == 4
