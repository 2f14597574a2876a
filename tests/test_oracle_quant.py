"""Pins for the oracle's quantizers, scale tiling and dequantizers (CPU only)."""
from fractions import Fraction
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def bf16_bits(vals):
    return synth.to_u16(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def unpack(q, cols):
    q = np.asarray(q, np.uint32)
    out = np.zeros(q.shape[:-1] + (cols,), np.uint8)
    for j in range(8):
        out[..., j::8] = (q >> np.uint32(4 * j)) & np.uint32(15)
    return out


def code_values(codes):
    c = np.asarray(codes, np.int64)
    v = E2M1[c & 7]
    return np.where(c & 8, -v, v)


# ---- hand-derived worked examples ----------------------------------------

@pytest.mark.parametrize("ex", GOLDEN["nvfp4"])
def test_nvfp4_worked_examples(ex):
    x = bf16_bits([ex["x"]])
    q, s = oracle.nvfp4_quantize(x, ex["gs"])
    assert s[0, 0] == ex["scale"]
    assert unpack(q, 16)[0].tolist() == ex["codes"]
    if "words" in ex:
        assert q[0].tolist() == ex["words"]


@pytest.mark.parametrize("ex", GOLDEN["mxfp4"])
def test_mxfp4_worked_examples(ex):
    vals = ex["x_head"] + [0.0] * (32 - len(ex["x_head"]))
    q, s = oracle.mxfp4_quantize(bf16_bits([vals]))
    assert s[0, 0] == ex["scale"]
    assert unpack(q, 32)[0, :len(ex["codes_head"])].tolist() == ex["codes_head"]


def test_padded_dims_and_alpha_golden():
    for ex in GOLDEN["padded_dims"]:
        assert list(oracle.padded_dims(ex["rows"], ex["cols"])) == ex["padded"]
    for ex in GOLDEN["alpha"]:
        a = oracle.alpha_from_amax(ex["amax_x"], ex["amax_w"])
        assert a == pytest.approx(ex["alpha"], rel=2 ** -22)


def test_alpha_equals_product_of_multiplier_global_scales():
    rng = np.random.default_rng(3)
    for _ in range(200):
        ax, aw = np.float32(rng.uniform(0.1, 100)), np.float32(rng.uniform(0.01, 10))
        gx, gw = np.float32(ax / np.float32(2688)), np.float32(aw / np.float32(2688))
        a = oracle.alpha_from_amax(float(ax), float(aw))
        assert a == pytest.approx(float(gx) * float(gw), rel=4 * 2 ** -23)
        assert a == pytest.approx(float(ax) * float(aw) / (448 * 6) ** 2, rel=2 * 2 ** -23)


# ---- NVFP4 invariants ------------------------------------------------------

def _e4m3_via_torch(v):
    t = torch.tensor(np.minimum(np.asarray(v, np.float32), np.float32(448)))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("with_gs", [False, True])
def test_nvfp4_scale_and_codes_are_nearest(with_gs):
    x = synth.activations_with_outliers(64, 256, seed=5)
    xb = synth.to_u16(x)
    xf = x.float().numpy()
    gs = oracle.global_scale(xb) if with_gs else None
    q, s = oracle.nvfp4_quantize(xb, gs)
    g = np.float32(gs if gs is not None else 1.0)
    blocks = xf.reshape(64, 16, 16)
    b = np.abs(blocks).max(-1).astype(np.float32)
    p = np.float32(np.float32(6) * g)
    want_s = _e4m3_via_torch(np.where(b == 0, np.float32(0), (b / p).astype(np.float32)))
    assert np.array_equal(s, want_s)
    # each code is the nearest e2m1 point (ties to even code) to fl(x * fl(1/fl(s8*gs)))
    s8 = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).float().numpy()
    d = (s8 * g).astype(np.float32)
    r = np.where(d == 0, np.float32(0), (np.float32(1) / d).astype(np.float32)).astype(np.float32)
    scaled = (blocks * r[..., None]).astype(np.float32)
    codes = unpack(q, 256).reshape(64, 16, 16)
    for v, c in zip(scaled.ravel()[:4000].tolist(), codes.ravel()[:4000].tolist()):
        a = min(abs(Fraction(v)), Fraction(6))
        dist = [abs(a - Fraction(m)) for m in E2M1]
        best = min(dist)
        assert dist[c & 7] == best
        if dist.count(best) > 1:
            assert (c & 7) % 2 == 0
        assert bool(c & 8) == (math.copysign(1, v) < 0)


def test_nvfp4_requantize_of_exact_block_is_identity():
    # blocks made of e2m1 values times an E4M3-exact scale with a +-6 present
    rng = np.random.default_rng(7)
    rows = 256
    codes = rng.integers(0, 16, size=(rows, 16))
    codes[:, 0] = np.where(rng.random(rows) < 0.5, 7, 15)
    scale_bytes = rng.integers(0x08, 0x70, size=rows)  # normal E4M3, products exact in bf16
    sval = torch.from_numpy(scale_bytes.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    vals = code_values(codes) * sval[:, None]
    xb = bf16_bits(vals.tolist())
    assert np.array_equal(synth.from_u16(xb).double().numpy(), vals)  # exact in bf16
    q, s = oracle.nvfp4_quantize(xb, None)
    assert np.array_equal(s[:, 0], scale_bytes.astype(np.uint8))
    got = unpack(q, 16)
    # +-0 codes may differ only in the sign of zero
    same = (got == codes) | (((got & 7) == 0) & ((codes & 7) == 0))
    assert same.all()


def test_nvfp4_global_scale_maps_tensor_amax_to_top_scale():
    x = synth.bf16_normal((32, 64), 0.02, seed=11)
    xb = synth.to_u16(x)
    gs = oracle.global_scale(xb)
    amax = float(np.abs(x.float().numpy()).max())
    assert gs == pytest.approx(amax / 2688, rel=2 ** -23)
    q, s = oracle.nvfp4_quantize(xb, gs)
    s8 = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert s8.max() == 448.0  # the block holding amax gets the largest E4M3 scale
    deq = oracle.dequantize_f64(q, s, None, oracle.MODE_NVFP4, 16, gs)
    assert np.abs(deq).max() == pytest.approx(amax, rel=0.07)


# ---- MXFP4 invariants ------------------------------------------------------

def test_mxfp4_scale_is_floor_log2_minus_2():
    x = synth.activations_with_outliers(32, 512, seed=2)
    xb = synth.to_u16(x)
    q, s = oracle.mxfp4_quantize(xb)
    b = np.abs(x.float().numpy()).reshape(32, 16, 32).max(-1)
    want = np.clip(np.floor(np.log2(b)).astype(np.int64) - 2, -127, 127) + 127
    assert np.array_equal(s.astype(np.int64), want)
    # scaled block maxima lie in [4, 8): top code is 6 (4.0) or 7 (6.0)
    deq = oracle.dequantize_f64(q, s, None, oracle.MODE_MXFP4, 32)
    err = np.abs(deq - x.double().numpy()).reshape(32, 16, 32)
    scale = np.exp2(s.astype(np.float64) - 127)
    # in-range elements are within half a grid step (<= 1 * 2^se), saturated ones
    # within (8 - 6) * 2^se
    assert (err <= 2.0 * scale[..., None]).all()


def test_mxfp4_zero_and_subnormal_groups():
    vals = np.zeros((2, 32))
    vals[1, 0] = 2.0 ** -130  # bf16 subnormal
    xb = bf16_bits(vals.tolist())
    q, s = oracle.mxfp4_quantize(xb)
    assert s[0, 0] == 0 and (q[0] == 0).all()
    # floor(log2 2^-130) - 2 = -132 clamps to -127 -> byte 0; 2^-130 * 2^127 = 1/8 -> 0
    assert s[1, 0] == 0


# ---- affine generator ------------------------------------------------------

def test_affine_quantize_error_within_half_step():
    w = synth.bf16_normal((16, 256), 0.02, seed=3)
    wb = synth.to_u16(w)
    q, s, b = oracle.affine_quantize(wb, 64)
    codes = unpack(q, 256)
    assert codes.max() <= 15
    deq = oracle.dequantize_f64(q, s, b, oracle.MODE_AFFINE, 64)
    sv = oracle.bf16_bits_to_f64(s)
    err = np.abs(deq - w.double().numpy()).reshape(16, 4, 64)
    assert (err <= sv[..., None] * 0.5 + 1e-3 * sv[..., None] + 1e-7).all()
    # the minimum of each group maps to code 0
    assert (codes.reshape(16, 4, 64).min(-1) == 0).all()


# ---- tiled scale layout -----------------------------------------------------

def test_tiled_offset_known_positions():
    cp = 8
    assert oracle.tiled_offset(0, 0, cp) == 0
    assert oracle.tiled_offset(1, 0, cp) == 16
    assert oracle.tiled_offset(32, 0, cp) == 4
    assert oracle.tiled_offset(0, 3, cp) == 3
    assert oracle.tiled_offset(0, 4, cp) == 512       # next column tile
    assert oracle.tiled_offset(128, 0, cp) == 1024    # next row tile (cp/4 = 2 tiles per row tile)
    assert oracle.tiled_offset(127, 7, cp) == 512 + 31 * 16 + 3 * 4 + 3


def test_tile_untile_bijection_and_zero_padding():
    rng = np.random.default_rng(0)
    for rows, cols in [(1, 32), (130, 5), (256, 320), (300, 9)]:
        lin = rng.integers(1, 256, size=(rows, cols), dtype=np.uint8)
        t = oracle.tile_scales(lin)
        rp, cp = oracle.padded_dims(rows, cols)
        assert t.shape == (rp, cp)
        assert np.array_equal(oracle.untile_scales(t, rows, cols), lin)
        # exactly rows*cols non-zero bytes: everything else is zero padding
        assert np.count_nonzero(t) == rows * cols
        offs = {oracle.tiled_offset(r, c, cp) for r in range(rows) for c in range(cols)}
        assert len(offs) == rows * cols and max(offs) < rp * cp


# ---- dequantize -------------------------------------------------------------

@pytest.mark.parametrize("mode", [oracle.MODE_NVFP4, oracle.MODE_MXFP4, oracle.MODE_AFFINE])
def test_dequantize_bf16_within_half_ulp_of_exact(mode):
    w = synth.bf16_normal((8, 256), 0.02, seed=4)
    wb = synth.to_u16(w)
    gs = None
    if mode == oracle.MODE_NVFP4:
        gs = oracle.global_scale(wb)
        q, s = oracle.nvfp4_quantize(wb, gs)
        b, g = None, 16
    elif mode == oracle.MODE_MXFP4:
        q, s = oracle.mxfp4_quantize(wb)
        b, g = None, 32
    else:
        q, s, b = oracle.affine_quantize(wb, 64)
        g = 64
    exact = oracle.dequantize_f64(q, s, b, mode, g, gs)
    got = oracle.bf16_bits_to_f64(oracle.dequantize_bf16(q, s, b, mode, g, gs))
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert (np.abs(got - exact) <= 0.5 * ulp * (1 + 2 ** -15)).all()


def test_dequantize_mxfp4_closed_form():
    codes = np.arange(16)
    q = np.zeros((1, 4), np.uint32)
    for k in range(32):
        q[0, k // 8] |= np.uint32(codes[k % 16]) << np.uint32(4 * (k % 8))
    s = np.array([[120]], np.uint8)
    out = oracle.dequantize_f64(q, s, None, oracle.MODE_MXFP4, 32)
    assert np.array_equal(out[0, :16], code_values(codes) * 2.0 ** -7)
