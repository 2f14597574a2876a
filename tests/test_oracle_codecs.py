"""Pins for the oracle's scalar codecs (CPU only).

Each check is independent of the oracle's own code path: exact rational
brute force (fractions), torch's float8 dtypes as an outside library, the
format definitions' closed forms, and hand-derived tie cases.
"""
from fractions import Fraction
import math
import struct

import numpy as np
import pytest
import torch

import oracle

E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


def test_e2m1_decode_matches_the_eight_magnitudes():
    for c in range(8):
        assert oracle.e2m1_decode(c) == E2M1_VALUES[c]
        assert oracle.e2m1_decode(c | 8) == -E2M1_VALUES[c] or (c == 0 and oracle.e2m1_decode(8) == 0.0)
    assert math.copysign(1.0, oracle.e2m1_decode(8)) == -1.0
    assert max(oracle.e2m1_decode(c) for c in range(16)) == 6.0  # e2m1 max 6


def _nearest_even_code_fraction(v: Fraction) -> int:
    """Exact brute force: nearest magnitude, ties to the even code index."""
    a = abs(v)
    best, bestd = None, None
    for c, m in enumerate(E2M1_VALUES):
        d = abs(a - Fraction(m))
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    return best


def test_e2m1_encode_dense_sweep_brute_force():
    # every multiple of 2^-7 in [-8, 8] plus +-1 ulp around every midpoint
    pts = set()
    for i in range(-1024, 1025):
        pts.add(f32(i / 128.0))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0]
    for m in mids:
        for s in (1, -1):
            v = np.float32(s * m)
            pts.add(float(v))
            pts.add(float(np.nextafter(v, np.float32(np.inf))))
            pts.add(float(np.nextafter(v, np.float32(-np.inf))))
    for v in sorted(pts):
        got = oracle.e2m1_encode(v)
        want = _nearest_even_code_fraction(Fraction(v))
        if abs(v) > 6:
            want = 7
        want |= 8 if math.copysign(1.0, v) < 0 else 0
        assert got == want, (v, got, want)


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
    (6.0, 7), (7.0, 7), (1e30, 7), (float("inf"), 7), (-float("inf"), 15),
    (-0.0, 8), (-0.1, 8), (0.0, 0), (-5.0, 14), (0.2500001, 1),
])
def test_e2m1_ties_saturation_and_sign(v, code):
    assert oracle.e2m1_encode(v) == code


def test_e4m3_decode_all_bytes_against_torch_float8():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        got = oracle.e4m3_decode(b)
        if math.isnan(ref[b]):
            assert math.isnan(got), b
        else:
            assert got == ref[b], (b, got, ref[b])
    assert oracle.e4m3_decode(0x7E) == 448.0  # E4M3 max 448
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9  # smallest subnormal


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.uniform(0, 448, 20000),
        np.exp2(rng.uniform(-12, 8.8, 20000)),
    ]).astype(np.float32)
    # all decoded values and all midpoints (ties) with their neighbours
    grid = np.array([oracle.e4m3_decode(b) for b in range(0x7F)], np.float64)
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, grid.astype(np.float32), mids,
                           np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0))])
    vals = vals[vals <= 448.0]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(vals.tolist(), ref.tolist()):
        assert oracle.e4m3_encode(v) == r, (v, r)


@pytest.mark.parametrize("v", [448.0, 448.5, 463.9, 464.0, 470.0, 1e9, float("inf")])
def test_e4m3_encode_satfinite(v):
    assert oracle.e4m3_encode(v) == 0x7E


def test_e4m3_roundtrip_every_finite_byte():
    for b in range(256):
        v = oracle.e4m3_decode(b)
        if math.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == b


def test_e8m0_decode_closed_form_and_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for b in range(255):
        assert oracle.e8m0_decode(b) == 2.0 ** (b - 127)
        assert oracle.e8m0_decode(b) == ref[b]
    assert math.isnan(oracle.e8m0_decode(255))


def test_bf16_rounding_matches_torch_for_fp32_inputs():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000),
                        [3.3895313892515355e38, 3.4e38, 1e-40, -1e-42, 0.0, -0.0]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(x)) for x in v], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_is_single_rounding_from_double():
    # 1 + 2^-8 + 2^-40 is just above the bf16 midpoint between 1 and 1+2^-7:
    # a direct rounding goes up; rounding through fp32 first would tie to 1.0.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.bf16_from_double(v) == 0x3F81
    assert oracle.bf16_from_double(1.0 + 2.0 ** -8) == 0x3F80  # exact tie -> even
    assert oracle.bf16_from_double(3.4e38) == 0x7F80  # overflow -> inf
