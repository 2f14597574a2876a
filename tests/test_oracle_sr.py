"""Pins of the oracle's stochastic-rounding quantizer: its random numbers
against an independent implementation of Philox4x32-10 (cuRAND's host
generator), and the rounding rule against the properties that define it
(two-neighbour support, exactness on the grid, the extreme random words,
unbiasedness, saturation and sign)."""
import ctypes
import json
import os

import numpy as np
import pytest

import oracle
from block_scaled_fp4_fp_gb300 import synth

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _curand():
    for p in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            return ctypes.CDLL(p)
        except OSError:
            continue
    return None


def test_philox_known_answer_vectors():
    """The published known-answer vectors of Philox4x32-10 (tests/golden)."""
    kat = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")))
    for v in kat["vectors"]:
        ctr = [int(h, 16) for h in v["counter"]]
        key = [int(h, 16) for h in v["key"]]
        assert oracle.philox4x32_10(ctr, key) == [int(h, 16) for h in v["out"]]


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 2 ** 64 - 1])
def test_philox_matches_curand_host_generator(seed):
    """cuRAND's host Philox4x32-10 generator (an independent implementation)
    with the same 64-bit seed as key emits, in its default ordering, output
    block j = Philox(counter = (j / 65536, 0, j % 65536, 0)): compare blocks
    across both counter words it exercises."""
    L = _curand()
    if L is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    assert L.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # CURAND_RNG_PSEUDO_PHILOX4_32_10
    try:
        assert L.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        n = 4 * (2 * 65536 + 64)
        out = np.zeros(n, np.uint32)
        assert L.curandGenerate(gen, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), n) == 0
    finally:
        L.curandDestroyGenerator(gen)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for j in list(range(64)) + list(range(65536, 65536 + 64)) + [65535, 2 * 65536 + 5]:
        assert oracle.philox4x32_10([j // 65536, 0, j % 65536, 0], key) == out[4 * j:4 * j + 4].tolist(), j


def test_philox_counter_carry_and_key_words():
    """The counter is offset + e / 4 over 128 bits (a carry out of the low 64
    bits lands in word 2) and the seed's two halves are the key words."""
    e, off = 8, 2 ** 64 - 1  # block offset + 2 wraps to 1 with a carry
    assert oracle.sr_word(5, off, e) == oracle.philox4x32_10([1, 0, 1, 0], [5, 0])[0]
    s = (0xAABBCCDD << 32) | 0x11223344
    assert oracle.sr_word(s, 3, 6) == oracle.philox4x32_10([4, 0, 0, 0], [0x11223344, 0xAABBCCDD])[2]


def test_sr_support_is_the_two_neighbours_and_grid_values_are_exact():
    rng = np.random.default_rng(0)
    for v in np.concatenate([rng.uniform(-6.5, 6.5, 400), [0.0, -0.0, 0.5, 1.5, 3.0, 6.0, -4.0]]):
        v = float(np.float32(v))
        a = abs(v)
        lo = max(x for x in E2M1 if x <= a) if a < 6 else 6.0
        hi = min(x for x in E2M1 if x >= a) if a < 6 else 6.0
        for u in (0, 1 << 8, rng.integers(0, 2 ** 32), 2 ** 32 - 1):
            c = oracle.e2m1_encode_sr(v, int(u))
            mag = E2M1[c & 7]
            assert mag in (lo, hi), (v, u, c)
            assert (c >> 3) == (1 if np.signbit(v) else 0)
            if a in E2M1:
                assert mag == a


def test_sr_extreme_random_words():
    """u = 0 rounds every off-grid value up (the threshold is at least 1), the
    largest word rounds every value down (u >> 8 = 2^24 - 1 is never below it)."""
    for v in (0.01, 0.3, 0.74, 1.2, 2.9, 3.01, 5.99, -2.5):
        a = abs(v)
        lo = max(x for x in E2M1 if x <= a)
        hi = min(x for x in E2M1 if x > a)
        assert E2M1[oracle.e2m1_encode_sr(v, 0) & 7] == hi
        assert E2M1[oracle.e2m1_encode_sr(v, 2 ** 32 - 1) & 7] == lo


def test_sr_is_unbiased():
    """E[SR(v)] = v: the probability of rounding up is the fraction of the step
    (to 2^-24), so the mean over many uniform words matches v within 4 sigma."""
    rng = np.random.default_rng(1)
    n = 20000
    us = rng.integers(0, 2 ** 32, n, dtype=np.uint64)
    for v in (0.3, 1.1, 2.25, 3.7, 4.9, -0.05):
        vals = np.array([np.sign(v) * E2M1[oracle.e2m1_encode_sr(v, int(u)) & 7] for u in us])
        a = abs(v)
        lo = max(x for x in E2M1 if x <= a)
        hi = min(x for x in E2M1 if x > a)
        sigma = (hi - lo) * 0.5 / np.sqrt(n)
        assert abs(vals.mean() - v) < 4 * sigma, (v, vals.mean())


def test_sr_saturates_and_keeps_sign():
    for v, code in ((6.0, 7), (7.5, 7), (1e30, 7), (float("inf"), 7), (-9.0, 15), (-0.0, 8), (0.0, 0)):
        for u in (0, 12345, 2 ** 32 - 1):
            assert oracle.e2m1_encode_sr(v, u) == code, (v, u)


@pytest.mark.parametrize("mode,use_gs", [(2, True), (2, False), (1, False)])
def test_sr_quantize_scales_match_rn_and_mean_is_x(mode, use_gs):
    """Block scales are the round-to-nearest ones; averaged over 64 seeds the
    dequantized values approach x (each element's expectation is x exactly,
    up to the rounding of the reciprocal scale and saturation at 6)."""
    x = synth.to_u16(synth.bf16_normal((8, 256), 1.0, seed=4))
    gs = oracle.global_scale(x) if use_gs else None
    q0, s0 = oracle.quantize(x, mode, gs)
    g = 16 if mode == 2 else 32
    acc = np.zeros((8, 256))
    seeds = 64
    for sd in range(seeds):
        q, s = oracle.quantize_sr(x, mode, gs, seed=sd, offset=3)
        assert np.array_equal(s, s0)
        acc += oracle.dequantize_f64(q, s, None, mode, g, gs)
    mean = acc / seeds
    xf = oracle.bf16_bits_to_f64(x)
    # the step of the e2m1 grid at each element (2 x its largest round-to-nearest error
    # over the block), and the elements MXFP4 saturates (|x| 2^-se above 6)
    bs = oracle.dequantize_f64(np.full_like(q0, 0x77777777), s0, None, mode, g, gs) / 6.0
    unsat = np.abs(xf) <= 6.0 * bs
    step = 2.0 * bs  # the widest e2m1 step is 2 in units of the block scale
    # per element the mean of 64 draws is within 4 sigma (sigma <= step / 2 / 8) of x
    assert np.all((np.abs(mean - xf) <= 4 * step / 16 + 1e-6) | ~unsat)
    assert unsat.mean() > 0.9
    # and it differs from round-to-nearest on some elements, which plain rounding would not
    assert not np.array_equal(oracle.quantize_sr(x, mode, gs, seed=0)[0], q0)
