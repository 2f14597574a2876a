"""GPU parity: amax/global scale, fp_quantize (NVFP4, MXFP4; linear and tiled
scales) and dequantize are bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import bf16_u16, u32, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


def _inputs(kind, rows, cols, seed):
    if kind == "w":
        return synth.bf16_normal((rows, cols), 0.02, seed=seed)
    if kind == "x":
        return synth.bf16_normal((rows, cols), 1.0, seed=seed)
    return synth.activations_with_outliers(rows, cols, seed=seed, outlier_seed=seed + 1)


SHAPES = [("w", 256, 512), ("x", 1, 512), ("o", 130, 96), ("o", 3, 4096), ("w", 257, 160)]


@pytest.mark.parametrize("kind,rows,cols", SHAPES)
def test_global_scale_bit_exact(B, kind, rows, cols):
    x = _inputs(kind, rows, cols, 3)
    gs = B.fp4_amax_global_scale(x.cuda())
    assert gs.item() == oracle.global_scale(synth.to_u16(x))


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 123457])
def test_amax_ragged_lengths(B, n):
    x = synth.activations_with_outliers(1, n, seed=n)
    amax = torch.empty((), dtype=torch.float32, device="cuda")
    gs = torch.empty((), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.lib().fp4_amax_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    B._check(B.lib().fp4_amax_global_scale(x.cuda().data_ptr(), n, gs.data_ptr(), amax.data_ptr(), ws.data_ptr(),
                                           ws.numel(), torch.cuda.current_stream().cuda_stream), "amax")
    assert amax.item() == oracle.amax(synth.to_u16(x))


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("kind,rows,cols", SHAPES)
def test_quantize_bit_exact(B, kind, rows, cols, mode, layout):
    if mode == 1 and cols % 32:
        pytest.skip("MXFP4 needs cols % 32 == 0")
    x = _inputs(kind, rows, cols, 11)
    xb = synth.to_u16(x)
    gs = None
    gsd = None
    if mode == 2:
        gsd = B.fp4_amax_global_scale(x.cuda())
        gs = oracle.global_scale(xb)
    q, s = B.fp4_quantize(x.cuda(), mode, global_scale=gsd, layout=layout)
    oq, os_ = oracle.quantize(xb, mode, gs)
    assert np.array_equal(u32(q), oq)
    if layout == 1:
        assert np.array_equal(u8(s), oracle.tile_scales(os_))
    else:
        assert np.array_equal(u8(s), os_)


@pytest.mark.parametrize("mode", [2, 1])
def test_quantize_full_size_activations(B, mode):
    """The activation-quantize workload: 4096 x 5120 with 0.1 % outliers x50."""
    x = synth.activations_with_outliers(4096, 5120, seed=0, outlier_seed=1)
    xb = synth.to_u16(x)
    gsd = B.fp4_amax_global_scale(x.cuda()) if mode == 2 else None
    gs = oracle.global_scale(xb) if mode == 2 else None
    q, s = B.fp4_quantize(x.cuda(), mode, global_scale=gsd, layout=1)
    oq, os_ = oracle.quantize(xb, mode, gs)
    assert np.array_equal(u32(q), oq)
    assert np.array_equal(u8(s), oracle.tile_scales(os_))


def test_quantize_special_values(B):
    vals = np.zeros((4, 64), np.float32)
    vals[0, :16] = 0.0
    vals[0, 16:32] = -0.0
    vals[1, :32] = np.array([3.3895313892515355e38, -1e38] + [1e-40] * 30, np.float32)  # bf16 max, subnormals
    vals[2, :] = np.linspace(-7, 7, 64)
    vals[3, :] = 2.0 ** -130
    x = torch.from_numpy(vals).to(torch.bfloat16)
    xb = synth.to_u16(x)
    for mode in (2, 1):
        q, s = B.fp4_quantize(x.cuda(), mode)
        oq, os_ = oracle.quantize(xb, mode, None)
        assert np.array_equal(u32(q), oq), mode
        assert np.array_equal(u8(s), os_), mode


def test_e2m1_hardware_rounding_matches_definition(B):
    """MXFP4 groups whose max lies in [4, 8) have scale 2^0, so their codes are
    e2m1_rn_sat(x) of the raw values: every tie and +-1 ulp neighbour of every
    midpoint in [-8, 8] goes through the hardware converter."""
    vals = []
    for m in [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 0.125, 6.0, 0.5, 3.0]:
        for sgn in (1, -1):
            v = torch.tensor(sgn * m, dtype=torch.bfloat16)
            bits = v.view(torch.int16).item()
            for d in (-1, 0, 1):
                vals.append(torch.tensor(bits + d, dtype=torch.int16).view(torch.bfloat16).item())
    vals += [-0.0, 0.0]
    per = 31
    groups = []
    for i in range(0, len(vals), per):
        chunk = vals[i:i + per]
        chunk = chunk + [0.0] * (per - len(chunk))
        groups.append([6.0] + chunk)
    x = torch.tensor(groups, dtype=torch.float32).to(torch.bfloat16).reshape(-1, 32 * 1)
    x = torch.cat([x, torch.zeros((x.shape[0], 32), dtype=torch.bfloat16)], 1)
    xb = synth.to_u16(x)
    q, s = B.fp4_quantize(x.cuda(), 1)
    oq, os_ = oracle.mxfp4_quantize(xb)
    assert (os_[:, 0] == 127).all()
    assert np.array_equal(u32(q), oq)


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("mode", [2, 1, 0])
def test_dequantize_bit_exact(B, mode, layout):
    if mode == 0 and layout == 1:
        pytest.skip("affine scales are linear only")
    rows, cols = 130, 256
    w = synth.bf16_normal((rows, cols), 0.02, seed=5)
    wb = synth.to_u16(w)
    gs, gsd, b, bd = None, None, None, None
    if mode == 0:
        q, s, b = oracle.affine_quantize(wb, 64)
        sd = synth.from_u16(s, "cuda")
        bd = synth.from_u16(b, "cuda")
    else:
        if mode == 2:
            gs = oracle.global_scale(wb)
            gsd = torch.tensor(gs, dtype=torch.float32, device="cuda")
        q, s = oracle.quantize(wb, mode, gs)
        sd = torch.from_numpy(oracle.tile_scales(s) if layout == 1 else s).cuda()
    qd = torch.from_numpy(q.view(np.int32)).cuda()
    out = B.fp4_dequantize(qd, sd, bd, mode=mode, global_scale=gsd, layout=layout, rows=rows)
    ref = oracle.dequantize_bf16(q, s, b, mode, {0: 64, 1: 32, 2: 16}[mode], gs)
    assert np.array_equal(bf16_u16(out), ref)


def test_quantize_nvfp4_block_division_ranges(B):
    """The NVFP4 block scale e4m3(fl(b / fl(6 gs))) on blocks whose maxima and
    global scales reach every range of the division: a tensor so small that the
    divisor is subnormal; blocks of maxima 1, 1e-6, 1e-25 (quotients far below
    e4m3's range), 1e-31 (below 2^-100) and bf16 subnormals under one amax; and
    static global scales log-uniform over 1e-38 .. 1e38 (quotients up to
    saturation).  Codes and scales bit-exact against the oracle."""
    rng = np.random.default_rng(7)
    base = rng.standard_normal((8, 256)).astype(np.float32)
    cases = []
    cases.append((base * 1e-37, None))                      # amax ~ 1e-37: p = fl(6 gs) subnormal
    mixed = base.copy()
    for r, mag in enumerate([1.0, 1e-6, 1e-25, 1e-31, 1e-39, 3.0, 1e-12, 1e-20]):
        mixed[r] *= mag
    cases.append((mixed, None))
    for e in rng.uniform(-38, 38, 40):
        cases.append((base * float(rng.uniform(0.1, 10.0)), float(10.0 ** e)))
    for vals, gs_static in cases:
        x = torch.from_numpy(vals).to(torch.bfloat16)
        xb = synth.to_u16(x)
        if gs_static is None:
            gsd = B.fp4_amax_global_scale(x.cuda())
            gs = oracle.global_scale(xb)
            assert float(gsd.item()) == float(np.float32(gs))
        else:
            gs = float(np.float32(gs_static))
            gsd = torch.tensor(gs, dtype=torch.float32, device="cuda")
        q, s = B.fp4_quantize(x.cuda(), 2, global_scale=gsd)
        oq, os_ = oracle.quantize(xb, 2, gs)
        assert np.array_equal(u32(q), oq), f"codes, gs={gs}"
        assert np.array_equal(u8(s), os_), f"scales, gs={gs}"


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("rows,cols", [(130, 512), (257, 96), (1, 64)])
def test_quantize_tiled_scales_unaligned_buffer(B, mode, rows, cols):
    """Tiled scales into a buffer that starts one byte past an aligned address
    (the NVFP4 kernel then stores bytes instead of words): the same codes and
    scales as into an aligned buffer, and both equal the oracle's."""
    if cols % (16 if mode == 2 else 32):
        pytest.skip("cols not a multiple of the group")
    x = _inputs("o", rows, cols, 21)
    xb = synth.to_u16(x)
    gsd = B.fp4_amax_global_scale(x.cuda()) if mode == 2 else None
    gs = oracle.global_scale(xb) if mode == 2 else None
    q, s = B.fp4_quantize(x.cuda(), mode, global_scale=gsd, layout=1)
    raw = torch.full((s.numel() + 1,), 0xAB, dtype=torch.uint8, device="cuda")
    s_odd = raw[1:].view(s.shape)
    q2, _ = B.fp4_quantize(x.cuda(), mode, global_scale=gsd, layout=1, scales=s_odd)
    oq, os_ = oracle.quantize(xb, mode, gs)
    assert np.array_equal(u32(q), oq) and np.array_equal(u32(q2), oq)
    assert np.array_equal(u8(s), oracle.tile_scales(os_))
    assert np.array_equal(u8(s_odd), oracle.tile_scales(os_))
    assert raw[0].item() == 0xAB  # nothing written before the buffer


@pytest.mark.parametrize("mode,rows,cols", [(2, 300_000, 32), (1, 2_200_000, 32), (2, 300_001, 16)])
def test_quantize_tiled_scales_past_the_grid_height(B, mode, rows, cols):
    """Tiled scales for more 128-row tiles than one grid column of blocks covers
    (NVFP4 past 2047 tiles, MXFP4 past 16383): the kernel strides over tile rows.
    Every code and scale (and the padding) bit-exact against the oracle."""
    x = synth.bf16_normal((rows, cols), 1.0, seed=rows)
    xb = synth.to_u16(x)
    gsd = B.fp4_amax_global_scale(x.cuda()) if mode == 2 else None
    gs = oracle.global_scale(xb) if mode == 2 else None
    q, s = B.fp4_quantize(x.cuda(), mode, global_scale=gsd, layout=1)
    oq, os_ = oracle.quantize(xb, mode, gs)
    assert np.array_equal(u32(q), oq)
    assert np.array_equal(u8(s), oracle.tile_scales(os_))
