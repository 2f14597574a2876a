"""GPU parity of fp4_quantize_sr (stochastic-rounding fp_quantize, the USE_SR
variant named in "perf(cuda): enable hardware NVFP4/MXFP4 conversion on
Blackwell builds") against the oracle: codes and scales bit for bit, since the
random words are a function of (seed, offset, element index) on both sides."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import u8, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


@pytest.mark.parametrize("mode,use_gs", [(2, True), (2, False), (1, False)])
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 64), (130, 512), (257, 96)])
@pytest.mark.parametrize("seed,offset", [(0, 0), (0x0123456789ABCDEF, 12345), (2 ** 64 - 1, 2 ** 64 - 3)])
def test_quantize_sr_bit_exact(B, mode, use_gs, rows, cols, seed, offset):
    if cols % (16 if mode == 2 else 32):
        pytest.skip("cols not a multiple of the group")
    x = synth.activations_with_outliers(rows, cols, seed=rows + cols, outlier_seed=7)
    xb = synth.to_u16(x)
    gs = oracle.global_scale(xb) if use_gs else None
    gsd = torch.tensor(gs, dtype=torch.float32, device="cuda") if gs is not None else None
    q, s = B.fp4_quantize_sr(x.cuda(), mode, seed, offset, global_scale=gsd)
    oq, os_ = oracle.quantize_sr(xb, mode, gs, seed=seed, offset=offset)
    assert np.array_equal(u32(q), oq)
    assert np.array_equal(u8(s), os_)
    qt, st = B.fp4_quantize_sr(x.cuda(), mode, seed, offset, global_scale=gsd, layout=B.SCALES_TILED)
    assert np.array_equal(u32(qt), oq)
    assert np.array_equal(u8(st), oracle.tile_scales(os_))


@pytest.mark.parametrize("mode", [2, 1])
def test_quantize_sr_activation_workload_full_size(B, mode):
    """The activation-quantize workload (4096 x 5120, 0.1 % outliers x50), every
    code and scale; the block scales are the round-to-nearest quantizer's."""
    x = synth.activations_with_outliers(4096, 5120, seed=0, outlier_seed=1)
    xb = synth.to_u16(x)
    xd = x.cuda()
    gsd = B.fp4_amax_global_scale(xd) if mode == 2 else None
    gs = gsd.item() if gsd is not None else None
    q, s = B.fp4_quantize_sr(xd, mode, 2024, 7, global_scale=gsd, layout=B.SCALES_TILED)
    oq, os_ = oracle.quantize_sr(xb, mode, gs, seed=2024, offset=7)
    assert np.array_equal(u32(q), oq)
    assert np.array_equal(u8(s), oracle.tile_scales(os_))
    _, s_rn = B.fp4_quantize(xd, mode, global_scale=gsd, layout=B.SCALES_TILED)
    assert torch.equal(s, s_rn)
