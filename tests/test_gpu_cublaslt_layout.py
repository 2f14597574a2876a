"""The oracle's packed-code order and 128x4 scale-tile layout read by an
independent implementation: cuBLASLt's block-scaled FP4 GEMM (through
torch._scaled_mm on float4_e2m1fn_x2 operands with E4M3 block scales).

The pages fix the tile's size, padding and zero fill ("mlx 0.30.7.3 ->
0.30.7.6", qqmm_utils.h) and point to cuBLAS's block-scaling-factor layout
without restating the byte order inside a tile; the oracle's reading of that
order, and its low-nibble-first packing, are otherwise pinned only by
identities of the oracle itself.  Here the oracle quantizes x and W (NVFP4),
tiles the scales, and cuBLASLt multiplies those very bytes; its bf16 output is
compared with the oracle's product (alpha = 1, the same single rounding).  A
different tile order or nibble order would scramble the scales or codes and
fail by orders of magnitude.  cuBLASLt is not part of the library: this test
checks the oracle against the vendor's reading of the format."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import assert_close_to_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (300, 384, 1024), (128, 512, 256)])
def test_oracle_layout_read_by_cublaslt(M, N, K):
    f4 = getattr(torch, "float4_e2m1fn_x2", None)
    if f4 is None:
        pytest.skip("this PyTorch has no float4_e2m1fn_x2")
    x = synth.to_u16(synth.bf16_normal((M, K), 1.0, seed=M + 7))
    w = synth.to_u16(synth.bf16_normal((N, K), 0.02, seed=N + 8))
    gx, gw = oracle.global_scale(x), oracle.global_scale(w)
    xq, xs = oracle.quantize(x, 2, gx)
    wq, ws = oracle.quantize(w, 2, gw)
    xt, wt = oracle.tile_scales(xs), oracle.tile_scales(ws)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    a = dev(xq.view(np.uint8)).view(f4)                     # [M, K/2]
    b = dev(wq.view(np.uint8)).view(f4).t()                 # [K/2, N], column-major
    sa = dev(xt.reshape(-1)).view(torch.float8_e4m3fn)
    sb = dev(wt.reshape(-1)).view(torch.float8_e4m3fn)
    try:
        out = torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
    except RuntimeError as e:  # a PyTorch or cuBLASLt build without this GEMM
        pytest.skip(f"cuBLASLt block-scaled FP4 GEMM unavailable: {str(e).splitlines()[0][:120]}")
    ref = oracle.qqmm(xq, xs, wq, ws, 2, alpha=1.0)
    assert_close_to_oracle(out, ref, f"cuBLASLt on the oracle's bytes {M}x{N}x{K}")
