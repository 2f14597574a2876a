"""GPU parity of the decode step exactly as bench.py times it: `bench.DecodeStack`
(64 layers of the hidden-5120 stack in the fused layout, every launch through
qmv_grouped naming the next launch's weights) captured in a CUDA graph by the
bench's own `capture` and replayed.  Every output row of layers 0 and 63, and a
seeded sample of rows of every other layer, is compared with the oracle's fp64
GEMV of the library's own quantized weights."""
import numpy as np
import pytest
import torch

import bench
import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import MAX_ABS_RMS, assert_close_to_oracle, bf16_f64, bf16_u16, u8, u32

pytestmark = pytest.mark.gpu
GROUP = {0: 64, 1: 32, 2: 16}


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


@pytest.mark.parametrize("mode", [2, 1, 0])
def test_bench_decode_step_matches_oracle(B, mode):
    dev = torch.device("cuda", 0)
    stack = bench.DecodeStack(B, mode, synth.LAYERS, dev, layout="fused", prefetch=True)
    stream = torch.cuda.Stream()
    graph = bench.capture(stack.step, stream)
    for y in stack.y:
        y.fill_(float("nan"))  # the replays below must write every output
    with torch.cuda.stream(stream):
        graph.replay()
        graph.replay()
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    xh = {K: synth.to_u16(v.cpu()) for K, v in stack.x.items()}
    per_layer = len(stack.mats) // synth.LAYERS
    rng = np.random.default_rng(77 + mode)
    got, want = [], []
    for i, (m, y) in enumerate(zip(stack.mats, stack.y)):
        layer = i // per_layer
        N, K = m["N"], m["K"]
        what = f"bench step, mode {mode}, layer {layer}, matrix {i % per_layer} ({N}x{K})"
        rows = (np.arange(N) if layer in (0, synth.LAYERS - 1)
                else np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 14)])))
        rd = torch.from_numpy(rows).cuda()
        qh = u32(m["q"][rd])
        sh = bf16_u16(m["s"][rd]) if mode == 0 else u8(m["s"][rd])
        bh = bf16_u16(m["b"][rd]) if m["b"] is not None else None
        gs = m["gs"].item() if m["gs"] is not None else None
        ref = oracle.qmv(xh[K], qh, sh, bh, mode, GROUP[mode], gs)
        if len(rows) == N:
            assert_close_to_oracle(y, ref, what)
        else:
            yg = bf16_f64(y[rd])
            rms = np.sqrt(np.mean(ref ** 2))
            assert np.all(np.isfinite(yg)), f"{what}: non-finite output"
            assert np.max(np.abs(yg - ref)) <= MAX_ABS_RMS * rms, f"{what}: max-abs"
            got.append(y[rd].cpu())
            want.append(ref)
    # rel-L2 over the union of the samples, as the per-layer samples are too small alone
    assert_close_to_oracle(torch.cat(got), np.concatenate(want), f"bench step sampled rows, mode {mode}")
