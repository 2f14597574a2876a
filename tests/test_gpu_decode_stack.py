"""GPU parity of the decode qmv stack exactly as the bench builds it: 64 layers
of a hidden-5120 model (q, k, v, o 5120x5120; gate, up 17408x5120; down
5120x17408), weights drawn on the GPU and quantized by the library, x drawn on
the GPU, in the one-matrix-per-projection layout and in the fused layout
(q|k|v and gate|up stacked as rows).

For layers 0 and 63 every row of every projection is compared with the oracle,
and the library's quantized weights are first compared bit for bit with the
oracle's quantization of the same bf16 weights.  Every other layer is checked
on a seeded sample of rows (the first, the last and 14 random ones per
matrix), the samples judged together by the tolerance rule."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import MAX_ABS_RMS, assert_close_to_oracle, bf16_f64, bf16_u16, u8, u32

pytestmark = pytest.mark.gpu
GROUP = {0: 64, 1: 32, 2: 16}
FULL_LAYERS = (0, synth.LAYERS - 1)


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


def make(B, mode, layer, N, K, grp):
    """The bench's weights for one GEMV of the stack: (q, s, b, gs, bf16 W or None)."""
    if mode == 0:
        q, s, b = synth.affine_synthetic(N, K, synth.layer_seed(layer, grp[0]), device="cuda")
        return q, s, b, None, None
    w = synth.decode_weight(layer, grp, device="cuda")
    gs = B.fp4_amax_global_scale(w) if mode == 2 else None
    q, s = B.fp4_quantize(w, mode, global_scale=gs)
    return q, s, None, gs, w


def host(mode, q, s, b):
    return u32(q), (bf16_u16(s) if mode == 0 else u8(s)), (bf16_u16(b) if b is not None else None)


@pytest.mark.parametrize("mode,layout", [(2, "split"), (1, "split"), (0, "split"), (2, "fused"), (1, "fused")])
def test_decode_stack_every_layer(B, mode, layout):
    xs = {K: synth.decode_x(K, device="cuda") for K in (synth.HIDDEN, synth.MLP)}
    xh = {K: synth.to_u16(v) for K, v in xs.items()}
    rng = np.random.default_rng(1000 + 10 * mode + (layout == "fused"))
    got, want = [], []  # sampled rows of every other layer, judged together by the tolerance rule
    for layer in range(synth.LAYERS):
        full = layer in FULL_LAYERS
        for N, K, grp in synth.layer_groups(layout):
            q, s, b, gs, w = make(B, mode, layer, N, K, grp)
            y = B.qmv(xs[K], q, s, b, gs, mode=mode, group_size=GROUP[mode])
            gsv = gs.item() if gs is not None else None
            what = f"layer {layer} group {grp} mode {mode} {layout}"
            if full:
                qh, sh, bh = host(mode, q, s, b)
                if w is not None:
                    wb = synth.to_u16(w)
                    if mode == 2:
                        g_ref = oracle.global_scale(wb)
                        assert gsv == g_ref, f"{what}: global scale {gsv} != {g_ref}"
                    oq, os_ = oracle.quantize(wb, mode, gsv)
                    assert np.array_equal(qh, oq), f"{what}: codes differ from the oracle"
                    assert np.array_equal(sh, os_), f"{what}: scales differ from the oracle"
                    del wb, oq, os_
                ref = oracle.qmv(xh[K], qh, sh, bh, mode, GROUP[mode], gsv)
                assert_close_to_oracle(y, ref, what)
            else:
                rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 14)]))
                rd = torch.from_numpy(rows).cuda()
                qh, sh, bh = host(mode, q[rd], s[rd], b[rd] if b is not None else None)
                ref = oracle.qmv(xh[K], qh, sh, bh, mode, GROUP[mode], gsv)
                yg = bf16_f64(y[rd])
                rms = np.sqrt(np.mean(ref ** 2))
                assert np.max(np.abs(yg - ref)) <= MAX_ABS_RMS * rms, f"{what}: max-abs"
                got.append(y[rd].cpu())
                want.append(ref)
            del q, s, b, w, y
    # rel-L2 over the union of the samples (a 16-row sample alone is too small for it:
    # one output rounding to the neighbouring bf16 moves its rel-L2 by ~1e-3)
    assert_close_to_oracle(torch.cat(got), np.concatenate(want), f"sampled rows, mode {mode} {layout}")
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
