"""GPU parity of qmv_grouped: one x against several matrices of the same K in
one launch (q, k and v stored apart; gate and up), each y against the oracle's
fp64 GEMV of its own matrix."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_fp_gb300 import synth
from helpers import assert_close_to_oracle
from test_gpu_qmv import make_weights, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.fp4_init(0)
    return binding


def run_group(B, mode, Ns, K, seed, rows_per=None, x=None):
    mats, host = [], []
    for i, N in enumerate(Ns):
        q, s, b, gs, g = make_weights(mode, N, K, seed=seed + 17 * i)
        host.append((q, s, b, gs, g))
        mats.append(to_dev(mode, q, s, b, gs))
    if x is None:
        x = synth.bf16_normal((K,), 1.0, seed=seed + 5)
    ys = B.qmv_grouped(x.cuda(), mats, mode=mode, group_size=host[0][4])
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    for i, (N, (q, s, b, gs, g), y) in enumerate(zip(Ns, host, ys)):
        rows = None if rows_per is None else rows_per(N, i)
        ref = oracle.qmv(synth.to_u16(x), q, s, b, mode, g, gs, rows=rows)
        yy = y if rows is None else y[torch.from_numpy(rows).cuda()]
        assert_close_to_oracle(yy, ref, f"grouped mode {mode} matrix {i} of {Ns}x{K}")


@pytest.mark.parametrize("mode", [2, 1, 0])
@pytest.mark.parametrize("Ns,K", [([256], 512), ([300, 7, 129], 1024), ([1, 1, 1, 1], 512),
                                  ([1000, 2000], 2048), ([33, 4000, 33], 4096)])
def test_qmv_grouped_small(B, mode, Ns, K):
    """Every matrix's rows are dealt whole row blocks (ragged matrices, one-row
    matrices, up to four matrices); affine runs as separate launches."""
    run_group(B, mode, Ns, K, seed=sum(Ns) + K)


@pytest.mark.parametrize("mode", [2, 1, 0])
@pytest.mark.parametrize("Ns", [[synth.HIDDEN] * 3, [17408, 17408]])
def test_qmv_grouped_decode_shapes_sampled(B, mode, Ns):
    """q, k, v (3 x 5120 x 5120) and gate, up (2 x 17408 x 5120) stored apart, in
    the launch configuration the bench uses (FP4 on the tensor-core GEMV, affine
    g64 on the affine GEMV, one launch each); the oracle checks a seeded sample
    of rows of every matrix, including the first and last rows."""
    K = synth.HIDDEN

    def rows_per(N, i):
        return np.unique(np.concatenate([np.arange(8), N - 1 - np.arange(8),
                                         np.random.default_rng(N + i).integers(0, N, 120)]))

    run_group(B, mode, Ns, K, seed=Ns[0] + mode, rows_per=rows_per)


@pytest.mark.parametrize("mode", [2, 1])
def test_qmv_grouped_split_k(B, mode):
    """A K long enough that the stacked rows take the K-split plan (clusters)."""
    run_group(B, mode, [300, 700], 34816, seed=77)


@pytest.mark.parametrize("mode", [2, 1, 0])
def test_qmv_grouped_prefetch_hint_changes_nothing(B, mode):
    """A chain of launches each naming the next one's weights (the L2 warm-up
    hint, wrapping around): every y is bit-identical to the same launches without
    hints, and matches the oracle."""
    K = 1024
    shapes = [[300, 700], [64], [1000, 1000, 5], [2048]]
    groups, host = [], []
    for j, Ns in enumerate(shapes):
        mats, hm = [], []
        for i, N in enumerate(Ns):
            q, s, b, gs, g = make_weights(mode, N, K, seed=100 * j + i)
            hm.append((q, s, b, gs, g))
            mats.append(to_dev(mode, q, s, b, gs))
        groups.append(mats)
        host.append(hm)
    x = synth.bf16_normal((K,), 1.0, seed=3).cuda()
    plain = [B.qmv_grouped(x, m, mode=mode) for m in groups]
    hinted = [B.qmv_grouped(x, m, mode=mode, prefetch_next=groups[(j + 1) % len(groups)])
              for j, m in enumerate(groups)]
    torch.cuda.synchronize()
    assert B.fp4_check_device_error() == B.FP4_OK
    for j in range(len(groups)):
        for i, (q, s, b, gs, g) in enumerate(host[j]):
            assert torch.equal(plain[j][i], hinted[j][i])
            ref = oracle.qmv(synth.to_u16(x.cpu()), q, s, b, mode, g, gs)
            assert_close_to_oracle(hinted[j][i], ref, f"hinted launch {j} matrix {i}")
