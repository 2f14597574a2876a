"""fp4_amax_global_scale_noalloc: the global-scale entry point for callers that
cannot allocate device memory (stream capture, pre-planned memory arenas,
allocation-free latency paths).  It keeps its scratch in a fixed device array
inside the library; this test checks, through the C ABI, that two calls in a
row give exactly the results of the regular entry point that takes
caller-provided scratch.  The second call uses a smaller input with a smaller
maximum, so a stale partial maximum left in the shared array by the first
call would show up.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from block_scaled_fp4_fp_gb300 import synth

pytestmark = pytest.mark.gpu


def _regular(B, x):
    gs = torch.empty((), dtype=torch.float32, device="cuda")
    amax = torch.empty((), dtype=torch.float32, device="cuda")
    wsb = B.lib().fp4_amax_workspace_bytes(x.numel())
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    st = B.lib().fp4_amax_global_scale(x.data_ptr(), x.numel(), gs.data_ptr(), amax.data_ptr(), ws.data_ptr(),
                                       wsb, torch.cuda.current_stream().cuda_stream)
    assert st == B.FP4_OK
    return gs, amax


def _noalloc(B, x):
    gs = torch.empty((), dtype=torch.float32, device="cuda")
    amax = torch.empty((), dtype=torch.float32, device="cuda")
    st = B.lib().fp4_amax_global_scale_noalloc(x.data_ptr(), x.numel(), gs.data_ptr(), amax.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
    assert st == B.FP4_OK
    return gs, amax


def test_noalloc_matches_regular_entry_point_on_two_calls():
    from block_scaled_fp4_fp_gb300 import build, binding as B
    build.build()
    B.fp4_init(0)
    big = synth.activations_with_outliers(4096, 5120, seed=3, outlier_seed=4).cuda()
    small = synth.bf16_normal((1, 1000), 0.5, seed=5).cuda()  # much smaller max, fewer blocks
    for x in (big, small):
        g_ref, a_ref = _regular(B, x)
        g, a = _noalloc(B, x)
        torch.cuda.synchronize()
        assert g.item() == g_ref.item()
        assert a.item() == a_ref.item()
    assert B.fp4_check_device_error() == B.FP4_OK


def test_noalloc_rejects_sizes_beyond_its_maximum():
    from block_scaled_fp4_fp_gb300 import binding as B
    p = ctypes.c_void_p(256)
    assert B.lib().fp4_amax_global_scale_noalloc(p, (1 << 36) + 1, p, None, None) == B.FP4_ERR_INVALID_ARG
