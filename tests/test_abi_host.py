"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every entry point declared in include/, and argument validation rejects
bad calls before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from block_scaled_fp4_fp_gb300 import build, binding
    build.build()
    binding.lib()
    return binding


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                                src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(B):
    names = declared_functions()
    assert {"fp4_quantize", "fp4_dequantize", "qmv", "qqmm", "gather_qmm"} <= set(names)
    L = B.lib()
    for n in names:
        assert hasattr(L, n), n
        assert n in B.SIGNATURES, f"binding has no signature for {n}"


def test_status_strings_and_padded_dims(B):
    for s in range(6):
        assert B.status_string(s)
    assert B.padded_scale_dims(1, 32) == (128, 32)
    assert B.padded_scale_dims(300, 5) == (384, 8)
    assert B.padded_scale_dims(4096, 320) == (4096, 320)
    assert B.lib().fp4_amax_workspace_bytes(1 << 20) >= 4


def test_validation_rejects_before_launch(B):
    L = B.lib()
    p = ctypes.c_void_p(256)  # never dereferenced: every call below fails validation first
    # unsupported bits / group / mode
    assert L.qmv(p, p, p, None, None, 64, 64, B.MODE_NVFP4, 3, 16, p, None) == B.FP4_ERR_UNSUPPORTED
    assert L.qmv(p, p, p, None, None, 64, 64, B.MODE_NVFP4, 4, 32, p, None) == B.FP4_ERR_UNSUPPORTED
    assert L.qmv(p, p, p, p, None, 64, 64, B.MODE_AFFINE, 4, 16, p, None) == B.FP4_ERR_UNSUPPORTED
    assert L.fp4_quantize(p, 4, 64, B.MODE_AFFINE, 4, 64, None, p, p, 0, None) == B.FP4_ERR_UNSUPPORTED
    assert L.qqmm(p, p, p, p, None, None, 1, 8, 256, B.MODE_AFFINE, p, None) == B.FP4_ERR_UNSUPPORTED
    # null pointers, bad sizes, indivisible shapes
    assert L.fp4_quantize(None, 4, 64, B.MODE_NVFP4, 4, 16, None, p, p, 0, None) == B.FP4_ERR_INVALID_ARG
    assert L.fp4_quantize(p, 4, 40, B.MODE_NVFP4, 4, 16, None, p, p, 0, None) == B.FP4_ERR_INVALID_ARG
    assert L.fp4_quantize(p, 0, 64, B.MODE_NVFP4, 4, 16, None, p, p, 0, None) == B.FP4_ERR_INVALID_ARG
    assert L.fp4_quantize(p, 4, 64, B.MODE_MXFP4, 4, 32, p, p, p, 0, None) == B.FP4_ERR_INVALID_ARG  # gs w/ MXFP4
    assert L.qqmm(p, p, p, p, None, None, 1, 8, 320, B.MODE_NVFP4, p, None) == B.FP4_ERR_INVALID_ARG  # K % 256
    assert L.qqmm(p, p, p, p, None, None, 1, 12, 256, B.MODE_NVFP4, p, None) == B.FP4_ERR_INVALID_ARG  # N % 8
    assert L.qmv(p, p, p, None, None, 64, 48, B.MODE_NVFP4, 4, 16, p, None) == B.FP4_ERR_INVALID_ARG  # K % 32
    assert L.qmv(p, p, p, None, None, 64, 64, B.MODE_AFFINE, 4, 64, p, None) == B.FP4_ERR_INVALID_ARG  # no biases
    assert L.gather_qmm(p, p, p, 8, p, p, None, 2, 32, 64, B.MODE_MXFP4, 4, 32, 0, p, None) == B.FP4_ERR_UNSUPPORTED
    # alignment
    odd = ctypes.c_void_p(258)
    assert L.qmv(odd, p, p, None, None, 64, 64, B.MODE_NVFP4, 4, 16, p, None) == B.FP4_ERR_ALIGNMENT
    assert L.qqmm(p, odd, p, p, None, None, 1, 8, 256, B.MODE_NVFP4, p, None) == B.FP4_ERR_ALIGNMENT
    assert L.fp4_amax_global_scale(p, 16, p, None, p, 2, None) == B.FP4_ERR_INVALID_ARG  # ws too small
    # empty problems: every size must be at least 1
    assert L.fp4_amax_global_scale(p, 0, p, None, p, 4096, None) == B.FP4_ERR_INVALID_ARG
    assert L.fp4_quantize(p, 4, 0, B.MODE_NVFP4, 4, 16, None, p, p, 0, None) == B.FP4_ERR_INVALID_ARG
    assert L.fp4_dequantize(p, p, None, 0, 64, B.MODE_NVFP4, 4, 16, None, 0, p, None) == B.FP4_ERR_INVALID_ARG
    assert L.qmv(p, p, p, None, None, 0, 64, B.MODE_NVFP4, 4, 16, p, None) == B.FP4_ERR_INVALID_ARG
    assert L.qmv(p, p, p, None, None, 64, 0, B.MODE_NVFP4, 4, 16, p, None) == B.FP4_ERR_INVALID_ARG
    assert L.qqmm(p, p, p, p, None, None, 0, 8, 256, B.MODE_NVFP4, p, None) == B.FP4_ERR_INVALID_ARG
    assert L.gather_qmm(p, p, p, 0, p, p, None, 2, 32, 64, B.MODE_MXFP4, 4, 32, 1, p, None) == B.FP4_ERR_INVALID_ARG
    assert L.gather_qmm(p, p, p, 8, p, p, None, 0, 32, 64, B.MODE_MXFP4, 4, 32, 1, p, None) == B.FP4_ERR_INVALID_ARG
    assert L.qqmv(p, None, p, p, None, 64, 64, B.MODE_AFFINE, p, None) == B.FP4_ERR_UNSUPPORTED
    assert L.qqmv(p, p, p, p, None, 64, 64, B.MODE_MXFP4, p, None) == B.FP4_ERR_INVALID_ARG  # gs_x w/ MXFP4
    assert L.qqmv(p, None, p, p, None, 64, 48, B.MODE_NVFP4, p, None) == B.FP4_ERR_INVALID_ARG  # K % 32
    assert L.qqmv(p, None, p, p, None, 0, 64, B.MODE_NVFP4, p, None) == B.FP4_ERR_INVALID_ARG
    assert L.qqmv(odd, None, p, p, None, 64, 64, B.MODE_NVFP4, p, None) == B.FP4_ERR_ALIGNMENT
    assert L.fp4_quantize_sr(p, 4, 64, B.MODE_AFFINE, 4, 64, None, 1, 0, p, p, 0, None) == B.FP4_ERR_UNSUPPORTED
    assert L.fp4_quantize_sr(p, 4, 40, B.MODE_NVFP4, 4, 16, None, 1, 0, p, p, 0, None) == B.FP4_ERR_INVALID_ARG
    assert L.fp4_quantize_sr(p, 4, 64, B.MODE_MXFP4, 4, 32, p, 1, 0, p, p, 0, None) == B.FP4_ERR_INVALID_ARG
    assert L.fp4_quantize_sr(odd, 4, 64, B.MODE_NVFP4, 4, 16, None, 1, 0, p, p, 0, None) == B.FP4_ERR_ALIGNMENT
    assert L.qmm(p, p, p, None, None, 4, 16, 96, B.MODE_NVFP4, 4, 16, p, None) == B.FP4_ERR_INVALID_ARG  # K % 64
    assert L.qmm(p, p, p, None, None, 4, 24, 64, B.MODE_NVFP4, 4, 16, p, None) == B.FP4_ERR_INVALID_ARG  # N % 16
    assert L.qmm(p, p, p, None, None, 0, 16, 64, B.MODE_NVFP4, 4, 16, p, None) == B.FP4_ERR_INVALID_ARG  # M = 0
    assert L.qmm(p, p, p, None, None, 4, 16, 64, B.MODE_AFFINE, 4, 64, p, None) == B.FP4_ERR_INVALID_ARG  # no biases
    assert L.qmm(p, p, p, None, p, 4, 16, 64, B.MODE_MXFP4, 4, 32, p, None) == B.FP4_ERR_INVALID_ARG  # gs w/ MXFP4
    assert L.qmm(odd, p, p, None, None, 4, 16, 64, B.MODE_NVFP4, 4, 16, p, None) == B.FP4_ERR_ALIGNMENT
    # batched qqmm: overlapping or misaligned batch strides
    assert L.qqmm_batched(p, p, p, p, None, None, 2, 128, 256, 256, 100, 16384, 0, 0, 128 * 256, B.MODE_NVFP4,
                          p, None) == B.FP4_ERR_INVALID_ARG  # stride_xq < M K / 8
    assert L.qqmm_batched(p, p, p, p, None, None, 2, 128, 256, 256, 4096, 1024, 0, 0, 128 * 256, B.MODE_NVFP4,
                          p, None) == B.FP4_ERR_INVALID_ARG  # stride_sx < the 2048 padded scale bytes
    assert L.qqmm_batched(p, p, p, p, None, None, 2, 128, 256, 256, 4098, 16400, 0, 0, 128 * 256, B.MODE_NVFP4,
                          p, None) == B.FP4_ERR_ALIGNMENT  # stride_xq not 16-byte
    assert L.qqmm_batched(p, p, p, p, None, None, 0, 128, 256, 256, 4096, 16384, 0, 0, 128 * 256, B.MODE_NVFP4,
                          p, None) == B.FP4_ERR_INVALID_ARG  # batch 0
    wsb = L.qqmm_quantize_x_workspace_bytes(128, 256, B.MODE_NVFP4)
    assert wsb >= 128 * 128 + 128 * 16
    assert L.qqmm_quantize_x(p, None, p, p, None, 128, 256, 256, B.MODE_NVFP4, p, wsb - 1, None, p,
                             None) == B.FP4_ERR_INVALID_ARG  # workspace too small
    assert L.qqmm_quantize_x(p, p, p, p, None, 128, 256, 256, B.MODE_MXFP4, p, wsb, None, p,
                             None) == B.FP4_ERR_INVALID_ARG  # global scale with MXFP4
    assert L.qqmm_quantize_x(p, None, p, p, None, 128, 256, 320, B.MODE_NVFP4, p, 1 << 20, None, p,
                             None) == B.FP4_ERR_INVALID_ARG  # K % 256
    assert L.qqmm_quantize_x(p, None, p, p, None, 128, 256, 256, B.MODE_NVFP4, ctypes.c_void_p(256 + 64), wsb, None,
                             p, None) == B.FP4_ERR_ALIGNMENT  # workspace not 128-byte aligned
    def grp(count=1, w=256, K=256, N=64):
        g = B.MatrixGroup()
        g.count = count
        for i in range(4):
            g.w[i], g.scales[i], g.N[i] = w, 256, N
        g.K = K
        return g
    Y = (ctypes.c_void_p * 4)(256, 256, 256, 256)
    for g, want in ((grp(count=0), B.FP4_ERR_INVALID_ARG), (grp(count=5), B.FP4_ERR_INVALID_ARG),
                    (grp(K=48), B.FP4_ERR_INVALID_ARG), (grp(N=0), B.FP4_ERR_INVALID_ARG),
                    (grp(w=258), B.FP4_ERR_ALIGNMENT)):
        assert L.qmv_grouped(p, ctypes.byref(g), B.MODE_NVFP4, 4, 16, Y, None, None) == want
    # the prefetch hint is validated as strictly as the group
    assert L.qmv_grouped(p, ctypes.byref(grp()), B.MODE_NVFP4, 4, 16, Y, ctypes.byref(grp(w=258)),
                         None) == B.FP4_ERR_ALIGNMENT
    assert L.qmv_grouped(p, ctypes.byref(grp()), B.MODE_AFFINE, 4, 64, Y, None,
                         None) == B.FP4_ERR_INVALID_ARG  # affine without biases
    assert L.gather_rows(p, 4, p, 8, 12, p, None) == B.FP4_ERR_INVALID_ARG  # K % 8
    assert L.gather_rows(p, 0, p, 8, 16, p, None) == B.FP4_ERR_INVALID_ARG  # no x rows
    assert L.gather_rows(p, 4, p, 0, 16, p, None) == B.FP4_ERR_INVALID_ARG  # R = 0
    assert L.gather_rows(None, 4, p, 8, 16, p, None) == B.FP4_ERR_INVALID_ARG
    assert L.gather_rows(odd, 4, p, 8, 16, p, None) == B.FP4_ERR_ALIGNMENT
    assert L.fp4_debug_stream_weights(p, p, 64, 320, None) == B.FP4_ERR_INVALID_ARG  # K % 256
    assert L.fp4_debug_stream_weights(odd, p, 64, 256, None) == B.FP4_ERR_ALIGNMENT
