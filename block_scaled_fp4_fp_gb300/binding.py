"""Thin Python binding of libfp4gb300 (ctypes).

Functions carry the C ABI's names and only marshal arguments: shapes and
device pointers of torch tensors, the current CUDA stream, and output
allocation with torch (PyTorch is the memory allocator here, nothing more).
Every step of the computation runs in the library's CUDA kernels; there is no
CPU fallback -- if the shared library is missing the first call raises.

Packed 4-bit codes are held in ``torch.int32`` tensors (uint32 bit patterns),
scales in ``torch.uint8`` (NVFP4/MXFP4) or ``torch.bfloat16`` (affine).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp4gb300.so")

FP4_OK, FP4_ERR_INVALID_ARG, FP4_ERR_UNSUPPORTED, FP4_ERR_ALIGNMENT, FP4_ERR_CUDA, FP4_ERR_TIMEOUT = range(6)
MODE_AFFINE, MODE_MXFP4, MODE_NVFP4 = 0, 1, 2
SCALES_LINEAR, SCALES_TILED = 0, 1
GROUP = {MODE_NVFP4: 16, MODE_MXFP4: 32, MODE_AFFINE: 64}

_lock = threading.Lock()
_lib = None

# (name, restype, argtypes) of every entry point the header declares
c = ctypes
_VP, _I64, _INT, _F = c.c_void_p, c.c_int64, c.c_int, c.c_float
SIGNATURES = {
    "fp4_init": (_INT, [_INT]),
    "fp4_status_string": (c.c_char_p, [_INT]),
    "fp4_check_device_error": (_INT, [_VP]),
    "fp4_padded_scale_dims": (None, [_I64, _I64, c.POINTER(_I64), c.POINTER(_I64)]),
    "fp4_amax_workspace_bytes": (c.c_size_t, [_I64]),
    "fp4_amax_global_scale": (_INT, [_VP, _I64, _VP, _VP, _VP, c.c_size_t, _VP]),
    "fp4_quantize": (_INT, [_VP, _I64, _I64, _INT, _INT, _INT, _VP, _VP, _VP, _INT, _VP]),
    "fp4_quantize_sr": (_INT, [_VP, _I64, _I64, _INT, _INT, _INT, _VP, c.c_uint64, c.c_uint64, _VP, _VP, _INT,
                               _VP]),
    "fp4_dequantize": (_INT, [_VP, _VP, _VP, _I64, _I64, _INT, _INT, _INT, _VP, _INT, _VP, _VP]),
    "qmv": (_INT, [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _INT, _INT, _INT, _VP, _VP]),
    "qqmv": (_INT, [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _INT, _VP, _VP]),
    "qqmm": (_INT, [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _INT, _VP, _VP]),
    "gather_rows": (_INT, [_VP, _I64, _VP, _I64, _I64, _VP, _VP]),
    "qmv_grouped": (_INT, [_VP, _VP, _INT, _INT, _INT, _VP, _VP, _VP]),
    "gather_qmm": (_INT, [_VP, _VP, _VP, _I64, _VP, _VP, _VP, _I64, _I64, _I64, _INT, _INT, _INT, _INT,
                          _VP, _VP]),
    "qqmm_batched": (_INT, [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                            _INT, _VP, _VP]),
    "qqmm_quantize_x_workspace_bytes": (c.c_size_t, [_I64, _I64, _INT]),
    "qqmm_quantize_x": (_INT, [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _INT, _VP, c.c_size_t, _VP, _VP, _VP]),
    "qmm": (_INT, [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _INT, _INT, _INT, _VP, _VP]),
    "fp4_debug_inject_wait_timeout": (_INT, [_INT]),
    "fp4_debug_stream_weights": (_INT, [_VP, _VP, _I64, _I64, _VP]),
    "fp4_amax_global_scale_noalloc": (_INT, [_VP, _I64, _VP, _VP, _VP]),
}


class Fp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib():
    """Load libfp4gb300.so (built in-tree by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fp4_status_string(int(status)).decode()


def _check(st: int, where: str):
    if st != FP4_OK:
        raise Fp4Error(st, where)


def _p(t):
    return None if t is None else t.data_ptr()


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def padded_scale_dims(rows: int, scale_cols: int):
    pr, pc = c.c_int64(), c.c_int64()
    lib().fp4_padded_scale_dims(rows, scale_cols, c.byref(pr), c.byref(pc))
    return pr.value, pc.value


def fp4_init(device: int = 0):
    _check(lib().fp4_init(device), "fp4_init")


def fp4_check_device_error(stream=None) -> int:
    """Returns the status (FP4_OK or FP4_ERR_TIMEOUT...) without raising."""
    return lib().fp4_check_device_error(_s(stream))


def fp4_amax_global_scale(x: torch.Tensor, gs_out=None, amax_out=None, ws=None, stream=None):
    n = x.numel()
    if gs_out is None:
        gs_out = torch.empty((), dtype=torch.float32, device=x.device)
    wsb = lib().fp4_amax_workspace_bytes(n)
    if ws is None:
        ws = torch.empty(wsb, dtype=torch.uint8, device=x.device)
    _check(lib().fp4_amax_global_scale(_p(x), n, _p(gs_out), _p(amax_out), _p(ws), ws.numel() * ws.element_size(),
                                       _s(stream)), "fp4_amax_global_scale")
    return gs_out


def fp4_amax_global_scale_noalloc(x: torch.Tensor, gs_out=None, amax_out=None, stream=None):
    """Allocation-free global scale: the library uses its own fixed device scratch."""
    if gs_out is None:
        gs_out = torch.empty((), dtype=torch.float32, device=x.device)
    _check(lib().fp4_amax_global_scale_noalloc(_p(x), x.numel(), _p(gs_out), _p(amax_out), _s(stream)),
           "fp4_amax_global_scale_noalloc")
    return gs_out


def scales_shape(rows: int, cols: int, group: int, layout: int):
    if layout == SCALES_TILED:
        return padded_scale_dims(rows, cols // group)
    return rows, cols // group


def fp4_quantize(x: torch.Tensor, mode: int, group_size: int = None, global_scale=None,
                 layout: int = SCALES_LINEAR, xq=None, scales=None, stream=None):
    group_size = group_size or GROUP[mode]
    rows, cols = x.shape
    if xq is None:
        xq = torch.empty((rows, cols // 8), dtype=torch.int32, device=x.device)
    if scales is None:
        scales = torch.empty(scales_shape(rows, cols, group_size, layout), dtype=torch.uint8, device=x.device)
    _check(lib().fp4_quantize(_p(x), rows, cols, mode, 4, group_size, _p(global_scale), _p(xq), _p(scales), layout,
                              _s(stream)), "fp4_quantize")
    return xq, scales


def fp4_quantize_sr(x: torch.Tensor, mode: int, seed: int, offset: int = 0, group_size: int = None,
                    global_scale=None, layout: int = SCALES_LINEAR, xq=None, scales=None, stream=None):
    """fp_quantize with stochastic rounding of the elements (Philox4x32-10 words
    from seed and offset); block scales as fp4_quantize."""
    group_size = group_size or GROUP[mode]
    rows, cols = x.shape
    if xq is None:
        xq = torch.empty((rows, cols // 8), dtype=torch.int32, device=x.device)
    if scales is None:
        scales = torch.empty(scales_shape(rows, cols, group_size, layout), dtype=torch.uint8, device=x.device)
    _check(lib().fp4_quantize_sr(_p(x), rows, cols, mode, 4, group_size, _p(global_scale), int(seed), int(offset),
                                 _p(xq), _p(scales), layout, _s(stream)), "fp4_quantize_sr")
    return xq, scales


def fp4_dequantize(wq: torch.Tensor, scales: torch.Tensor, biases=None, mode: int = MODE_NVFP4,
                   group_size: int = None, global_scale=None, layout: int = SCALES_LINEAR, out=None,
                   stream=None, rows: int = None):
    group_size = group_size or GROUP[mode]
    rows = rows if rows is not None else wq.shape[0]
    cols = wq.shape[-1] * 8
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.bfloat16, device=wq.device)
    _check(lib().fp4_dequantize(_p(wq), _p(scales), _p(biases), rows, cols, mode, 4, group_size,
                                _p(global_scale), layout, _p(out), _s(stream)), "fp4_dequantize")
    return out


def qmv(x: torch.Tensor, w: torch.Tensor, scales: torch.Tensor, biases=None, global_scale_w=None,
        mode: int = MODE_NVFP4, group_size: int = None, y=None, stream=None):
    group_size = group_size or GROUP[mode]
    N, K = w.shape[0], w.shape[1] * 8
    if y is None:
        y = torch.empty((N,), dtype=torch.bfloat16, device=w.device)
    _check(lib().qmv(_p(x), _p(w), _p(scales), _p(biases), _p(global_scale_w), N, K, mode, 4, group_size, _p(y),
                     _s(stream)), "qmv")
    return y


def qqmv(x: torch.Tensor, w: torch.Tensor, scales: torch.Tensor, global_scale_x=None, global_scale_w=None,
         mode: int = MODE_NVFP4, y=None, stream=None):
    """One-row quantized-activation GEMV: x is quantized and dequantized (bf16)
    inside the kernel, then multiplied by the 4-bit W."""
    N, K = w.shape[0], w.shape[1] * 8
    if y is None:
        y = torch.empty((N,), dtype=torch.bfloat16, device=w.device)
    _check(lib().qqmv(_p(x), _p(global_scale_x), _p(w), _p(scales), _p(global_scale_w), N, K, mode, _p(y),
                      _s(stream)), "qqmv")
    return y


def qqmm(xq: torch.Tensor, sx: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor, global_scale_x=None,
         global_scale_w=None, mode: int = MODE_NVFP4, out=None, stream=None, M: int = None):
    M = M if M is not None else xq.shape[0]
    N, K = wq.shape[0], wq.shape[1] * 8
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=wq.device)
    _check(lib().qqmm(_p(xq), _p(sx), _p(wq), _p(sw), _p(global_scale_x), _p(global_scale_w), M, N, K, mode,
                      _p(out), _s(stream)), "qqmm")
    return out


def qqmm_batched(xq: torch.Tensor, sx: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor, global_scale_x=None,
                 global_scale_w=None, mode: int = MODE_NVFP4, out=None, stream=None):
    """Batched FP4 x FP4 GEMM: xq [B, M, K/8] and its tiled scales [B, Mp, Cp];
    wq [B, N, K/8] (or [N, K/8], shared) and scales; out [B, M, N]; global
    scales as [B] arrays or None."""
    Bt, M, K = xq.shape[0], xq.shape[1], xq.shape[2] * 8
    shared = wq.dim() == 2
    N = wq.shape[-2]
    if out is None:
        out = torch.empty((Bt, M, N), dtype=torch.bfloat16, device=wq.device)
    _check(lib().qqmm_batched(_p(xq), _p(sx), _p(wq), _p(sw), _p(global_scale_x), _p(global_scale_w), Bt, M, N, K,
                              xq.stride(0), sx.stride(0), 0 if shared else wq.stride(0), 0 if shared else sw.stride(0),
                              out.stride(0), mode, _p(out), _s(stream)), "qqmm_batched")
    return out


def qqmm_quantize_x_workspace(M: int, K: int, mode: int = MODE_NVFP4, device="cuda"):
    """A zero-filled workspace for qqmm_quantize_x (allocate once, reuse)."""
    n = lib().qqmm_quantize_x_workspace_bytes(M, K, mode)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def qqmm_quantize_x(x: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor, ws: torch.Tensor, global_scale_x=None,
                    global_scale_w=None, mode: int = MODE_NVFP4, global_scale_x_out=None, out=None, stream=None):
    """Quantize bf16 x [M, K] and multiply by FP4 W in one launch."""
    M, K = x.shape
    N = wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=wq.device)
    _check(lib().qqmm_quantize_x(_p(x), _p(global_scale_x), _p(wq), _p(sw), _p(global_scale_w), M, N, K, mode,
                                 _p(ws), ws.numel(), _p(global_scale_x_out), _p(out), _s(stream)), "qqmm_quantize_x")
    return out


def gather_qmm(x: torch.Tensor, lhs_idx: torch.Tensor, rhs_idx: torch.Tensor, w: torch.Tensor,
               scales: torch.Tensor, biases=None, mode: int = MODE_MXFP4, group_size: int = None,
               sorted_indices: bool = True, out=None, stream=None):
    group_size = group_size or GROUP[mode]
    R = lhs_idx.numel()
    E, N, K = w.shape[0], w.shape[1], w.shape[2] * 8
    if out is None:
        out = torch.empty((R, N), dtype=torch.bfloat16, device=w.device)
    _check(lib().gather_qmm(_p(x), _p(lhs_idx), _p(rhs_idx), R, _p(w), _p(scales), _p(biases), E, N, K, mode, 4,
                            group_size, 1 if sorted_indices else 0, _p(out), _s(stream)), "gather_qmm")
    return out


class MatrixGroup(c.Structure):
    """fp4_matrix_group: up to 4 matrices of one K for qmv_grouped."""
    _fields_ = [("count", c.c_int), ("w", c.c_void_p * 4), ("scales", c.c_void_p * 4), ("biases", c.c_void_p * 4),
                ("global_scale_w", c.c_void_p * 4), ("N", c.c_int64 * 4), ("K", c.c_int64)]


def matrix_group(mats) -> MatrixGroup:
    """mats: a list of (w, scales, biases, global_scale_w) tuples (None where absent)."""
    g = MatrixGroup()
    g.count = len(mats)
    for i, (w, s, b, gs) in enumerate(mats):
        g.w[i] = w.data_ptr()
        g.scales[i] = s.data_ptr()
        g.biases[i] = b.data_ptr() if b is not None else None
        g.global_scale_w[i] = gs.data_ptr() if gs is not None else None
        g.N[i] = w.shape[0]
    g.K = mats[0][0].shape[1] * 8
    return g


def qmv_grouped(x: torch.Tensor, mats, mode: int = MODE_NVFP4, group_size: int = None, ys=None, stream=None,
                prefetch_next=None):
    """One x against up to 4 matrices of the same K in one launch.  mats: a list of
    (w, scales, biases, global_scale_w) tuples; prefetch_next: the same for the
    GEMV launched next (an L2 warm-up hint) or None.  Returns the y vectors."""
    group_size = group_size or GROUP[mode]
    g = mats if isinstance(mats, MatrixGroup) else matrix_group(mats)
    if ys is None:
        ys = [torch.empty((int(g.N[i]),), dtype=torch.bfloat16, device=x.device) for i in range(g.count)]
    yy = (c.c_void_p * g.count)(*[y.data_ptr() for y in ys])
    nx = None
    if prefetch_next is not None:
        nx = prefetch_next if isinstance(prefetch_next, MatrixGroup) else matrix_group(prefetch_next)
    _check(lib().qmv_grouped(_p(x), c.byref(g), mode, 4, group_size, yy, c.byref(nx) if nx is not None else None,
                             _s(stream)), "qmv_grouped")
    return ys


def gather_rows(x: torch.Tensor, idx: torch.Tensor, out=None, stream=None):
    """out[i] = x[idx[i]] (bf16 rows; the routed activations in routing order)."""
    R, (T, K) = idx.numel(), x.shape
    if out is None:
        out = torch.empty((R, K), dtype=x.dtype, device=x.device)
    _check(lib().gather_rows(_p(x), T, _p(idx), R, K, _p(out), _s(stream)), "gather_rows")
    return out


def qmm(x: torch.Tensor, w: torch.Tensor, scales: torch.Tensor, biases=None, global_scale_w=None,
        mode: int = MODE_NVFP4, group_size: int = None, out=None, stream=None):
    """Dense W4A16 GEMM: out = x . deq(W)^T with x bf16 [M, K] and 4-bit W [N, K]."""
    group_size = group_size or GROUP[mode]
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=w.device)
    _check(lib().qmm(_p(x), _p(w), _p(scales), _p(biases), _p(global_scale_w), M, N, K, mode, 4, group_size, _p(out),
                     _s(stream)), "qmm")
    return out


def fp4_debug_stream_weights(wq: torch.Tensor, scales: torch.Tensor, stream=None):
    """Stream NVFP4 weights as qmv's tensor-core path does, computing nothing
    (the launch-and-stream ceiling of that kernel shape)."""
    N, K = wq.shape[0], wq.shape[1] * 8
    _check(lib().fp4_debug_stream_weights(_p(wq), _p(scales), N, K, _s(stream)), "fp4_debug_stream_weights")


def fp4_debug_inject_wait_timeout(enable: bool):
    _check(lib().fp4_debug_inject_wait_timeout(1 if enable else 0), "fp4_debug_inject_wait_timeout")
