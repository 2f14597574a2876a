"""CPU oracle for block-scaled 4-bit quantization and matmul.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` import this
package.  The product path (``block_scaled_fp4_fp_gb300``) never imports it, and
the two share no code: the arithmetic lives in ``fp4_oracle.c`` (plain C,
scalar loops, fp64 accumulation), and this module only marshals numpy arrays
through ``ctypes``.

bf16 arrays are passed as ``numpy.uint16`` bit patterns.  Parity status of each
function is stated in ``fp4_oracle.c``; every function here is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4_oracle.c")
_HDR = os.path.join(_HERE, "fp4_oracle.h")
_LIB = os.path.join(_HERE, "libfp4oracle.so")
_lock = threading.Lock()
_lib = None

MODE_AFFINE, MODE_MXFP4, MODE_NVFP4 = 0, 1, 2

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile ``fp4_oracle.c`` into ``libfp4oracle.so`` next to it (gcc)."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _p(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t)) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            c = ctypes
            i64, u16, u32, u8, f32, f64, i32 = (c.c_int64, c.c_uint16, c.c_uint32, c.c_uint8,
                                                c.c_float, c.c_double, c.c_int32)
            P = c.POINTER
            sig = {
                "orc_e2m1_decode": (f64, [c.c_uint]),
                "orc_e2m1_encode": (c.c_uint, [f32]),
                "orc_e4m3_decode": (f64, [c.c_uint]),
                "orc_e4m3_encode": (c.c_uint, [f32]),
                "orc_e8m0_decode": (f64, [c.c_uint]),
                "orc_bf16_to_double": (f64, [u16]),
                "orc_bf16_from_double": (u16, [f64]),
                "orc_bf16_from_float": (u16, [f32]),
                "orc_amax": (f32, [P(u16), i64]),
                "orc_global_scale": (f32, [P(u16), i64]),
                "orc_alpha_from_amax": (f32, [f32, f32]),
                "orc_nvfp4_quantize": (None, [P(u16), i64, i64, P(f32), P(u32), P(u8)]),
                "orc_mxfp4_quantize": (None, [P(u16), i64, i64, P(u32), P(u8)]),
                "orc_affine_quantize": (None, [P(u16), i64, i64, c.c_int, P(u32), P(u16), P(u16)]),
                "orc_philox4x32_10": (None, [P(u32), P(u32), P(u32)]),
                "orc_sr_word": (u32, [c.c_uint64, c.c_uint64, c.c_uint64]),
                "orc_e2m1_encode_sr": (c.c_uint, [f32, u32]),
                "orc_nvfp4_quantize_sr": (None, [P(u16), i64, i64, P(f32), c.c_uint64, c.c_uint64, P(u32), P(u8)]),
                "orc_mxfp4_quantize_sr": (None, [P(u16), i64, i64, c.c_uint64, c.c_uint64, P(u32), P(u8)]),
                "orc_padded_rows": (i64, [i64]),
                "orc_padded_cols": (i64, [i64]),
                "orc_tiled_offset": (i64, [i64, i64, i64]),
                "orc_tile_scales": (None, [P(u8), i64, i64, P(u8)]),
                "orc_untile_scales": (None, [P(u8), i64, i64, P(u8)]),
                "orc_dequantize_f64": (None, [P(u32), c.c_void_p, P(u16), i64, i64, c.c_int, c.c_int,
                                              P(f32), P(f64)]),
                "orc_dequantize_bf16": (None, [P(u32), c.c_void_p, P(u16), i64, i64, c.c_int, c.c_int,
                                               P(f32), P(u16)]),
                "orc_qmv": (None, [P(u16), P(u32), c.c_void_p, P(u16), P(f32), i64, i64, c.c_int,
                                   c.c_int, P(i64), i64, P(f64)]),
                "orc_qqmm": (None, [P(u32), P(u8), P(u32), P(u8), f32, i64, i64, i64, c.c_int,
                                    P(i64), i64, P(i64), i64, P(f64)]),
                "orc_qmm": (None, [P(u16), i64, P(u32), c.c_void_p, P(u16), P(f32), i64, i64, c.c_int, c.c_int,
                                   P(i64), i64, P(f64)]),
                "orc_gather_qmm": (None, [P(u16), P(i32), P(i32), i64, P(u32), c.c_void_p, P(u16),
                                          i64, i64, i64, c.c_int, c.c_int, P(i64), i64, P(f64)]),
                "orc_num_threads": (c.c_int, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _f32p(v):
    if v is None:
        return None
    return ctypes.pointer(ctypes.c_float(float(v)))


# ---- scalar codecs ---------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def e4m3_decode(b: int) -> float:
    return lib().orc_e4m3_decode(int(b))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def e8m0_decode(b: int) -> float:
    return lib().orc_e8m0_decode(int(b))


def bf16_from_double(v: float) -> int:
    return lib().orc_bf16_from_double(float(v))


def bf16_to_double(b: int) -> float:
    return lib().orc_bf16_to_double(int(b))


def bf16_round_array(a: np.ndarray) -> np.ndarray:
    """Round every fp64 value of ``a`` to bf16 (RNE); returns uint16 bits."""
    f = lib().orc_bf16_from_double
    flat = np.asarray(a, dtype=np.float64).ravel()
    return np.fromiter((f(float(v)) for v in flat), dtype=np.uint16, count=flat.size).reshape(np.shape(a))


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ---- global scale ----------------------------------------------------------

def amax(x: np.ndarray) -> float:
    x = _c(x, np.uint16)
    return lib().orc_amax(_p(x, ctypes.c_uint16), x.size)


def global_scale(x: np.ndarray) -> float:
    x = _c(x, np.uint16)
    return lib().orc_global_scale(_p(x, ctypes.c_uint16), x.size)


def alpha_from_amax(amax_x: float, amax_w: float) -> float:
    return lib().orc_alpha_from_amax(float(amax_x), float(amax_w))


# ---- quantizers ------------------------------------------------------------

def nvfp4_quantize(x: np.ndarray, gs=None):
    """x: uint16 bf16 bits [rows, cols]; gs: float or None -> (q u32 [rows, cols/8], s u8 [rows, cols/16])."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    q = np.zeros((rows, cols // 8), np.uint32)
    s = np.zeros((rows, cols // 16), np.uint8)
    lib().orc_nvfp4_quantize(_p(x, ctypes.c_uint16), rows, cols, _f32p(gs),
                             _p(q, ctypes.c_uint32), _p(s, ctypes.c_uint8))
    return q, s


def mxfp4_quantize(x: np.ndarray):
    x = _c(x, np.uint16)
    rows, cols = x.shape
    q = np.zeros((rows, cols // 8), np.uint32)
    s = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_mxfp4_quantize(_p(x, ctypes.c_uint16), rows, cols, _p(q, ctypes.c_uint32),
                             _p(s, ctypes.c_uint8))
    return q, s


def affine_quantize(w: np.ndarray, group: int = 64):
    w = _c(w, np.uint16)
    rows, cols = w.shape
    q = np.zeros((rows, cols // 8), np.uint32)
    s = np.zeros((rows, cols // group), np.uint16)
    b = np.zeros((rows, cols // group), np.uint16)
    lib().orc_affine_quantize(_p(w, ctypes.c_uint16), rows, cols, group, _p(q, ctypes.c_uint32),
                              _p(s, ctypes.c_uint16), _p(b, ctypes.c_uint16))
    return q, s, b


def quantize(x: np.ndarray, mode: int, gs=None):
    if mode == MODE_NVFP4:
        return nvfp4_quantize(x, gs)
    if mode == MODE_MXFP4:
        return mxfp4_quantize(x)
    raise ValueError("oracle quantize: mode must be NVFP4 or MXFP4")


# ---- stochastic rounding ---------------------------------------------------

def philox4x32_10(ctr, key):
    """Philox4x32-10 of a 4-word counter under a 2-word key -> 4 uint32 words."""
    c = (ctypes.c_uint32 * 4)(*[int(v) & 0xFFFFFFFF for v in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(v) & 0xFFFFFFFF for v in key])
    o = (ctypes.c_uint32 * 4)()
    lib().orc_philox4x32_10(c, k, o)
    return [int(v) for v in o]


def sr_word(seed: int, offset: int, e: int) -> int:
    return int(lib().orc_sr_word(int(seed), int(offset), int(e)))


def e2m1_encode_sr(v: float, u: int) -> int:
    return int(lib().orc_e2m1_encode_sr(float(v), int(u)))


def quantize_sr(x: np.ndarray, mode: int, gs=None, seed: int = 0, offset: int = 0):
    """Stochastic-rounding fp_quantize (rule and random numbers in fp4_oracle.c)."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    g = 16 if mode == MODE_NVFP4 else 32
    q = np.zeros((rows, cols // 8), np.uint32)
    s = np.zeros((rows, cols // g), np.uint8)
    if mode == MODE_NVFP4:
        lib().orc_nvfp4_quantize_sr(_p(x, ctypes.c_uint16), rows, cols, _f32p(gs), int(seed), int(offset),
                                    _p(q, ctypes.c_uint32), _p(s, ctypes.c_uint8))
    elif mode == MODE_MXFP4:
        if gs is not None:
            raise ValueError("MXFP4 has no global scale")
        lib().orc_mxfp4_quantize_sr(_p(x, ctypes.c_uint16), rows, cols, int(seed), int(offset),
                                    _p(q, ctypes.c_uint32), _p(s, ctypes.c_uint8))
    else:
        raise ValueError("oracle quantize_sr: mode must be NVFP4 or MXFP4")
    return q, s


# ---- tiles -----------------------------------------------------------------

def padded_dims(rows: int, cols: int):
    L = lib()
    return L.orc_padded_rows(rows), L.orc_padded_cols(cols)


def tiled_offset(r: int, c: int, padded_cols: int) -> int:
    return lib().orc_tiled_offset(r, c, padded_cols)


def tile_scales(lin: np.ndarray) -> np.ndarray:
    lin = _c(lin, np.uint8)
    rows, cols = lin.shape
    rp, cp = padded_dims(rows, cols)
    t = np.zeros((rp, cp), np.uint8)
    lib().orc_tile_scales(_p(lin, ctypes.c_uint8), rows, cols, _p(t, ctypes.c_uint8))
    return t


def untile_scales(tiled: np.ndarray, rows: int, cols: int) -> np.ndarray:
    tiled = _c(tiled, np.uint8)
    lin = np.zeros((rows, cols), np.uint8)
    lib().orc_untile_scales(_p(tiled, ctypes.c_uint8), rows, cols, _p(lin, ctypes.c_uint8))
    return lin


# ---- dequantize ------------------------------------------------------------

def _scales_arg(mode, scales):
    if mode == MODE_AFFINE:
        s = _c(scales, np.uint16)
    else:
        s = _c(scales, np.uint8)
    return s, ctypes.c_void_p(s.ctypes.data)


def dequantize_f64(q, scales, biases, mode, group, gs=None):
    q = _c(q, np.uint32)
    rows, cols = q.shape[0], q.shape[1] * 8
    s, sp = _scales_arg(mode, scales)
    b = _c(biases, np.uint16) if biases is not None else None
    out = np.zeros((rows, cols), np.float64)
    lib().orc_dequantize_f64(_p(q, ctypes.c_uint32), sp, _p(b, ctypes.c_uint16), rows, cols, mode,
                             group, _f32p(gs), _p(out, ctypes.c_double))
    return out


def dequantize_bf16(q, scales, biases, mode, group, gs=None):
    q = _c(q, np.uint32)
    rows, cols = q.shape[0], q.shape[1] * 8
    s, sp = _scales_arg(mode, scales)
    b = _c(biases, np.uint16) if biases is not None else None
    out = np.zeros((rows, cols), np.uint16)
    lib().orc_dequantize_bf16(_p(q, ctypes.c_uint32), sp, _p(b, ctypes.c_uint16), rows, cols, mode,
                              group, _f32p(gs), _p(out, ctypes.c_uint16))
    return out


# ---- matmuls ---------------------------------------------------------------

def qmv(x, w, scales, biases, mode, group, gs_w=None, rows=None):
    """y[i] = x . deq(W)[rows[i]] in fp64 (all rows when ``rows`` is None)."""
    x = _c(x, np.uint16).ravel()
    w = _c(w, np.uint32)
    N, K = w.shape[0], w.shape[1] * 8
    s, sp = _scales_arg(mode, scales)
    b = _c(biases, np.uint16) if biases is not None else None
    r = _c(rows, np.int64) if rows is not None else None
    n_out = len(r) if r is not None else N
    y = np.zeros(n_out, np.float64)
    lib().orc_qmv(_p(x, ctypes.c_uint16), _p(w, ctypes.c_uint32), sp, _p(b, ctypes.c_uint16),
                  _f32p(gs_w), N, K, mode, group, _p(r, ctypes.c_int64), n_out,
                  _p(y, ctypes.c_double))
    return y


def qqmm(xq, sx, wq, sw, mode, alpha=1.0, mrows=None, ncols=None):
    """alpha * (code*scale of xq) . (code*scale of wq)^T in fp64; linear scales."""
    xq = _c(xq, np.uint32)
    wq = _c(wq, np.uint32)
    sx = _c(sx, np.uint8)
    sw = _c(sw, np.uint8)
    M, K = xq.shape[0], xq.shape[1] * 8
    N = wq.shape[0]
    mr = _c(mrows, np.int64) if mrows is not None else None
    nc = _c(ncols, np.int64) if ncols is not None else None
    om = len(mr) if mr is not None else M
    on = len(nc) if nc is not None else N
    out = np.zeros((om, on), np.float64)
    lib().orc_qqmm(_p(xq, ctypes.c_uint32), _p(sx, ctypes.c_uint8), _p(wq, ctypes.c_uint32),
                   _p(sw, ctypes.c_uint8), float(alpha), M, N, K, mode, _p(mr, ctypes.c_int64), om,
                   _p(nc, ctypes.c_int64), on, _p(out, ctypes.c_double))
    return out


def qmm(x, w, scales, biases, mode, group, gs_w=None, rows=None):
    """out[i] = x[rows[i]] . deq(W)^T in fp64 (all rows of x when ``rows`` is None);
    x is [M, K] bf16 bits, W [N, K/8] packed."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint32)
    M, K = x.shape
    N = w.shape[0]
    s, sp = _scales_arg(mode, scales)
    b = _c(biases, np.uint16) if biases is not None else None
    r = _c(rows, np.int64) if rows is not None else None
    om = len(r) if r is not None else M
    out = np.zeros((om, N), np.float64)
    lib().orc_qmm(_p(x, ctypes.c_uint16), M, _p(w, ctypes.c_uint32), sp, _p(b, ctypes.c_uint16), _f32p(gs_w), N, K,
                  mode, group, _p(r, ctypes.c_int64), om, _p(out, ctypes.c_double))
    return out


def gather_qmm(x, lhs, rhs, w, scales, biases, mode, group, rows=None):
    """out[i] = x[lhs[r_i]] . deq(W[rhs[r_i]])^T; w is [E, N, K/8]."""
    x = _c(x, np.uint16)
    lhs = _c(lhs, np.int32)
    rhs = _c(rhs, np.int32)
    w = _c(w, np.uint32)
    E, N, K = w.shape[0], w.shape[1], w.shape[2] * 8
    s, sp = _scales_arg(mode, scales)
    b = _c(biases, np.uint16) if biases is not None else None
    R = lhs.size
    r = _c(rows, np.int64) if rows is not None else None
    n_out = len(r) if r is not None else R
    out = np.zeros((n_out, N), np.float64)
    lib().orc_gather_qmm(_p(x, ctypes.c_uint16), _p(lhs, ctypes.c_int32), _p(rhs, ctypes.c_int32),
                         R, _p(w, ctypes.c_uint32), sp, _p(b, ctypes.c_uint16), E, N, K, mode, group,
                         _p(r, ctypes.c_int64), n_out, _p(out, ctypes.c_double))
    return out


GROUP_OF = {MODE_NVFP4: 16, MODE_MXFP4: 32}


def gather_rows(x, idx):
    """The routed activations in routing order: out[i] = x[idx[i]] (bf16 bits,
    "epic: NVIDIA Volta (sm_70) inference acceleration program #1536",
    Diagnosis 5: the grouped GEMM gathers each routed row)."""
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint16)[np.asarray(idx, dtype=np.int64)])


def quantize_dequantize(x, mode, gs=None):
    """fp_quantize_dequantize: quantize bf16 ``x`` [rows, cols] (NVFP4 with the
    optional multiplier-form global scale ``gs``, or MXFP4) and dequantize it
    back to bf16 bits -- the activation that the one-row route of QQMatmul
    multiplies ("mlx 0.30.7.3 -> 0.30.7.6", qqmm.cpp, QQMatmul::eval_gpu: with
    quantized W and one row, x goes through fp_quantize_dequantize into an array
    of x's own dtype, then fp_qmv).  Composition of the pinned quantizer and
    bf16 dequantizer; pinned by tests/test_oracle_qqmv.py."""
    q, s = quantize(x, mode, gs)
    return dequantize_bf16(q, s, None, mode, GROUP_OF[mode], gs)


def qqmv(x, w, scales, mode, gs_x=None, gs_w=None, rows=None):
    """The one-row quantized-activation GEMV: y = x_hat . deq(W)^T in fp64, where
    x_hat = quantize_dequantize(x) (bf16) and deq(W) includes the NVFP4 weight
    global scale ``gs_w`` (applied by this library's epilogue; MLX's fp_qmv
    leaves it to the caller)."""
    xh = quantize_dequantize(_c(x, np.uint16).reshape(1, -1), mode, gs_x)
    return qmv(xh.ravel(), w, scales, None, mode, GROUP_OF[mode], gs_w, rows)


def num_threads() -> int:
    return lib().orc_num_threads()
