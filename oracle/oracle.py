"""ctypes wrapper around the C oracle (``nvfp4_oracle.c``).

Test infrastructure only (see the package docstring). Arrays cross the
boundary as numpy arrays: bfloat16 tensors travel as their uint16 bit
patterns, packed codes and E4M3 scales as uint8.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def lib_path() -> str:
    return _LIB


_CFLAGS = ["-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall"]


def _digest() -> str:
    """SHA-256 of the oracle source and the compiler flags."""
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(_CFLAGS).encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, OpenMP, no FMA
    contraction, no fast-math). Rebuilds whenever the SHA-256 of the source
    and flags differs from the one recorded at the last build (file times
    are not consulted)."""
    stamp = _LIB + ".sha256"
    digest = _digest()
    if not force and os.path.exists(_LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc"] + _CFLAGS + ["-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e2m1_value.argtypes = [ctypes.c_int]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_int]
        lib.oracle_e4m3_rne_satfinite.restype = ctypes.c_uint8
        lib.oracle_e4m3_rne_satfinite.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_rne_satfinite.restype = ctypes.c_int
        lib.oracle_e2m1_rne_satfinite.argtypes = [ctypes.c_float]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_global_scale.restype = ctypes.c_float
        lib.oracle_global_scale.argtypes = [_u16p, _i64, _i64, _i64]
        lib.oracle_quantize.restype = None
        lib.oracle_quantize.argtypes = [_u16p, _i64, _i64, _i64, ctypes.c_float,
                                        _u8p, _u8p]
        lib.oracle_quantize_rule.restype = None
        lib.oracle_quantize_rule.argtypes = [_u16p, _i64, _i64, _i64, ctypes.c_float,
                                             ctypes.c_int, _u8p, _u8p]
        lib.oracle_dequantize.restype = None
        lib.oracle_dequantize.argtypes = [_u8p, _u8p, ctypes.c_float, _i64, _i64,
                                          _f64p]
        lib.oracle_gemm_rows.restype = None
        lib.oracle_gemm_rows.argtypes = [_u8p, _u8p, ctypes.c_float, _u8p, _u8p,
                                         ctypes.c_float, _i64, _i64, _i64,
                                         _i64p, _i64, _u16p, _u16p, _f64p]
        lib.oracle_lora_rows.restype = None
        lib.oracle_lora_rows.argtypes = [_u16p, _i64, _i64, _u16p, _i64, _u16p, _i64,
                                         ctypes.c_double, _i64p, _i64, _f64p]
        lib.oracle_round_bf16.restype = None
        lib.oracle_round_bf16.argtypes = [_f64p, _i64, _u16p]
        lib.oracle_symmetric_quantize.restype = ctypes.c_double
        lib.oracle_symmetric_quantize.argtypes = [_f64p, _i64, ctypes.c_int,
                                                  _i32p, _f64p]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """Threads the oracle's parallel loops use (OpenMP)."""
    return int(_load().oracle_num_threads())


def e2m1_value(code: int) -> float:
    return float(_load().oracle_e2m1_value(int(code)))


def e4m3_value(byte: int) -> float:
    return float(_load().oracle_e4m3_value(int(byte)))


def e4m3_rne_satfinite(v: float) -> int:
    return int(_load().oracle_e4m3_rne_satfinite(float(v)))


def e2m1_rne_satfinite(y: float) -> int:
    return int(_load().oracle_e2m1_rne_satfinite(float(y)))


def bf16_from_double(y: float) -> int:
    return int(_load().oracle_bf16_from_double(float(y)))


def global_scale(x_bits: np.ndarray) -> float:
    """Per-tensor global scale of a 2-D bfloat16 tensor given as uint16 bits."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    return float(_load().oracle_global_scale(_ptr(x, _u16p), rows, cols, cols))


SCALE_ABSMAX, SCALE_FOUR_OVER_SIX, SCALE_MSE = 0, 1, 2


def quantize(x_bits: np.ndarray, g: float, rule: int = SCALE_ABSMAX):
    """Quantize a 2-D bfloat16 tensor (uint16 bits, cols % 16 == 0) with the
    decode-direction global scale ``g`` and a block-scale rule (absmax,
    four-over-six or MSE; "nvfp4-gemma4" page, section 2). Returns (codes
    uint8 rows x cols/2, scales uint8 rows x cols/16), both row-major."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    if cols % 16:
        raise ValueError("cols must be a multiple of 16")
    if rule not in (SCALE_ABSMAX, SCALE_FOUR_OVER_SIX, SCALE_MSE):
        raise ValueError("unknown scale rule %r" % rule)
    q = np.empty((rows, cols // 2), np.uint8)
    s = np.empty((rows, cols // 16), np.uint8)
    if rule == SCALE_ABSMAX:
        _load().oracle_quantize(_ptr(x, _u16p), rows, cols, cols, float(g),
                                _ptr(q, _u8p), _ptr(s, _u8p))
    else:
        _load().oracle_quantize_rule(_ptr(x, _u16p), rows, cols, cols, float(g), int(rule),
                                     _ptr(q, _u8p), _ptr(s, _u8p))
    return q, s


def dequantize(q: np.ndarray, s: np.ndarray, g: float) -> np.ndarray:
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    rows, half = q.shape
    out = np.empty((rows, half * 2), np.float64)
    _load().oracle_dequantize(_ptr(q, _u8p), _ptr(s, _u8p), float(g), rows,
                              half * 2, _ptr(out, _f64p))
    return out


def gemm_rows(xq, xs, g_x, wq, ws, g_w, rows=None, want_fp64=False, bias=None):
    """Reference Y = bf16((Xhat @ What^T) * g_x * g_w + bias) for the listed
    rows of X (all rows if ``rows`` is None; ``bias``: optional bfloat16 bits,
    uint16 of length N, added in FP64 before the rounding). Returns uint16
    bf16 bits (and the FP64 values before rounding when ``want_fp64``)."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.uint8)
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.uint8)
    M, kh = xq.shape
    N = wq.shape[0]
    K = kh * 2
    if rows is None:
        ids = None
        n_rows = M
    else:
        ids = _c(rows, np.int64)
        n_rows = ids.shape[0]
    y = np.empty((n_rows, N), np.uint16)
    yd = np.empty((n_rows, N), np.float64) if want_fp64 else None
    b = None if bias is None else _c(bias, np.uint16)
    if b is not None:
        assert b.shape == (N,)
    _load().oracle_gemm_rows(
        _ptr(xq, _u8p), _ptr(xs, _u8p), float(g_x), _ptr(wq, _u8p),
        _ptr(ws, _u8p), float(g_w), M, N, K,
        None if ids is None else _ptr(ids, _i64p), n_rows,
        None if b is None else _ptr(b, _u16p),
        _ptr(y, _u16p), None if yd is None else _ptr(yd, _f64p))
    return (y, yd) if want_fp64 else y


def gemm(xq, xs, g_x, wq, ws, g_w, want_fp64=False, bias=None):
    return gemm_rows(xq, xs, g_x, wq, ws, g_w, None, want_fp64, bias)


def lora_rows(x_bits, a_bits, b_bits, scale, rows=None):
    """FP64 low-rank correction scale * (X @ A^T) @ B^T on the bfloat16
    activation (uint16 bits M x K), A r x K, B N x r, for the listed rows."""
    x = _c(x_bits, np.uint16)
    a = _c(a_bits, np.uint16)
    b = _c(b_bits, np.uint16)
    M, K = x.shape
    r = a.shape[0]
    N = b.shape[0]
    assert a.shape == (r, K) and b.shape == (N, r)
    ids = None if rows is None else _c(rows, np.int64)
    n_rows = M if ids is None else ids.shape[0]
    out = np.empty((n_rows, N), np.float64)
    _load().oracle_lora_rows(_ptr(x, _u16p), K, K, _ptr(a, _u16p), r, _ptr(b, _u16p), N,
                             float(scale), None if ids is None else _ptr(ids, _i64p), n_rows,
                             _ptr(out, _f64p))
    return out


def round_bf16(y: np.ndarray) -> np.ndarray:
    """Round FP64 values once to bfloat16 bits."""
    yy = _c(y, np.float64)
    out = np.empty(yy.shape, np.uint16)
    _load().oracle_round_bf16(_ptr(yy, _f64p), yy.size, _ptr(out, _u16p))
    return out


def linear_lora_rows(xq, xs, g_x, wq, ws, g_w, x_bits, a_bits, b_bits, scale, rows=None):
    """Reference NVFP4 linear with a LoRA correction: bf16( (Xhat @ What^T)
    * g_x * g_w + scale * (X @ A^T) @ B^T ), both terms in FP64, one rounding."""
    _, yd = gemm_rows(xq, xs, g_x, wq, ws, g_w, rows, want_fp64=True)
    return round_bf16(yd + lora_rows(x_bits, a_bits, b_bits, scale, rows))


def symmetric_quantize(x, bits: int):
    """Symmetric integer quantization (FP64). Returns (s, q int32, x_hat)."""
    xx = _c(x, np.float64)
    n = xx.shape[0]
    q = np.empty(n, np.int32)
    xh = np.empty(n, np.float64)
    s = _load().oracle_symmetric_quantize(_ptr(xx, _f64p), n, int(bits),
                                          _ptr(q, _i32p), _ptr(xh, _f64p))
    return float(s), q, xh
