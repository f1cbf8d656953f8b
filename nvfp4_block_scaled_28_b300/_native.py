"""ctypes loader for the in-tree C-ABI library ``libnvfp4_b300.so``.

There is no fallback: if the library is missing or fails to load, every
entry point raises. Signatures mirror ``include/nvfp4.h``.
"""
from __future__ import annotations

import ctypes
import os
import threading

# NVFP4_B300_DEBUG=1 in the environment loads the debug build instead: the same
# kernels with device-side bounds checks (nvfp4_device_error reports a failed
# one as ERR_BOUNDS); build.build() compiles both.
DEBUG = os.environ.get("NVFP4_B300_DEBUG") == "1"
LIB_NAME = "libnvfp4_b300_debug.so" if DEBUG else "libnvfp4_b300.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), LIB_NAME)

# nvfp4_status
OK = 0
ERR_INVALID_ARG = 1
ERR_MISALIGNED = 2
ERR_UNSUPPORTED_SHAPE = 3
ERR_WORKSPACE_TOO_SMALL = 4
ERR_CUDA = 5
ERR_TIMEOUT = 6
ERR_BOUNDS = 7

# nvfp4_sf_layout
SF_ROW_MAJOR = 0
SF_MMA_128x4 = 1

# nvfp4_linear_mode
LINEAR_UNFUSED = 0
LINEAR_FUSED = 1
# nvfp4_scale_rule
SCALE_ABSMAX = 0
SCALE_FOUR_OVER_SIX = 1
SCALE_MSE = 2

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_INT = ctypes.c_int
_U32 = ctypes.c_uint32

# name -> (restype, argtypes), in header order
SIGNATURES = {
    "nvfp4_status_string": (ctypes.c_char_p, [_INT]),
    "nvfp4_sf_bytes": (_SZ, [_I64, _I64, _INT]),
    "nvfp4_global_scale": (_INT, [_P, _I64, _I64, _I64, _P, _P]),
    "nvfp4_quantize": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _INT, _P]),
    "nvfp4_quantize_select": (_INT, [_P, _I64, _I64, _I64, _P, _INT, _P, _P, _INT, _P]),
    "nvfp4_quantize_weight": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _INT, _P]),
    "nvfp4_sf_to_mma_layout": (_INT, [_P, _I64, _I64, _P, _P]),
    "nvfp4_gemm": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P]),
    "nvfp4_gemm_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "nvfp4_linear": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _I64, _P, _INT, _P,
                            _SZ, _P]),
    "nvfp4_linear_workspace_bytes": (_SZ, [_I64, _I64, _I64, _INT]),
    "nvfp4_linear_grouped": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _P, _INT, _P, _I64, _P,
                                    _INT, _P, _SZ, _P]),
    "nvfp4_linear_noalloc": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _I64, _P, _P]),
    "nvfp4_linear_bias_requant": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _P, _I64,
                                         _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_linear_bias_requant_dynamic": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _P,
                                                 _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_linear_lora": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _P, _I64,
                                 ctypes.c_float, _P, _I64, _P, _P, _SZ, _P]),
    "nvfp4_linear_lora_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I64]),
    "nvfp4_device_error": (_INT, [_INT]),
    "nvfp4_debug_set_fault_injection": (_INT, [_INT, _U32]),
    "nvfp4_debug_select_gemm_kernel": (_INT, [_INT]),
    "nvfp4_debug_capture_fused_operand": (_INT, [_INT]),
}

_lock = threading.Lock()
_lib = None


class NVFP4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s" % (fn, status_string(status)))


def load() -> ctypes.CDLL:
    """Load the library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                "%s is not built; run `python -m nvfp4_block_scaled_28_b300.build` "
                "(or __graft_entry__.build())" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


PROBE_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnvfp4_probe.so")
# the measurement library of include/nvfp4_probe.h
PROBE_SIGNATURES = {
    "nvfp4_mma_peak_probe": (_INT, [_INT, _INT, _INT, _P, _P]),
    "nvfp4_probe_error": (_INT, [_INT]),
}
_probe = None


def load_probe() -> ctypes.CDLL:
    """Load the measurement library (once). Raises if it has not been built."""
    global _probe
    with _lock:
        if _probe is not None:
            return _probe
        if not os.path.exists(PROBE_LIB_PATH):
            raise ImportError("%s is not built; run `python -m nvfp4_block_scaled_28_b300.build`"
                              % PROBE_LIB_PATH)
        lib = ctypes.CDLL(PROBE_LIB_PATH)
        for name, (res, args) in PROBE_SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _probe = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().nvfp4_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - only when the library is absent
        return "status %d" % status


def check(fn: str, status: int) -> None:
    if status != OK:
        raise NVFP4Error(fn, status)
