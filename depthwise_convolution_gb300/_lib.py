"""ctypes view of libdwconv.so (the C ABI declared in include/dwconv.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_CUDA, ERR_TIMEOUT = range(6)
INT8, FP32, FP16, BF16, FP8_E4M3 = range(5)
ACT_NONE, ACT_RELU, ACT_RELU6, ACT_SILU, ACT_GELU = range(5)
ACTIVATIONS = {"none": ACT_NONE, "relu": ACT_RELU, "relu6": ACT_RELU6, "silu": ACT_SILU, "gelu": ACT_GELU}

# Exported symbols and their C signatures: name -> (restype, argtypes).
_I, _P, _SZ = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
SIGNATURES = {
    "dwconv_output_size": (_I, [_I] * 7 + [ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "dwconv_fwd": (_I, [_I] * 9 + [_I, _P, _P, _P, _P, _P]),
    "dwconv_bwd_data": (_I, [_I] * 9 + [_I, _P, _P, _P, _P]),
    "dwconv_bwd_filter_workspace_size": (_SZ, [_I] * 9 + [_I]),
    "dwconv_bwd_filter": (_I, [_I] * 9 + [_I, _P, _P, _P, _P, _SZ, _P]),
    "dwconv_bwd_filter_static": (_I, [_I] * 9 + [_I, _P, _P, _P, _P]),
    "dwconv_check_device_errors": (_I, [_P]),
    "dwconv_selftest_timeout": (_I, [_P]),
    "dwconv_status_string": (ctypes.c_char_p, [_I]),
    "dwconv_bwd_bias_workspace_size": (ctypes.c_size_t, [_I] * 4),
    "dwconv_bwd_bias": (_I, [_I] * 4 + [_I, _P, _P, _P, ctypes.c_size_t, _P]),
    "dwconv_output_size_2d": (_I, [_I] * 10 + [ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "dwconv_fwd_2d": (_I, [_I] * 12 + [_I, _P, _P, _P, _P, _P]),
    "dwconv_bwd_data_2d": (_I, [_I] * 12 + [_I, _P, _P, _P, _P]),
    "dwconv_bwd_filter_workspace_size_2d": (_SZ, [_I] * 12 + [_I]),
    "dwconv_bwd_filter_2d": (_I, [_I] * 12 + [_I, _P, _P, _P, _P, _SZ, _P]),
    "dwconv_fwd_fused": (_I, [_I] * 9 + [_I, _P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _P]),
    "dwconv_fwd_fused_2d": (_I, [_I] * 12 + [_I, _P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _P]),
    "dwconv_bwd_filter_ha": (_I, [_I] * 9 + [_I, _P, _P, _P, _P, _SZ, _P]),
    "dwconv_bwd_filter_ha_2d": (_I, [_I] * 12 + [_I, _P, _P, _P, _P, _SZ, _P]),
    "dwconv_launch_count": (ctypes.c_ulonglong, []),
    "dwconv_last_kernel": (ctypes.c_char_p, []),
}


class DwconvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib_path() -> str:
    """The in-tree library, or the build named by DWCONV_LIB (for A/B timing)."""
    return os.environ.get("DWCONV_LIB") or _build.LIB


def load(build_if_missing: bool = True):
    """The loaded library.  Builds it first if it is missing and nvcc exists."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"libdwconv.so is not built ({path}); run "
                                       "python -m depthwise_convolution_gb300.build")
                _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().dwconv_status_string(status).decode()


def check(status: int, where: str) -> None:
    if status != OK:
        raise DwconvError(status, where)
