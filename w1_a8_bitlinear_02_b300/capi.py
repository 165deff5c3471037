"""ctypes declarations of libbitlinear.so (mirrors include/bitlinear.h).

Only argument marshalling lives here.  The library is loaded lazily on first
use and a missing build raises ImportError: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbitlinear.so")

BL_OK = 0
BL_ERR_NULL = 1
BL_ERR_SHAPE = 2
BL_ERR_DTYPE = 3
BL_ERR_ALIGN = 4
BL_ERR_WORKSPACE = 5
BL_ERR_CUDA = 6
BL_ERR_UNSUPPORTED = 7
BL_ERR_DEVICE = 8

BL_F32 = 0
BL_BF16 = 1

BL_ACT_NONE = 0
BL_ACT_RELU2 = 1


class ChainCall(ctypes.Structure):
    """bl_chain_call (include/bitlinear.h)."""
    _fields_ = [("packed", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("x_dtype", ctypes.c_int), ("act", ctypes.c_int), ("wait_prev", ctypes.c_int),
                ("M", ctypes.c_int)]


# name -> (restype, argtypes)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
SIGNATURES = {
    "bitlinear_version": (_INT, []),
    "bitlinear_status_string": (ctypes.c_char_p, [_INT]),
    "bitlinear_packed_row_bytes": (_INT, [_I64, ctypes.POINTER(_I64)]),
    "bitlinear_packed_bytes": (_INT, [_I64, _I64, ctypes.POINTER(_SZ)]),
    "bitlinear_pack_workspace_bytes": (_INT, [_I64, _I64, ctypes.POINTER(_SZ)]),
    "bitlinear_pack_weights": (_INT, [_P, _INT, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "bitlinear_quant_act": (_INT, [_P, _INT, _I64, _I64, _P, _P, _P]),
    "bitlinear_rmsnorm_quant_act": (_INT, [_P, _INT, _P, _F, _I64, _I64, _P, _P, _P]),
    "bitlinear_workspace_bytes": (_INT, [_I64, _I64, _I64, ctypes.POINTER(_SZ)]),
    "bitlinear_forward": (_INT, [_P, _P, _I64, _I64, _P, _INT, _I64, _P, _P, _SZ, _P]),
    "bitlinear_forward_q": (_INT, [_P, _P, _I64, _I64, _P, _P, _I64, _P, _P, _SZ, _P]),
    "bitlinear_matmul_i32": (_INT, [_P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P]),
    "bitlinear_forward_noalloc": (_INT, [_P, _P, _I64, _I64, _P, _INT, _I64, _P, _P]),
    "bitlinear_relu2_quant_act": (_INT, [_P, _INT, _I64, _I64, _P, _P, _P]),
    "bitlinear_forward_chain": (_INT, [_P, _INT, _P, _SZ, _P]),
    "bitlinear_chain_workspace_bytes": (_INT, [_P, _INT, ctypes.POINTER(_SZ)]),
    "bitlinear_forward_ex": (_INT, [_P, _P, _I64, _I64, _P, _INT, _I64, _INT, _P, _INT, _P, _P, _SZ, _P]),
    "bitlinear_pack_weights_grouped": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "bitlinear_forward_grouped": (_INT, [_P, _P, _I64, _I64, _I64, _P, _INT, _I64, _INT, _P, _INT, _P, _P, _SZ,
                                         _P]),
    "bitlinear_forward_relu2": (_INT, [_P, _P, _I64, _I64, _P, _INT, _I64, _P, _P, _SZ, _P]),
    "bitlinear_set_launch_overlap": (None, [_INT]),
    "bitlinear_get_launch_overlap": (_INT, []),
    "bitlinear_device_error": (_INT, [ctypes.POINTER(ctypes.c_uint), _INT]),
}

_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libbitlinear.so (built in-tree) and declare every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m w1_a8_bitlinear_02_b300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class BitLinearError(RuntimeError):
    def __init__(self, status: int, where: str):
        text = load().bitlinear_status_string(status).decode()
        super().__init__(f"{where}: status {status} ({text})")
        self.status = status


def check(status: int, where: str) -> None:
    if status != BL_OK:
        raise BitLinearError(status, where)
