"""ctypes loader for libqat.so, the CUDA library's C ABI (include/qat.h).

The library is built in-tree by ``fake_quant_numerics_gb300.build``.  There is
no fallback: if the shared object cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqat.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "qat.h")

# status codes and flags (include/qat.h)
QAT_OK = 0
QAT_ERR_INVALID_ARGUMENT = 1
QAT_ERR_DIMENSION_MISMATCH = 2
QAT_ERR_UNSUPPORTED = 3
QAT_ERR_CUDA = 4
QAT_ERR_MISALIGNED = 5
QAT_ERR_WORKSPACE = 6
FLAG_NONFINITE_CALIB = 1
FLAG_DEGENERATE = 2
FLAG_BAD_PARAMS = 4
FLAG_NONFINITE_INPUT = 8
FLAG_DEVICE_TIMEOUT = 16
F32, BF16 = 0, 1
SYMMETRIC, AFFINE = 0, 1
PER_TENSOR, PER_ROW, PER_GROUP, PER_COLUMN = 0, 1, 2, 3
E4M3, E5M2 = 0, 1

_lib = None

_vp, _i64, _int, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t

_u64 = ctypes.c_uint64


class AdamHparams(ctypes.Structure):
    """qat_adam_hparams (include/qat.h)."""
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("bias_correction1", ctypes.c_float), ("bias_correction2", ctypes.c_float)]


class CalibOptions(ctypes.Structure):
    """qat_calib_options (include/qat.h)."""
    _fields_ = [("clip", ctypes.c_float), ("scale_fp16", ctypes.c_int)]


PROTOTYPES = {
    "qat_status_string": ([_int], ctypes.c_char_p),
    "qat_workspace_bytes": ([_i64, _i64, _int, _i64], _sz),
    "qat_amax_stats": ([_vp, _int, _i64, _i64, _int, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "qat_fake_quant_int": ([_vp, _int, _i64, _i64, _int, _int, _int, _i64, _int, _vp, _vp, _vp, _vp,
                            _vp, _vp, _vp, _sz, _vp], _int),
    "qat_fake_quant_fp8": ([_vp, _int, _i64, _int, _int, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "qat_fake_quant_fp8_noalloc": ([_vp, _int, _i64, _int, _int, _vp, _vp, _vp, _vp, _vp, _vp], _int),
    "qat_fake_quant_int_opts": ([_vp, _int, _i64, _i64, _int, _int, _int, _i64, _vp, _int, _u64, _u64,
                                 _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "qat_fake_quant_block": ([_vp, _int, _i64, _int, _i64, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _sz, _vp], _int),
    "qat_percentile_workspace_bytes": ([], _sz),
    "qat_fake_quant_int_percentile": ([_vp, _int, _i64, _int, _int, ctypes.c_double, _int, _u64,
                                       _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "qat_fake_quant_int_sr": ([_vp, _int, _i64, _i64, _int, _int, _int, _i64, _int, _vp, _vp, _u64,
                               _u64, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "qat_optimizer_step": ([_vp, _vp, _vp, _vp, _i64, ctypes.POINTER(AdamHparams), _int, _int, _int,
                            _int, _u64, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "qat_fake_quant_fp8_sr": ([_vp, _int, _i64, _int, _int, _vp, _u64, _u64, _vp, _vp, _vp, _vp, _vp,
                               _sz, _vp], _int),
    "qat_ste_backward": ([_vp, _int, _i64, _vp, _vp, _vp], _int),
    "qat_quant4_double": ([_vp, _i64, _vp, _vp, _vp, _vp, _vp], _int),
    "qat_dequant4_double": ([_vp, _vp, _vp, _i64, _vp, _vp], _int),
    "qat_kernel_launch_count": ([], ctypes.c_uint64),
    "qat_debug_set_wait_limit": ([_i64], None),
}


class QatError(RuntimeError):
    """A non-OK status returned by the C ABI."""

    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().qat_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn}: {msg} (status {status})")


def header_symbols(path: str = HEADER):
    """Function names declared in include/qat.h."""
    with open(path) as f:
        txt = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(qat_\w+)\s*\(", txt, re.M)))


def load(build_if_missing: bool = True):
    """Load libqat.so (building it in-tree first if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        if not build_if_missing:
            raise RuntimeError(f"{LIB_PATH} is not built (run __graft_entry__.build())")
        from . import build as _build

        _build.build()
    L = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in PROTOTYPES.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return _lib


def lib():
    return _lib if _lib is not None else load()


def check(fn: str, status: int):
    if status != QAT_OK:
        raise QatError(fn, status)
