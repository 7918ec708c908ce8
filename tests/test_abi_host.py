"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before anything is enqueued.

No test here touches a GPU: every call is built so that validation fails
before the first CUDA call (the fake pointers are never dereferenced because
the call returns first).
"""
import ctypes

import pytest

from fake_quant_numerics_gb300 import _lib as L

A = ctypes.c_void_p(0x10000)        # 32-byte aligned fake address, never dereferenced
MIS = ctypes.c_void_p(0x10000 + 8)  # misaligned fake address


@pytest.fixture(scope="module")
def lib():
    from fake_quant_numerics_gb300 import build

    build.build()
    return L.load(build_if_missing=False)


def test_every_header_symbol_is_exported(lib):
    names = L.header_symbols()
    assert set(names) >= {"qat_amax_stats", "qat_fake_quant_int", "qat_fake_quant_fp8",
                          "qat_ste_backward", "qat_quant4_double", "qat_dequant4_double",
                          "qat_workspace_bytes", "qat_status_string", "qat_kernel_launch_count"}
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.PROTOTYPES, n


def test_status_strings(lib):
    for s in range(7):
        assert lib.qat_status_string(s)
    assert lib.qat_status_string(99) == b"unknown status"


def test_workspace_bytes(lib):
    assert lib.qat_workspace_bytes(1, 1 << 20, L.PER_TENSOR, 0) == 1024 * 16
    # per unit of the fallback: a dead byte and a zero point, each array
    # rounded up to 16 bytes
    assert lib.qat_workspace_bytes(4096, 4096, L.PER_ROW, 0) == 4096 * 5
    assert lib.qat_workspace_bytes(14336, 4096, L.PER_GROUP, 128) == 14336 * 32 * 5
    assert lib.qat_workspace_bytes(3, 5, L.PER_ROW, 0) == 16 + 16
    # per column: a 16-byte accumulator per column, then the fallback's arrays
    assert lib.qat_workspace_bytes(4096, 4096, L.PER_COLUMN, 0) == 4096 * 16 + 4096 + 16384
    assert lib.qat_workspace_bytes(7, 33, L.PER_COLUMN, 0) == 33 * 16 + 48 + 144


def _int(lib, **kw):
    a = dict(x=A, dt=L.F32, rows=4, cols=64, bits=8, scheme=L.SYMMETRIC, gran=L.PER_TENSOR, group=0,
             given=0, scale=A, zp=A, y=A, codes=A, mask=A, flags=None, ws=None, wsb=0)
    a.update(kw)
    return lib.qat_fake_quant_int(a["x"], a["dt"], a["rows"], a["cols"], a["bits"], a["scheme"],
                                  a["gran"], a["group"], a["given"], a["scale"], a["zp"], a["y"],
                                  a["codes"], a["mask"], a["flags"], a["ws"], a["wsb"], None)


def test_int_argument_errors(lib):
    assert _int(lib, bits=3) == L.QAT_ERR_UNSUPPORTED          # IntDtype::from_bits(3)
    assert _int(lib, bits=16) == L.QAT_ERR_UNSUPPORTED
    assert _int(lib, dt=7) == L.QAT_ERR_UNSUPPORTED
    assert _int(lib, scheme=5) == L.QAT_ERR_UNSUPPORTED
    assert _int(lib, rows=-1) == L.QAT_ERR_INVALID_ARGUMENT
    assert _int(lib, gran=9) == L.QAT_ERR_INVALID_ARGUMENT
    assert _int(lib, gran=L.PER_GROUP, group=0) == L.QAT_ERR_INVALID_ARGUMENT
    assert _int(lib, gran=L.PER_GROUP, group=48) == L.QAT_ERR_INVALID_ARGUMENT  # 48 does not divide 64
    assert _int(lib, x=None) == L.QAT_ERR_INVALID_ARGUMENT
    assert _int(lib, scale=None) == L.QAT_ERR_INVALID_ARGUMENT
    assert _int(lib, given=1, scheme=L.AFFINE, zp=None) == L.QAT_ERR_INVALID_ARGUMENT
    assert _int(lib, x=MIS) == L.QAT_ERR_MISALIGNED
    assert _int(lib, y=MIS) == L.QAT_ERR_MISALIGNED
    assert _int(lib, mask=ctypes.c_void_p(0x10004)) == L.QAT_ERR_MISALIGNED
    # per-tensor calibration needs the workspace
    assert _int(lib, ws=None) == L.QAT_ERR_WORKSPACE
    assert _int(lib, ws=A, wsb=100) == L.QAT_ERR_WORKSPACE
    # a unit length the fused kernels do not cover needs the fallback workspace
    assert _int(lib, gran=L.PER_ROW, cols=40, ws=None) == L.QAT_ERR_WORKSPACE
    # calibrated columns always take the column statistics workspace
    assert _int(lib, gran=L.PER_COLUMN, ws=None) == L.QAT_ERR_WORKSPACE
    need = lib.qat_workspace_bytes(4, 64, L.PER_COLUMN, 0)
    assert _int(lib, gran=L.PER_COLUMN, ws=A, wsb=need - 1) == L.QAT_ERR_WORKSPACE
    # empty tensors are a no-op even with NULL buffers
    assert _int(lib, rows=0, x=None, scale=None) == L.QAT_OK
    assert _int(lib, cols=0, x=None, scale=None) == L.QAT_OK


def test_fp8_argument_errors(lib):
    f = lib.qat_fake_quant_fp8
    assert f(A, L.F32, 100, 7, 0, A, A, None, None, None, None, 0, None) == L.QAT_ERR_UNSUPPORTED
    assert f(A, L.F32, -1, 0, 0, A, A, None, None, None, None, 0, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert f(A, L.F32, 0, 0, 0, None, None, None, None, None, None, 0, None) == L.QAT_OK
    assert f(A, L.F32, 100, 0, 0, A, None, None, None, None, None, 0, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert f(MIS, L.F32, 100, 0, 0, A, A, None, None, None, None, 0, None) == L.QAT_ERR_MISALIGNED
    assert f(A, L.F32, 100, 0, 0, A, A, None, None, None, None, 0, None) == L.QAT_ERR_WORKSPACE


def test_ste_and_q4_argument_errors(lib):
    assert lib.qat_ste_backward(A, L.F32, 10, None, A, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert lib.qat_ste_backward(A, 3, 10, A, A, None) == L.QAT_ERR_UNSUPPORTED
    assert lib.qat_ste_backward(MIS, L.F32, 10, A, A, None) == L.QAT_ERR_MISALIGNED
    assert lib.qat_ste_backward(None, L.F32, 0, None, None, None) == L.QAT_OK
    assert lib.qat_quant4_double(A, -5, A, A, A, None, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert lib.qat_quant4_double(A, 64, None, A, A, None, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert lib.qat_quant4_double(MIS, 64, A, A, A, None, None) == L.QAT_ERR_MISALIGNED
    assert lib.qat_quant4_double(A, 64, A, A, A, MIS, None) == L.QAT_ERR_MISALIGNED
    assert lib.qat_dequant4_double(A, A, A, 64, None, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert lib.qat_dequant4_double(A, A, A, 0, None, None) == L.QAT_OK


def test_stats_argument_errors(lib):
    f = lib.qat_amax_stats
    assert f(A, 9, 4, 4, L.PER_TENSOR, 0, None, None, None, None, A, 1 << 14, None) == L.QAT_ERR_UNSUPPORTED
    assert f(A, L.F32, 4, 4, L.PER_TENSOR, 0, None, None, None, None, None, 0, None) == L.QAT_ERR_WORKSPACE
    assert f(None, L.F32, 4, 4, L.PER_ROW, 0, None, None, None, None, None, 0, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert f(A, L.F32, 4, 6, L.PER_GROUP, 4, None, None, None, None, None, 0, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert f(MIS, L.F32, 4, 4, L.PER_ROW, 0, None, None, None, None, None, 0, None) == L.QAT_ERR_MISALIGNED
    assert f(A, L.F32, 4, 4, L.PER_COLUMN, 0, None, None, None, None, None, 0, None) == L.QAT_ERR_WORKSPACE
