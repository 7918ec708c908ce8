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
MIS = ctypes.c_void_p(0x10000 + 8)  # off the 32-byte grid (whole fp32 / bf16 elements)
ODD = ctypes.c_void_p(0x10000 + 1)  # inside an element of every dtype


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
    assert _int(lib, x=ODD) == L.QAT_ERR_MISALIGNED
    assert _int(lib, y=ODD) == L.QAT_ERR_MISALIGNED
    # whole elements off the vector grid are accepted (the element-per-lane
    # path); the missing workspace is then the error
    assert _int(lib, x=MIS, ws=None) == L.QAT_ERR_WORKSPACE
    assert _int(lib, y=MIS, ws=None) == L.QAT_ERR_WORKSPACE
    # per column they are not
    assert _int(lib, x=MIS, gran=L.PER_COLUMN, ws=A, wsb=1 << 20) == L.QAT_ERR_MISALIGNED
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
    assert f(ODD, L.F32, 100, 0, 0, A, A, None, None, None, None, 0, None) == L.QAT_ERR_MISALIGNED
    assert f(MIS, L.F32, 100, 0, 0, A, A, None, None, None, None, 0, None) == L.QAT_ERR_WORKSPACE
    assert f(A, L.F32, 100, 0, 0, A, A, None, None, None, None, 0, None) == L.QAT_ERR_WORKSPACE


def test_ste_and_q4_argument_errors(lib):
    assert lib.qat_ste_backward(A, L.F32, 10, None, A, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert lib.qat_ste_backward(A, 3, 10, A, A, None) == L.QAT_ERR_UNSUPPORTED
    assert lib.qat_ste_backward(ODD, L.F32, 10, A, A, None) == L.QAT_ERR_MISALIGNED
    assert lib.qat_ste_backward(A, L.BF16, 10, A, ODD, None) == L.QAT_ERR_MISALIGNED
    assert lib.qat_ste_backward(None, L.F32, 0, None, None, None) == L.QAT_OK
    assert lib.qat_quant4_double(A, -5, A, A, A, None, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert lib.qat_quant4_double(A, 64, None, A, A, None, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert lib.qat_quant4_double(ODD, 64, A, A, A, None, None) == L.QAT_ERR_MISALIGNED
    assert lib.qat_quant4_double(A, 64, A, A, A, ODD, None) == L.QAT_ERR_MISALIGNED
    assert lib.qat_quant4_double(A, 64, MIS, A, A, None, None) == L.QAT_ERR_MISALIGNED  # data: 16 B
    assert lib.qat_dequant4_double(A, A, A, 64, ODD, None) == L.QAT_ERR_MISALIGNED
    assert lib.qat_dequant4_double(A, A, A, 64, None, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert lib.qat_dequant4_double(A, A, A, 0, None, None) == L.QAT_OK


def test_stats_argument_errors(lib):
    f = lib.qat_amax_stats
    assert f(A, 9, 4, 4, L.PER_TENSOR, 0, None, None, None, None, A, 1 << 14, None) == L.QAT_ERR_UNSUPPORTED
    assert f(A, L.F32, 4, 4, L.PER_TENSOR, 0, None, None, None, None, None, 0, None) == L.QAT_ERR_WORKSPACE
    assert f(None, L.F32, 4, 4, L.PER_ROW, 0, None, None, None, None, None, 0, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert f(A, L.F32, 4, 6, L.PER_GROUP, 4, None, None, None, None, None, 0, None) == L.QAT_ERR_INVALID_ARGUMENT
    assert f(ODD, L.F32, 4, 4, L.PER_ROW, 0, None, None, None, None, None, 0, None) == L.QAT_ERR_MISALIGNED
    assert f(MIS, L.F32, 4, 4, L.PER_COLUMN, 0, None, None, None, None, A, 1 << 20, None) == \
        L.QAT_ERR_MISALIGNED
    assert f(A, L.F32, 4, 4, L.PER_COLUMN, 0, None, None, None, None, None, 0, None) == L.QAT_ERR_WORKSPACE


def _opts(lib, options, **kw):
    a = dict(x=A, dt=L.F32, rows=4, cols=64, bits=8, scheme=L.SYMMETRIC, gran=L.PER_TENSOR, group=0,
             sr=0, scale=A, zp=A, y=A, codes=A, mask=A, flags=None, ws=None, wsb=0)
    a.update(kw)
    return lib.qat_fake_quant_int_opts(a["x"], a["dt"], a["rows"], a["cols"], a["bits"],
                                       a["scheme"], a["gran"], a["group"], options, a["sr"], 1, 0,
                                       a["scale"], a["zp"], a["y"], a["codes"], a["mask"],
                                       a["flags"], a["ws"], a["wsb"], None)


def test_calibration_options_argument_errors(lib):
    for clip in (0.0, -0.5, 1.5, float("nan"), float("inf")):
        o = L.CalibOptions(clip, 0)
        assert _opts(lib, ctypes.addressof(o)) == L.QAT_ERR_INVALID_ARGUMENT, clip
    ok = L.CalibOptions(0.7, 1)
    # valid options, then the integer path's own checks
    assert _opts(lib, ctypes.addressof(ok), bits=3) == L.QAT_ERR_UNSUPPORTED
    assert _opts(lib, ctypes.addressof(ok), x=ODD) == L.QAT_ERR_MISALIGNED
    assert _opts(lib, ctypes.addressof(ok)) == L.QAT_ERR_WORKSPACE        # per tensor, no workspace
    assert _opts(lib, None, sr=1) == L.QAT_ERR_WORKSPACE                  # NULL options: plain
    assert _opts(lib, ctypes.addressof(ok), rows=0, x=None, scale=None) == L.QAT_OK
    f = lib.qat_fake_quant_int_sr
    assert f(A, L.F32, 4, 64, 5, 0, 0, 0, 0, A, A, 1, 0, A, A, A, None, None, 0, None) \
        == L.QAT_ERR_UNSUPPORTED
    assert f(A, L.F32, 4, 64, 8, 0, 0, 0, 0, A, A, 1, 0, A, A, A, None, None, 0, None) \
        == L.QAT_ERR_WORKSPACE


def _pct(lib, **kw):
    a = dict(x=A, dt=L.F32, n=1000, bits=8, scheme=L.SYMMETRIC, c=0.01, scale=A, zp=A, y=A, codes=A,
             mask=A, ws=A, wsb=lib.qat_percentile_workspace_bytes())
    a.update(kw)
    return lib.qat_fake_quant_int_percentile(a["x"], a["dt"], a["n"], a["bits"], a["scheme"],
                                             a["c"], 0, 0, 0, a["scale"], a["zp"], a["y"],
                                             a["codes"], a["mask"], None, a["ws"], a["wsb"], None)


def test_percentile_argument_errors(lib):
    assert lib.qat_percentile_workspace_bytes() >= 1024
    assert _pct(lib, bits=6) == L.QAT_ERR_UNSUPPORTED
    assert _pct(lib, dt=4) == L.QAT_ERR_UNSUPPORTED
    assert _pct(lib, scheme=2) == L.QAT_ERR_UNSUPPORTED
    # QuantParams::per_tensor_percentile takes a clip fraction in [0, 0.5)
    for c in (-0.01, 0.5, 0.75, float("nan")):
        assert _pct(lib, c=c) == L.QAT_ERR_INVALID_ARGUMENT, c
    assert _pct(lib, n=-1) == L.QAT_ERR_INVALID_ARGUMENT
    assert _pct(lib, n=(1 << 40) + 1) == L.QAT_ERR_INVALID_ARGUMENT
    assert _pct(lib, n=0, x=None, scale=None, ws=None) == L.QAT_OK
    assert _pct(lib, x=None) == L.QAT_ERR_INVALID_ARGUMENT
    assert _pct(lib, scale=None) == L.QAT_ERR_INVALID_ARGUMENT
    assert _pct(lib, x=MIS) == L.QAT_ERR_MISALIGNED
    assert _pct(lib, y=MIS) == L.QAT_ERR_MISALIGNED
    assert _pct(lib, codes=ctypes.c_void_p(0x10001)) == L.QAT_ERR_MISALIGNED
    assert _pct(lib, scale=ctypes.c_void_p(0x10002)) == L.QAT_ERR_MISALIGNED
    assert _pct(lib, ws=None) == L.QAT_ERR_WORKSPACE
    assert _pct(lib, wsb=lib.qat_percentile_workspace_bytes() - 1) == L.QAT_ERR_WORKSPACE
    assert _pct(lib, ws=MIS) == L.QAT_ERR_MISALIGNED


def _blk(lib, **kw):
    a = dict(x=A, dt=L.BF16, n=4096, elem=4, block=16, kind=1, ts=A, y=A, codes=A, bs=A, mask=A,
             ws=None, wsb=0)
    a.update(kw)
    return lib.qat_fake_quant_block(a["x"], a["dt"], a["n"], a["elem"], a["block"], a["kind"],
                                    a["ts"], a["y"], a["codes"], a["bs"], a["mask"], None, a["ws"],
                                    a["wsb"], None)


def test_block_scaled_argument_errors(lib):
    # element formats E4M3 .. E2M1 (0 .. 4), scales E8M0 / E4M3 / FP32 (0 .. 2)
    assert _blk(lib, dt=5) == L.QAT_ERR_UNSUPPORTED
    assert _blk(lib, elem=5) == L.QAT_ERR_UNSUPPORTED
    assert _blk(lib, elem=-1) == L.QAT_ERR_UNSUPPORTED
    assert _blk(lib, kind=3) == L.QAT_ERR_UNSUPPORTED
    for b in (8, 24, 64):
        assert _blk(lib, block=b) == L.QAT_ERR_UNSUPPORTED, b
    assert _blk(lib, n=-16) == L.QAT_ERR_INVALID_ARGUMENT
    assert _blk(lib, n=100) == L.QAT_ERR_INVALID_ARGUMENT          # not whole blocks of 16
    assert _blk(lib, n=48, block=32) == L.QAT_ERR_INVALID_ARGUMENT
    assert _blk(lib, n=0, x=None) == L.QAT_OK
    assert _blk(lib, x=None) == L.QAT_ERR_INVALID_ARGUMENT
    assert _blk(lib, x=MIS) == L.QAT_ERR_MISALIGNED
    assert _blk(lib, bs=ctypes.c_void_p(0x10002)) == L.QAT_ERR_MISALIGNED
    assert _blk(lib, ts=ctypes.c_void_p(0x10002)) == L.QAT_ERR_MISALIGNED
    # the E4M3 scale (NVFP4) needs the tensor statistics workspace
    assert _blk(lib, ws=None) == L.QAT_ERR_WORKSPACE
    assert _blk(lib, ws=A, wsb=15) == L.QAT_ERR_WORKSPACE
    assert _blk(lib, ws=MIS, wsb=1 << 20) == L.QAT_ERR_MISALIGNED


def test_a_failed_launch_is_reported_as_a_cuda_error(lib):
    """Failure detection on the host: on a machine without a usable CUDA
    device every launching call fails inside the CUDA runtime, and the library
    must return QAT_ERR_CUDA (after clearing the runtime's error) rather than
    crash or report success.  Skipped where a device exists, since the fake
    pointers would then reach a real launch."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("needs a host without a CUDA device")
    assert lib.qat_ste_backward(A, L.F32, 1024, A, A, None) == L.QAT_ERR_CUDA
    assert _int(lib, ws=A, wsb=16384) == L.QAT_ERR_CUDA
    assert lib.qat_fake_quant_fp8(A, L.F32, 1024, L.E4M3, 0, A, A, None, A, None, A, 16384,
                                  None) == L.QAT_ERR_CUDA
    assert lib.qat_quant4_double(A, 1024, A, A, A, None, None) == L.QAT_ERR_CUDA
    assert lib.qat_dequant4_double(A, A, A, 1024, A, None) == L.QAT_ERR_CUDA
    assert lib.qat_fake_quant_fp8_noalloc(A, L.F32, 1024, L.E4M3, 0, A, A, None, A, None,
                                          None) == L.QAT_ERR_CUDA
    # the status survives: the same call fails the same way again
    assert lib.qat_ste_backward(A, L.F32, 1024, A, A, None) == L.QAT_ERR_CUDA
