"""The workspace-free FP8 entry point, for callers that cannot allocate
device memory (a host framework that owns every allocation, or a loop that
must not call cudaMalloc).  Its scratch is a fixed device array inside the
library, shared by every call, so this test makes two different calls in a
row and checks both against the regular entry point (which takes a
caller-supplied workspace), bit for bit.

Kept in a file of its own that sorts last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _outputs(n, dtype):
    return (torch.empty(n, dtype=dtype, device="cuda"), torch.empty(n, dtype=torch.uint8, device="cuda"),
            torch.empty((n + 31) // 32, dtype=torch.int32, device="cuda"),
            torch.zeros(1, dtype=torch.float32, device="cuda"),
            torch.zeros(1, dtype=torch.int32, device="cuda"))


def _bits(t):
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()


def test_fp8_noalloc_matches_workspace_entry_point_twice():
    from fake_quant_numerics_gb300 import _lib
    from fake_quant_numerics_gb300 import workloads as W

    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    big = W.cfg3(rows=2048, cols=4096, seed=21).cuda()  # holds 1e6 outliers and NaN / Inf
    small = (torch.randn(100_003, device="cuda") * 1e-3).float()  # fewer blocks, smaller amax
    for x, fmt in ((big, _lib.E4M3), (small, _lib.E5M2), (big, _lib.E5M2), (small, _lib.E4M3)):
        n = x.numel()
        dt = _lib.BF16 if x.dtype == torch.bfloat16 else _lib.F32
        ref = _outputs(n, x.dtype)
        ws = torch.empty(lib.qat_workspace_bytes(1, n, _lib.PER_TENSOR, 0), dtype=torch.uint8,
                         device="cuda")
        st = lib.qat_fake_quant_fp8(_p(x), dt, n, fmt, 0, _p(ref[3]), _p(ref[0]), _p(ref[1]),
                                    _p(ref[2]), _p(ref[4]), _p(ws), ws.numel(), stream)
        assert st == _lib.QAT_OK
        got = _outputs(n, x.dtype)
        st = lib.qat_fake_quant_fp8_noalloc(_p(x), dt, n, fmt, 0, _p(got[3]), _p(got[0]),
                                            _p(got[1]), _p(got[2]), _p(got[4]), stream)
        assert st == _lib.QAT_OK
        torch.cuda.synchronize()
        for a, b, name in zip(ref, got, ("y", "codes", "mask", "scale", "flags")):
            assert np.array_equal(_bits(a), _bits(b)), f"{name} differs (fmt {fmt}, n {n})"


def test_fp8_noalloc_given_scale_and_ragged_tail():
    """The caller-scale branch (no statistics pass, so no scratch) and a size
    smaller than one tile, each bit for bit against the workspace entry point."""
    from fake_quant_numerics_gb300 import _lib

    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    g = torch.Generator().manual_seed(5)
    for n, dtype, given in ((33, torch.float32, 0), (33, torch.bfloat16, 0),
                            (70_001, torch.float32, 1), (33, torch.bfloat16, 1)):
        x = (torch.randn(n, generator=g) * 3.0).to(dtype).cuda()
        dt = _lib.BF16 if dtype == torch.bfloat16 else _lib.F32
        ref, got = _outputs(n, dtype), _outputs(n, dtype)
        if given:
            ref[3].fill_(0.013)
            got[3].fill_(0.013)
        ws = torch.empty(lib.qat_workspace_bytes(1, n, _lib.PER_TENSOR, 0), dtype=torch.uint8,
                         device="cuda")
        assert lib.qat_fake_quant_fp8(_p(x), dt, n, _lib.E4M3, given, _p(ref[3]), _p(ref[0]),
                                      _p(ref[1]), _p(ref[2]), _p(ref[4]), _p(ws), ws.numel(),
                                      stream) == _lib.QAT_OK
        assert lib.qat_fake_quant_fp8_noalloc(_p(x), dt, n, _lib.E4M3, given, _p(got[3]),
                                              _p(got[0]), _p(got[1]), _p(got[2]), _p(got[4]),
                                              stream) == _lib.QAT_OK
        torch.cuda.synchronize()
        for a, b, name in zip(ref, got, ("y", "codes", "mask", "scale", "flags")):
            assert np.array_equal(_bits(a), _bits(b)), f"{name} differs (n {n}, given {given})"


def test_fp8_noalloc_argument_errors_before_any_launch():
    """Argument errors come back as status codes before anything runs: a
    pointer not aligned to its element, an unknown format, a negative size;
    n = 0 is a no-op that touches nothing."""
    from fake_quant_numerics_gb300 import _lib

    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    x = torch.zeros(256, device="cuda")
    y, codes, mask, scale, flags = _outputs(256, torch.float32)
    raw = ctypes.c_void_p(x.data_ptr() + 1)  # inside an fp32 element
    c0 = lib.qat_kernel_launch_count()
    args = (_p(scale), _p(y), _p(codes), _p(mask), _p(flags), stream)
    assert lib.qat_fake_quant_fp8_noalloc(raw, _lib.F32, 64, _lib.E4M3, 0, *args) == \
        _lib.QAT_ERR_MISALIGNED
    assert lib.qat_fake_quant_fp8_noalloc(_p(x), _lib.F32, 64, 7, 0, *args) == \
        _lib.QAT_ERR_UNSUPPORTED
    assert lib.qat_fake_quant_fp8_noalloc(_p(x), _lib.F32, -1, _lib.E4M3, 0, *args) == \
        _lib.QAT_ERR_INVALID_ARGUMENT
    y.fill_(7.0)
    assert lib.qat_fake_quant_fp8_noalloc(_p(x), _lib.F32, 0, _lib.E4M3, 0, *args) == _lib.QAT_OK
    torch.cuda.synchronize()
    assert lib.qat_kernel_launch_count() == c0
    assert bool((y == 7.0).all())
