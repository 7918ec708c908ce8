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
