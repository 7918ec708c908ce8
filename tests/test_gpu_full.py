"""GPU parity at the five workloads' full sizes, in the calls the benchmark
times: every output element against the oracle (bit patterns), plus the
tolerance check against the binary64 evaluation of the same formulas.
"""
import numpy as np
import pytest
import torch

from fake_quant_numerics_gb300 import workloads as W
from gpu_helpers import assert_same, bits, oracle_input
from tolerance import int_check

pytestmark = pytest.mark.gpu


def _int_full(qat, orc, x, rows, cols, bits_, scheme, gran, group=0, grad=None, f64=True):
    r = qat.fake_quant_int(x.cuda(), bits=bits_, scheme=scheme, granularity=gran, group=group)
    dx = qat.fake_quant_backward(grad.cuda(), r.mask) if grad is not None else None
    torch.cuda.synchronize()
    xo = oracle_input(x)
    o = orc.fake_quant_int(xo, rows, cols, bits_, {"symmetric": 0, "affine": 1}[scheme],
                           {"tensor": 0, "row": 1, "group": 2}[gran], group)
    tag = f"{x.dtype} {rows}x{cols} int{bits_} {scheme} {gran}"
    gy = bits(r.y)
    assert_same(gy, o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"], "y " + tag)
    assert_same(bits(r.codes), o["codes"].view(np.uint8), "codes " + tag)
    assert_same(bits(r.mask), o["mask"], "mask " + tag)
    assert_same(bits(r.scale), o["scale"].view(np.uint32), "scale " + tag)
    assert int(r.flags.item()) == o["flags"] == 0
    if dx is not None:
        assert_same(bits(dx), orc.ste_backward(oracle_input(grad), o["mask"]), "dx " + tag)
    if f64:
        o64 = orc.fake_quant_int_f64(xo, rows, cols, bits_, {"symmetric": 0, "affine": 1}[scheme],
                                     {"tensor": 0, "row": 1, "group": 2}[gran], group)
        L = rows * cols if gran == "tensor" else (cols if gran == "row" else group)
        yv = r.y.float().cpu().numpy().reshape(-1, L).astype(np.float64)
        xv = x.float().numpy().reshape(-1, L).astype(np.float64)
        ok, ties = int_check(yv, o64["y"].reshape(-1, L), xv, o64["scale"][:, None],
                             x.dtype == torch.bfloat16)
        assert ok, tag
        assert ties <= max(8, x.numel() // 100), (tag, ties)


def test_workload1_per_tensor_int8_fwd_bwd(qat, orc):
    x, g = W.cfg1()
    _int_full(qat, orc, x, 1, x.numel(), 8, "symmetric", "tensor", grad=g)


def test_workload2_per_row_affine_int8_and_sym_int4(qat, orc):
    w = W.cfg2()
    _int_full(qat, orc, w, 4096, 4096, 8, "affine", "row")
    _int_full(qat, orc, w, 4096, 4096, 4, "symmetric", "row")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_workload3_fp8_per_tensor(qat, orc, fmt):
    a = W.cfg3()
    r = qat.fake_quant_fp8(a.cuda(), fmt, want_codes=True)
    torch.cuda.synchronize()
    f = {"e4m3": 0, "e5m2": 1}[fmt]
    xo = oracle_input(a)
    o = orc.fake_quant_fp8(xo, f)
    assert_same(bits(r.y), o["y"], "fp8 y")
    assert_same(bits(r.codes), o["codes"], "fp8 codes")
    assert_same(bits(r.mask), o["mask"], "fp8 mask")
    assert bits(r.scale)[0] == np.float32(o["scale"]).view(np.uint32)
    assert int(r.flags.item()) == o["flags"] == 8  # the workload holds NaN / Inf
    # binary64 evaluation: the same grid point, or a neighbour where fp32 and
    # f64 quotients straddle a rounding boundary; bf16 output rounding on top
    o64 = orc.fake_quant_fp8_f64(xo, f)
    y = r.y.float().cpu().numpy().astype(np.float64).reshape(-1)
    fin = np.isfinite(o64["y"])
    assert np.array_equal(np.isnan(y), np.isnan(o64["y"]))
    s = o64["scale"]
    mb = 3 if f == 0 else 2
    step = np.where(np.abs(o64["y"]) > 0,
                    2.0 ** (np.floor(np.log2(np.maximum(np.abs(o64["y"]) / s, 2.0 ** -20))) - mb), 0)
    tol = (step + 2.0 ** -9) * s * 1.01 + np.abs(o64["y"]) * 2.0 ** -8
    d = np.abs(y[fin] - o64["y"][fin])
    assert np.all(d <= tol[fin])
    exact = np.mean(d <= np.abs(o64["y"][fin]) * 2.0 ** -8)
    assert exact > 0.999


def test_workload4_per_group_int4_fwd_bwd(qat, orc):
    w, g = W.cfg4()
    _int_full(qat, orc, w, 14336, 4096, 4, "symmetric", "group", 128, grad=g)


def test_workload5_double_quant_round_trip(qat, orc):
    x = W.cfg5()
    dq = qat.quantize_4bit_double(x.cuda())
    y = qat.dequantize_4bit_double(dq)
    torch.cuda.synchronize()
    o = orc.quant4_double(x.numpy(), roundtrip=True)
    assert_same(bits(dq.data), o["data"], "data")
    assert_same(bits(dq.quantized_scales), o["qscales"], "qscales")
    assert_same(bits(dq.super_scales), o["super_scales"].view(np.uint32), "super scales")
    assert_same(bits(y), o["y"].view(np.uint32), "y")
    n = x.numel()
    assert dq.memory_bytes() == orc.q4d_memory_bytes(n)
    assert abs(dq.memory_bytes() * 8 / n - 4.127) < 1e-3
