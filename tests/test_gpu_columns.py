"""GPU parity of per-column integer fake quant (one scale / zero point per
column of a row-major [rows, cols] tensor) against the oracle: y, codes, mask,
scale, zero point and flags bit for bit, calibrated and with given
parameters, nearest and stochastic rounding, and the per-column statistics.

Shapes cover both device paths: the column-strip kernels (cols a multiple of
32: whole strips, a partial strip, many row chunks) and the per-element unit
kernel (any other row length, including rows that are not 16-byte aligned).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import Poisoned, assert_same, bits, oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
COL = 3
STRIP_SHAPES = [(64, 128), (333, 96), (1000, 4096), (5, 160), (1, 256), (3000, 32), (17, 1024)]
OTHER_SHAPES = [(7, 33), (100, 40), (64, 1), (9, 100), (2, 4), (50, 7), (1, 1)]


def column_input(rows, cols, dtype, seed, special_cols=False):
    """Columns with their own spread and offset; zeros of both signs; with
    special_cols, an all-zero column, a column holding NaN, one holding -Inf,
    a constant column and columns of tiny and huge magnitude (their scales
    fall outside the reciprocal's safe range)."""
    rng = np.random.default_rng(seed)
    sig = np.exp(rng.uniform(np.log(0.01), np.log(3.0), size=(1, cols))).astype(np.float32)
    off = rng.uniform(-0.3, 0.3, size=(1, cols)).astype(np.float32)
    a = rng.standard_normal((rows, cols)).astype(np.float32) * sig + off
    flat = a.reshape(-1)
    if flat.size:
        flat[rng.integers(0, flat.size, size=max(1, flat.size // 97))] = 0.0
        flat[rng.integers(0, flat.size, size=max(1, flat.size // 211))] = -0.0
    if special_cols and cols >= 8:
        a[:, 0] = 0.0
        a[rows // 2, 1] = np.nan
        a[rows // 3, 2] = -np.inf
        a[:, 3] = 0.75
        a[:, 4] *= np.float32(1e-30)
        a[:, 5] *= np.float32(1e36)
    t = torch.from_numpy(a)
    return t.to(dtype) if dtype != torch.float32 else t


def run_cols(qat, orc, x, rows, cols, bits_, scheme, scale=None, zp=None, sr=None):
    dev = "cuda"
    n = rows * cols
    xd = x.to(dev).contiguous()
    y = Poisoned(n, x.dtype)
    codes = Poisoned(n if bits_ == 8 else (n + 1) // 2, torch.int8 if bits_ == 8 else torch.uint8)
    mask = Poisoned((n + 31) // 32, torch.int32)
    given = scale is not None
    if given:
        sc = torch.tensor(np.asarray(scale, np.float32), device=dev)
        zpt = torch.tensor(np.asarray(zp, np.int32), device=dev) if zp is not None else None
    else:
        scp, zpp = Poisoned(cols, torch.float32), Poisoned(cols, torch.int32)
        sc, zpt = scp.t, zpp.t
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(max(qat.qat_workspace_bytes(rows, cols, COL, 0), 16), dtype=torch.uint8,
                     device=dev)
    ws.fill_(0xA5)  # scratch contents on entry must not matter
    if sr is None:
        qat.qat_fake_quant_int(xd, rows, cols, bits_, scheme, COL, 0, given, sc, zpt, y.t, codes.t,
                               mask.t, flags, ws)
        o = orc.fake_quant_int(oracle_input(x), rows, cols, bits_, scheme, COL, 0, scale=scale,
                               zero_point=zp)
    else:
        seed, offset = sr
        qat.qat_fake_quant_int_sr(xd, rows, cols, bits_, scheme, COL, 0, given, sc, zpt, seed,
                                  offset, y.t, codes.t, mask.t, flags, ws)
        o = orc.fake_quant_int_sr(oracle_input(x), rows, cols, bits_, scheme, COL, 0, seed=seed,
                                  offset=offset, scale=scale, zero_point=zp)
    torch.cuda.synchronize()
    for b, name in ((y, "y"), (codes, "codes"), (mask, "mask")):
        assert b.canary_ok(), f"write past the end of {name}"
    tag = f"{x.dtype} bits={bits_} scheme={scheme} cols ({rows},{cols}) given={given} sr={sr}"
    yo = o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"]
    assert_same(bits(y.t), yo, "y " + tag)
    assert_same(bits(codes.t), o["codes"].view(np.uint8), "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    if not given:
        assert scp.canary_ok() and zpp.canary_ok()
        assert_same(bits(sc), o["scale"].view(np.uint32), "scale " + tag)
        if scheme == 1:
            assert_same(zpt.cpu().numpy(), o["zero_point"], "zero point " + tag)
    assert int(flags.item()) == o["flags"], f"flags {tag}: {int(flags.item())} vs {o['flags']}"
    return o


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("scheme", [0, 1])
def test_columns_calibrated(qat, orc, dt, bits_, scheme):
    for i, (r, c) in enumerate(STRIP_SHAPES + OTHER_SHAPES):
        x = column_input(r, c, DT[dt], seed=1300 + i)
        run_cols(qat, orc, x, r, c, bits_, scheme)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_columns_special_columns(qat, orc, dt, scheme):
    """Dead columns (zero, NaN, Inf), a constant column and scales outside the
    reciprocal's safe range, on both device paths."""
    for bits_ in (8, 4):
        for i, (r, c) in enumerate([(40, 64), (300, 256), (33, 40), (12, 100)]):
            x = column_input(r, c, DT[dt], seed=1400 + i, special_cols=True)
            o = run_cols(qat, orc, x, r, c, bits_, scheme)
            assert o["flags"] & orc.FLAG_NONFINITE


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_columns_given_params(qat, orc, dt, scheme):
    rng = np.random.default_rng(1500)
    for bits_ in (8, 4):
        for r, c in ((50, 64), (9, 33)):
            x = column_input(r, c, DT[dt], seed=1501, special_cols=True)
            sc = rng.uniform(0.001, 0.05, size=c).astype(np.float32)
            zp = rng.integers(-5, 5, size=c).astype(np.int32)
            sc[6] = 0.0
            sc[7] = -1.0
            sc[1] = np.inf
            if scheme:
                zp[2] = 500
            o = run_cols(qat, orc, x, r, c, bits_, scheme, scale=sc, zp=zp if scheme else None)
            assert o["flags"] & orc.FLAG_BAD_PARAMS


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("scheme", [0, 1])
def test_columns_stochastic(qat, orc, dt, bits_, scheme):
    for i, (r, c) in enumerate([(64, 128), (333, 96), (5, 160), (7, 33), (50, 7)]):
        x = column_input(r, c, DT[dt], seed=1600 + i, special_cols=(i == 0))
        for sr in ((0, 0), (0x9E3779B97F4A7C15, 12345), (7, (1 << 40) - 3)):
            run_cols(qat, orc, x, r, c, bits_, scheme, sr=sr)
    x = column_input(20, 64, DT[dt], seed=1610)
    sc = np.random.default_rng(1611).uniform(0.001, 0.05, size=64).astype(np.float32)
    run_cols(qat, orc, x, 20, 64, bits_, scheme, scale=sc, zp=np.zeros(64, np.int32) if scheme
             else None, sr=(5, 77))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_columns_full_size(qat, orc, dt):
    """The measured workload's shape, [4096, 4096], every output compared."""
    x = column_input(4096, 4096, DT[dt], seed=1700)
    for scheme, bits_ in ((1, 8), (0, 4)):
        run_cols(qat, orc, x, 4096, 4096, bits_, scheme)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_columns_amax_stats(qat, orc, dt):
    for i, (r, c) in enumerate(STRIP_SHAPES[:4] + OTHER_SHAPES):
        x = column_input(r, c, DT[dt], seed=1800 + i, special_cols=True)
        a, mn, mx = (Poisoned(c, torch.float32) for _ in range(3))
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.empty(max(qat.qat_workspace_bytes(r, c, COL, 0), 16), dtype=torch.uint8,
                         device="cuda")
        qat.qat_amax_stats(x.cuda(), r, c, COL, 0, a.t, mn.t, mx.t, flags, ws)
        torch.cuda.synchronize()
        omn, omx, oa, bad = orc.column_stats(oracle_input(x), r, c)
        tag = f"column stats {dt} ({r},{c})"
        assert_same(bits(mn.t), omn.copy().view(np.uint32), "min " + tag)
        assert_same(bits(mx.t), omx.copy().view(np.uint32), "max " + tag)
        assert_same(bits(a.t), oa.copy().view(np.uint32), "absmax " + tag)
        assert int(flags.item()) == (8 if bad.sum() else 0), tag
        assert a.canary_ok() and mn.canary_ok() and mx.canary_ok()


def test_columns_named_op(qat, orc):
    """fake_quant_int(granularity="column") over a 3-d tensor: the columns are
    the last dimension."""
    import fake_quant_numerics_gb300 as fq
    x = column_input(6 * 50, 192, torch.float32, seed=1900).reshape(6, 50, 192)
    r = fq.fake_quant_int(x.cuda(), 8, "affine", "column")
    o = orc.fake_quant_int(x.numpy().reshape(-1), 300, 192, 8, 1, COL)
    assert_same(bits(r.y).reshape(-1), o["y"].view(np.uint32), "named op y")
    assert_same(bits(r.scale), o["scale"].view(np.uint32), "named op scale")
    assert r.scale.numel() == 192 and r.zero_point.numel() == 192


def test_affine_calibrated_without_zero_point_array(qat, orc):
    """The zero-point array is optional for calibrated units: the unit-kernel
    fallback then keeps the zero points in the workspace (per row and per
    column)."""
    for gran, r, c in ((1, 4, 40), (3, 7, 33), (3, 64, 128)):
        x = column_input(r, c, torch.float32, seed=1950 + c)
        n = r * c
        units = orc.n_units(r, c, gran, 0)
        y = torch.empty(n, dtype=torch.float32, device="cuda")
        sc = torch.empty(units, dtype=torch.float32, device="cuda")
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.empty(qat.qat_workspace_bytes(r, c, gran, 0), dtype=torch.uint8, device="cuda")
        qat.qat_fake_quant_int(x.cuda(), r, c, 8, 1, gran, 0, False, sc, None, y, None, None, flags,
                               ws)
        torch.cuda.synchronize()
        o = orc.fake_quant_int(x.numpy().reshape(-1), r, c, 8, 1, gran, 0)
        assert_same(bits(y), o["y"].view(np.uint32), f"y gran={gran} ({r},{c})")
        assert_same(bits(sc), o["scale"].view(np.uint32), f"scale gran={gran} ({r},{c})")
