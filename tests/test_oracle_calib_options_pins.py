"""Pins for the oracle's calibration options: the clip factor (the range
c * max|x| of the teaching script's demo 2), binary16 scales (the FP16 group
scales of its demo 3) and percentile calibration (the QAT module's
per_tensor_percentile: nearest-rank quantiles, then from_minmax).

The binary16 rounding is checked against numpy's float16 conversion, the
quantiles against numpy's quantile with the 'lower' / 'higher' methods and
against a sort of order keys, the clipped and fp16 maps against the oracle's
given-parameter path, and the page's own worked cases (the module's
percentile test, demo 2's U-shaped error).  CPU only.
"""
import numpy as np
import pytest

F32 = np.float32


def keys(x):
    """Order keys of float32 values (total order, -0 < +0)."""
    u = np.ascontiguousarray(x, F32).view(np.uint32)
    return np.where(u >> 31, ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def test_round_fp16_matches_numpy(orc):
    rng = np.random.default_rng(40)
    parts = [
        rng.standard_normal(20000).astype(F32),
        (rng.random(20000) * 2e-4).astype(F32),            # binary16 subnormals and small normals
        (rng.random(5000) * 40 + 65490).astype(F32),       # the top binade and the overflow edge
        np.exp(rng.uniform(-30, 12, 20000)).astype(F32),   # far below and above the range
    ]
    # exact midpoints between neighbouring binary16 values (ties to even)
    h = np.arange(0, 0x7C00, 97, dtype=np.uint16).view(np.float16).astype(np.float64)
    nxt = (np.arange(0, 0x7C00, 97, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    parts.append(((h + nxt) / 2).astype(F32))
    x = np.concatenate(parts)
    x = np.concatenate([x, -x, np.array([0.0, -0.0, 65504, 65519.99, 65520, np.inf, -np.inf], F32)])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(F32)
    got = orc.round_fp16(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_clip_one_and_no_fp16_is_the_plain_calibration(orc):
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((6, 512)) * 0.3 + 0.1).astype(F32).reshape(-1)
    for gran, g in ((0, 0), (1, 0), (2, 128), (3, 0)):
        for bits, scheme in ((8, 0), (8, 1), (4, 0), (4, 1)):
            a = orc.fake_quant_int_opts(x, 6, 512, bits, scheme, gran, g)
            b = orc.fake_quant_int(x, 6, 512, bits, scheme, gran, g)
            for k in ("y", "codes", "mask", "scale", "zero_point"):
                assert np.array_equal(a[k], b[k]), (gran, bits, scheme, k)


@pytest.mark.parametrize("scheme", [0, 1])
def test_power_of_two_clip_scales_exactly(orc, scheme):
    """c = 2^-k scales the range exactly, so the scale is c times the plain
    one and the zero point is unchanged."""
    rng = np.random.default_rng(42)
    x = (rng.standard_t(4, size=4 * 1024) * 0.2 + 0.05).astype(F32)
    plain = orc.fake_quant_int_opts(x, 4, 1024, 8, scheme, 1)
    for c in (0.5, 0.25, 0.125):
        r = orc.fake_quant_int_opts(x, 4, 1024, 8, scheme, 1, clip=c)
        assert np.array_equal(r["scale"], plain["scale"] * F32(c))
        assert np.array_equal(r["zero_point"], plain["zero_point"])


@pytest.mark.parametrize("scheme", [0, 1])
@pytest.mark.parametrize("fp16", [False, True])
def test_clipped_and_fp16_maps_equal_the_given_parameter_path(orc, scheme, fp16):
    """Calibration with options, then the map: the same elements as the
    given-parameter path with the scales it chose (elements beyond the clipped
    range take the end codes)."""
    rng = np.random.default_rng(43)
    x = (rng.standard_t(3, size=8 * 256) * 0.5).astype(F32)
    for bits in (8, 4):
        for c in (1.0, 0.7, 0.3):
            r = orc.fake_quant_int_opts(x, 8, 256, bits, scheme, 2, 64, clip=c, fp16=fp16)
            g = orc.fake_quant_int(x, 8, 256, bits, scheme, 2, 64, scale=r["scale"],
                                   zero_point=r["zero_point"] if scheme else None)
            for k in ("y", "codes", "mask"):
                assert np.array_equal(r[k], g[k]), (bits, c, k)
            if fp16:
                # the scales are binary16 values: numpy's float16 of the plain scales
                plain = orc.fake_quant_int_opts(x, 8, 256, bits, scheme, 2, 64, clip=c)
                if scheme == 0:
                    assert np.array_equal(r["scale"], plain["scale"].astype(np.float16).astype(F32))
                assert np.array_equal(r["scale"].astype(np.float16).astype(F32), r["scale"])
            if c < 1.0:
                # the clipped range: some elements sit at the end codes
                qmax = 127 if bits == 8 else 7
                codes = r["codes"].astype(np.int32) if bits == 8 else None
                if codes is not None:
                    assert np.any(np.abs(codes) >= qmax - (1 if scheme else 0))


def test_demo2_clipping_error_is_u_shaped(orc):
    """The teaching script's demo 2: symmetric int4 per tensor with the range
    c * max|x|; for heavy tails the best c lies below 1, and too small a c is
    worse again (the U-shaped trade of rounding against clipping error)."""
    rng = np.random.default_rng(0)
    n = 1 << 18
    cs = (1.0, 0.8, 0.6, 0.5, 0.4, 0.3, 0.25, 0.2, 0.15, 0.1, 0.07, 0.05)
    for name, z in (("laplace", rng.laplace(size=n)), ("student-t5", rng.standard_t(5, n))):
        z = z.astype(F32)
        errs = []
        for c in cs:
            y = orc.fake_quant_int_opts(z, 1, n, 4, 0, 0, clip=c)["y"].astype(np.float64)
            errs.append(np.linalg.norm(y - z) / np.linalg.norm(z))
        best = int(np.argmin(errs))
        assert cs[best] < 1.0 and errs[best] < errs[0], name
        assert errs[-1] > errs[best], name


def test_percentile_module_example(orc):
    """The module's percentile_calibration_clips_outliers: 0.00 .. 0.99 and an
    outlier 1000, clip fraction 0.02: last = 100, the quantile indexes are 2
    and 98, so the symmetric scale is 0.98 / 127 (binary32), below the plain
    absmax scale."""
    data = np.concatenate([np.arange(100) / 100.0, [1000.0]]).astype(F32)
    r = orc.fake_quant_int_percentile(data, 8, 0, 0.02)
    plain = orc.fake_quant_int(data, 1, data.size, 8, 0, 0)
    assert r["flags"] == 0
    assert r["scale"][0] == F32(F32(0.98) / F32(127))
    assert r["scale"][0] < plain["scale"][0]
    lo, hi, _ = orc.percentile_minmax(data, 0.02)
    assert lo == F32(0.02) and hi == F32(0.98)


def test_percentile_quantiles_match_numpy(orc):
    rng = np.random.default_rng(44)
    for n in (1, 2, 3, 10, 101, 1000, 4097):
        x = rng.standard_normal(n).astype(F32)
        x[x == 0] = F32(0.5)
        for c in (0.0, 0.001, 0.02, 0.1, 0.25, 0.4999):
            lo, hi, fl = orc.percentile_minmax(x, c)
            assert fl == 0
            x64 = x.astype(np.float64)
            assert lo == np.quantile(x64, c, method="lower"), (n, c)
            assert hi == np.quantile(x64, 1.0 - c, method="higher"), (n, c)


def test_percentile_orders_signed_zeros(orc):
    """The total order puts -0 before +0: a tensor of zeros of both signs
    picks by the sorted order keys."""
    x = np.array([0.0, -0.0, 0.0, -0.0, -0.0, 1.0, -1.0], F32)
    srt = np.sort(keys(x))
    last = x.size - 1
    for c in (0.0, 0.2, 0.3, 0.45):
        lo, hi, _ = orc.percentile_minmax(x, c)
        lo_i = int(np.floor(c * last))
        hi_i = min(int(np.ceil((1.0 - c) * last)), last)
        assert keys(np.array([lo], F32))[0] == srt[lo_i], c
        assert keys(np.array([hi], F32))[0] == srt[hi_i], c


def test_percentile_zero_fraction_is_the_plain_calibration(orc):
    rng = np.random.default_rng(45)
    x = (rng.standard_normal(5000) * 0.4 - 0.1).astype(F32)
    for bits, scheme in ((8, 0), (8, 1), (4, 0), (4, 1)):
        a = orc.fake_quant_int_percentile(x, bits, scheme, 0.0)
        b = orc.fake_quant_int(x, 1, x.size, bits, scheme, 0)
        for k in ("y", "codes", "mask", "scale", "zero_point"):
            assert np.array_equal(a[k], b[k]), (bits, scheme, k)


def test_percentile_map_and_errors(orc):
    rng = np.random.default_rng(46)
    x = rng.standard_t(2, size=3000).astype(F32)
    for bits, scheme in ((8, 0), (8, 1), (4, 0), (4, 1)):
        for sr in (False, True):
            r = orc.fake_quant_int_percentile(x, bits, scheme, 0.01, stochastic=sr, seed=9,
                                              offset=3)
            if sr:
                g = orc.fake_quant_int_sr(x, 1, x.size, bits, scheme, 0, seed=9, offset=3,
                                          scale=r["scale"],
                                          zero_point=r["zero_point"] if scheme else None)
            else:
                g = orc.fake_quant_int(x, 1, x.size, bits, scheme, 0, scale=r["scale"],
                                       zero_point=r["zero_point"] if scheme else None)
            for k in ("y", "codes", "mask"):
                assert np.array_equal(r[k], g[k]), (bits, scheme, sr, k)
    bad = x.copy()
    bad[17] = np.nan
    r = orc.fake_quant_int_percentile(bad, 8, 0, 0.01)
    assert r["flags"] & orc.FLAG_NONFINITE and not np.any(r["y"]) and not np.any(r["mask"])
    for c in (-0.1, 0.5, 0.7, float("nan")):
        with pytest.raises(ValueError):
            orc.fake_quant_int_percentile(x, 8, 0, c)


@pytest.mark.parametrize("scheme", [0, 1])
def test_overflowing_quotient_takes_the_end_code(orc, scheme):
    """QuantParams::quantize clamps the rounded quotient to [qmin, qmax], so an
    element far beyond a clipped range takes the end code of its sign, even
    when x / scale overflows binary32 (1e30 against a scale near 8e-10), with
    mask 0; the values inside the range keep their own codes."""
    x = np.array([1e30, -1e30, 3e29, -2e20, 0.0, 1e-10, -5e-10], F32)
    r = orc.fake_quant_int_opts(x, 1, x.size, 8, scheme, 0, clip=1e-37)
    s = r["scale"][0]
    if scheme == 0:
        assert s == F32(F32(F32(1e-37) * F32(1e30)) / F32(127))
    codes = r["codes"].view(np.int8).astype(np.int32)
    zp = int(r["zero_point"][0]) if scheme else 0
    qmin, qmax = (-127, 127) if scheme == 0 else (-128, 127)
    assert list(codes[:4]) == [qmax, qmin, qmax, qmin]
    assert r["mask"][0] & 0b1111 == 0
    # elements inside the window round to nearest: |y - x| <= scale / 2
    for i in (4, 5, 6):
        assert codes[i] - zp == int(np.rint(np.float64(x[i]) / np.float64(s)))
    y = r["y"]
    assert y[0] == F32(qmax - zp) * s and y[1] == F32(qmin - zp) * s
