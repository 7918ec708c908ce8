"""Pins for the oracle's block-scaled formats (the teaching script's demo 4,
block_scaled, with the element formats of the OCP MX and NVFP4 definitions).

The element grids are decoded here from their bit fields, the rounding is
checked against a nearest-grid search and against the oracle's FP8 cast
(already pinned over every fp16 / bf16 pattern), the scales against the
page's stated properties, and the error orderings against demo 4's printed
observations.  CPU only.
"""
import numpy as np
import pytest

F32 = np.float32
# (ebits, mbits, bias, max) of E4M3, E5M2, E2M3, E3M2, E2M1
FIELDS = {0: (4, 3, 7, 448.0), 1: (5, 2, 15, 57344.0), 2: (2, 3, 1, 7.5), 3: (3, 2, 3, 28.0),
          4: (2, 1, 1, 6.0)}


def grid(fmt):
    """Every finite non-negative value of the format, from its fields."""
    eb, mb, bias, mx = FIELDS[fmt]
    vals = []
    for E in range(1 << eb):
        for M in range(1 << mb):
            v = (M / 2 ** mb) * 2.0 ** (1 - bias) if E == 0 else (1 + M / 2 ** mb) * 2.0 ** (E - bias)
            if v <= mx:
                vals.append((v, (E << mb) | M))
    return vals


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
def test_element_grid_decode_encode(orc, fmt):
    eb, mb, bias, mx = FIELDS[fmt]
    g = grid(fmt)
    assert max(v for v, _ in g) == mx
    for v, code in g:
        for sign in (0, 1):
            c = code | (sign << (eb + mb))
            val = -v if sign else v
            assert orc.elem_decode(np.array([c], np.uint8), fmt)[0] == F32(val)
            assert orc.elem_round(np.array([val], F32), fmt)[0] == F32(val)
            if v > 0:
                assert orc.elem_encode(np.array([val], F32), fmt)[0] == c


def test_fp4_grid_is_the_printed_e2m1(orc):
    assert [v for v, _ in grid(4)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
def test_element_rounding_is_nearest_even_saturating(orc, fmt):
    g = grid(fmt)
    vals = np.array([v for v, _ in g])
    codes = np.array([c for _, c in g])
    rng = np.random.default_rng(50 + fmt)
    mx = FIELDS[fmt][3]
    x = np.concatenate([rng.uniform(0, mx * 1.2, 4000), (vals[:-1] + vals[1:]) / 2]).astype(F32)
    got = orc.elem_round(x, fmt)
    for xi, gi in zip(x.astype(np.float64), got):
        if xi >= mx:
            assert gi == F32(mx)
            continue
        d = np.abs(vals - xi)
        best = np.flatnonzero(d == d.min())
        if best.size > 1:  # a tie: the even code (even mantissa)
            best = best[codes[best] % 2 == 0]
        assert gi == F32(vals[best[0]]), (xi, gi)
    assert np.array_equal(orc.elem_round(-x, fmt), -got)


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_elements_equal_the_fp8_cast(orc, fmt):
    rng = np.random.default_rng(60 + fmt)
    x = np.concatenate([rng.standard_normal(3000) * 10 ** rng.uniform(-6, 5, 3000)]).astype(F32)
    got = orc.elem_round(x, fmt)
    ref = np.array([orc.lib().or_fp8_cast(float(v), fmt) for v in x], F32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def student(n=1 << 20, seed=0):
    return (np.random.default_rng(seed).standard_t(5, size=n) * 0.02).astype(F32)


def rel(q, x):
    return np.linalg.norm(q.astype(np.float64) - x) / np.linalg.norm(x.astype(np.float64))


def test_e8m0_scales_put_the_block_max_in_the_top_binade(orc):
    """Demo 4: with power-of-two scales the block maximum divided by its
    scale lands in [2^emax, 2^(emax + 1)), e.g. [256, 512) for E4M3."""
    x = student(1 << 16, 1)
    for fmt in (0, 2, 3, 4):
        emax = int(np.floor(np.log2(FIELDS[fmt][3])))
        r = orc.fake_quant_block(x, fmt, 32, orc.SCALE_E8M0)
        X = np.ldexp(F32(1), r["bscales"].astype(np.int32) - 127)
        amax = np.abs(x.reshape(-1, 32)).max(axis=1)
        ratio = amax / X
        assert np.all((ratio >= 2.0 ** emax) & (ratio < 2.0 ** (emax + 1)))
        # y is code value times scale
        q = orc.elem_decode(r["codes"], fmt).reshape(-1, 32) * X[:, None]
        assert np.array_equal(q.reshape(-1), r["y"])


def test_nvfp4_scales(orc):
    x = student(1 << 16, 2)
    r = orc.fake_quant_block(x, 4, 16, orc.SCALE_E4M3)
    g = r["tensor_scale"]
    assert g == F32(np.abs(x).max() / F32(6.0 * 448.0))
    c = orc.elem_decode(r["bscales"], 0)
    assert np.all(c <= 448) and np.all(c >= 0)
    X = c * g
    q = orc.elem_decode(r["codes"], 4).reshape(-1, 16) * X[:, None]
    assert np.array_equal(q.reshape(-1).astype(F32), r["y"])
    # the exact scale: the block maximum maps to the element maximum
    e = orc.fake_quant_block(x, 4, 16, orc.SCALE_FP32)
    amax = np.abs(x.reshape(-1, 16)).max(axis=1)
    assert np.allclose(amax / e["bscales"], 6.0, rtol=2 ** -22)


def test_demo4_observations(orc):
    """The printed observations of demo 4 on Student-t(5) x 0.02, 2^20 values:
    for FP4 elements the E4M3 scale beats E8M0 and 16-blocks beat 32, the
    exact scale is close to E4M3; NVFP4 beats INT4 per 32 with FP16 scales;
    MXFP6 E2M3 beats E3M2."""
    x = student()
    e = {}
    for block in (32, 16):
        for kind in (0, 1, 2):
            e[(block, kind)] = rel(orc.fake_quant_block(x, 4, block, kind)["y"], x)
    assert e[(32, 0)] > e[(32, 1)] > e[(16, 1)]
    assert e[(16, 2)] <= e[(16, 1)] < 1.1 * e[(16, 2)]
    int4 = rel(orc.fake_quant_int_opts(x, 1, x.size, 4, 0, 2, 32, fp16=True)["y"], x)
    assert e[(16, 1)] < int4
    e23 = rel(orc.fake_quant_block(x, 2, 32, 0)["y"], x)
    e32 = rel(orc.fake_quant_block(x, 3, 32, 0)["y"], x)
    assert e23 < e32


def test_block_edges(orc):
    x = np.zeros(64, F32)
    x[32:] = student(32, 3)
    x[40] = np.nan
    x[41] = np.inf
    x[42] = -np.inf
    for kind in (0, 1, 2):
        r = orc.fake_quant_block(x, 4, 32, kind)
        assert np.all(r["y"][:32] == 0)
        assert np.isnan(r["y"][40]) and r["codes"][40] == 0
        assert r["y"][41] > 0 and r["y"][42] < 0 and r["codes"][41] == 0x7 and r["codes"][42] == 0xF
        assert r["flags"] & orc.FLAG_NONFINITE_INPUT
    assert orc.fake_quant_block(x, 4, 32, 0)["bscales"][0] == 127 - 2  # zero block: 2^-emax
    with pytest.raises(ValueError):
        orc.fake_quant_block(np.zeros(40, F32), 4, 32, 0)
