"""Pins for the CPU oracle: values, closed forms, invariants and brute force
that the sources fix, independent of the oracle's own code.

Every test here runs on the CPU (no GPU marker).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import golden_lines

FMT = {"E4M3": 0, "E5M2": 1}
SCHEME = {"sym": 0, "affine": 1}


# ---------------------------------------------------------------------------
# FP8: the format table, decoded from the field definitions in this file
# ---------------------------------------------------------------------------
def decode_fp8(code: int, fmt: str) -> float:
    """Value of an FP8 code from sign / exponent / mantissa fields."""
    eb, mb, bias = (4, 3, 7) if fmt == "E4M3" else (5, 2, 15)
    s = -1.0 if code & 0x80 else 1.0
    E = (code >> mb) & ((1 << eb) - 1)
    M = code & ((1 << mb) - 1)
    if fmt == "E4M3" and E == 15 and M == 7:
        return math.nan
    if fmt == "E5M2" and E == 31:
        return s * math.inf if M == 0 else math.nan
    if E == 0:
        return s * M * 2.0 ** (1 - bias - mb)
    return s * (1.0 + M / 2 ** mb) * 2.0 ** (E - bias)


def finite_grid(fmt):
    """Non-negative finite grid values in code order (codes 0x00..)."""
    vals, codes = [], []
    for c in range(0x80):
        v = decode_fp8(c, fmt)
        if math.isfinite(v):
            vals.append(v)
            codes.append(c)
    return np.array(vals), np.array(codes)


@pytest.mark.parametrize("row", golden_lines("fp8_format_table.txt"), ids=lambda r: r[0])
def test_fp8_format_table(row):
    fmt, _eb, mb, bias, mx, mn_norm, mn_sub, has_inf, nans = row
    vals = [decode_fp8(c, fmt) for c in range(256)]
    finite = [abs(v) for v in vals if math.isfinite(v)]
    assert max(finite) == float(mx)
    assert min(v for v in finite if v > 0) == float(mn_sub)
    assert 2.0 ** (1 - int(bias)) == float(mn_norm)
    assert 2.0 ** (1 - int(bias) - int(mb)) == float(mn_sub)
    assert any(math.isinf(v) for v in vals) == (has_inf == "yes")
    nan_codes = sorted(c for c in range(256) if math.isnan(vals[c]))
    assert nan_codes == sorted(int(t, 16) for t in nans.split(","))


@pytest.mark.parametrize("fmt", ["E4M3", "E5M2"])
def test_fp8_grid_points_are_fixed_points_and_encode(orc, fmt):
    for c in range(256):
        v = decode_fp8(c, fmt)
        if not math.isfinite(v):
            continue
        got = orc.fp8_cast(np.float32(v), FMT[fmt])
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (fmt, hex(c), v, got)
        assert orc.fp8_encode(np.float32(v), FMT[fmt]) == c, (fmt, hex(c))


@pytest.mark.parametrize("row", golden_lines("fp8_worked_values.txt"),
                         ids=lambda r: f"{r[0]}:{r[1]}")
def test_fp8_worked_values(orc, row):
    fmt, x, want = row[0], float(row[1]), float(row[2])
    got = orc.fp8_cast(np.float32(x), FMT[fmt])
    if math.isnan(want):
        assert math.isnan(got)
    else:
        assert got == want


def brute_force_fp8(a32: np.ndarray, fmt: str):
    """Nearest finite grid element, ties to the even code, saturating, sign kept.

    Returns (value as float64, code)."""
    grid, gcodes = finite_grid(fmt)
    with np.errstate(invalid="ignore"):
        a = a32.astype(np.float64)
    mag = np.abs(a)
    out = np.empty_like(a)
    code = np.zeros(a.shape, np.int64)
    fin = np.isfinite(a)
    i = np.clip(np.searchsorted(grid, mag[fin], side="left"), 1, len(grid) - 1)
    lo, hi = grid[i - 1], grid[i]
    dlo, dhi = mag[fin] - lo, hi - mag[fin]
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (gcodes[i] % 2 == 0))
    v = np.where(pick_hi, hi, lo)
    c = np.where(pick_hi, gcodes[i], gcodes[i - 1])
    big = mag[fin] >= grid[-1]
    v = np.where(big, grid[-1], v)
    c = np.where(big, gcodes[-1], c)
    neg = np.signbit(a[fin])
    out[fin] = np.where(neg, -v, v)
    code[fin] = np.where(neg, c | 0x80, c)
    inf = np.isinf(a)
    out[inf] = np.where(a[inf] > 0, grid[-1], -grid[-1])
    code[inf] = np.where(a[inf] > 0, gcodes[-1], gcodes[-1] | 0x80)
    nan = np.isnan(a)
    out[nan] = np.nan
    code[nan] = 0x7F
    return out, code


def _check_against_brute(orc, xs_f32, fmt, x_for_oracle):
    res = orc.fake_quant_fp8(x_for_oracle, FMT[fmt], scale=1.0)
    want, wcode = brute_force_fp8(xs_f32, fmt)
    got = (res["y"].astype(np.float64) if res["y"].dtype == np.float32
           else torch.from_numpy(res["y"].view(np.int16)).view(torch.bfloat16).double().numpy())
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    assert np.array_equal(res["codes"].astype(np.int64), wcode)


@pytest.mark.parametrize("fmt", ["E4M3", "E5M2"])
def test_fp8_cast_all_fp16_inputs_brute_force(orc, fmt):
    """All 2^16 fp16 bit patterns (exact in fp32) against nearest-grid brute force."""
    xs = np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float32)
    _check_against_brute(orc, xs, fmt, xs)


@pytest.mark.parametrize("fmt", ["E4M3", "E5M2"])
def test_fp8_cast_all_bf16_inputs_brute_force(orc, fmt):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    xs = (bits.astype(np.uint32) << 16).view(np.float32)
    _check_against_brute(orc, xs, fmt, bits)


@pytest.mark.parametrize("fmt", ["E4M3", "E5M2"])
def test_fp8_cast_random_fp32_brute_force(orc, fmt):
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    xs = bits.view(np.float32)
    _check_against_brute(orc, xs, fmt, xs)


@pytest.mark.parametrize("fmt", ["E4M3", "E5M2"])
def test_fp8_exact_ties_round_to_even_in_every_binade(orc, fmt):
    grid, gcodes = finite_grid(fmt)
    for k in range(len(grid) - 1):
        mid = (grid[k] + grid[k + 1]) / 2
        want = grid[k] if gcodes[k] % 2 == 0 else grid[k + 1]
        for sgn in (1.0, -1.0):
            got = orc.fp8_cast(np.float32(sgn * mid), FMT[fmt])
            assert got == sgn * want, (fmt, mid, got)
    # past the top: the tie between max and the next binade point saturates
    top = {"E4M3": (464.0, 448.0), "E5M2": (61440.0, 57344.0)}[fmt]
    assert orc.fp8_cast(np.float32(top[0]), FMT[fmt]) == top[1]


def test_fp8_negative_underflow_keeps_sign(orc):
    got = orc.fp8_cast(np.float32(-1e-30), 0)
    assert got == 0.0 and math.copysign(1, got) < 0
    assert orc.fp8_encode(np.float32(-0.0), 0) == 0x80


# ---------------------------------------------------------------------------
# integer grids
# ---------------------------------------------------------------------------
def test_int_ranges_and_widths(orc):
    for row in golden_lines("int_worked_values.txt"):
        if row[0] == "q_range":
            assert orc.q_range(int(row[1]), SCHEME[row[2]]) == (int(row[3]), int(row[4]))
        elif row[0] == "unsupported":
            with pytest.raises(ValueError):
                orc.q_range(int(row[1]), 0)


def test_int_from_absmax_worked_values(orc):
    for row in golden_lines("int_worked_values.txt"):
        if row[0] != "absmax":
            continue
        absmax, bits, want, tol = float(row[1]), int(row[2]), float(row[3]), float(row[4])
        _, qmax = orc.q_range(bits, 0)
        s, flag = orc.params_from_absmax(np.float32(absmax), qmax)
        assert flag == 0
        assert abs(s - want) <= max(tol, 0.0) + 1e-12 * want


def test_int8_grid_values_map_to_themselves(orc):
    s, _ = orc.params_from_absmax(np.float32(12.7), 127)
    for k in range(-120, 121):
        x = np.float32(np.float32(k) * np.float32(s))
        q = orc.quantize(x, s, 0, -127, 127)
        assert q == k
        assert orc.dequantize(q, s, 0) == x


def test_int4_round_trip_on_grid(orc):
    s, _ = orc.params_from_absmax(np.float32(7.0), 7)
    assert s == 1.0
    for k in range(-7, 8):
        assert orc.dequantize(orc.quantize(float(k), s, 0, -7, 7), s, 0) == k


def test_affine_grid_values_map_to_themselves(orc):
    data = np.array([-0.3, 1.7, 0.0, 0.9, -0.1], np.float32)
    r = orc.fake_quant_int(data, 1, 5, 8, 1, 0)
    s, z = float(r["scale"][0]), int(r["zero_point"][0])
    # scale = (1.7 - (-0.3)) / 255 in fp32; zero point = rne(-128 + 0.3 / scale) = -90
    assert s == np.float32(np.float32(np.float32(1.7) - np.float32(-0.3)) / np.float32(255))
    assert z == -90
    for q in range(-128, 128):
        g = orc.dequantize(q, s, z)
        assert orc.quantize(g, s, z, -128, 127) == q


def test_affine_zero_maps_to_zero_point_and_zero_output(orc):
    rng = np.random.default_rng(5)
    for _ in range(50):
        x = (rng.standard_normal(33) * rng.uniform(0.01, 5) + rng.uniform(-3, 3)).astype(np.float32)
        x[7] = 0.0
        for bits in (8, 4):
            r = orc.fake_quant_int(x, 1, 33, bits, 1, 0)
            z = int(r["zero_point"][0])
            codes = r["codes"] if bits == 8 else None
            if codes is not None:
                assert codes[7] == z
            assert r["y"][7] == 0.0 and not np.signbit(r["y"][7])


def test_int8_error_bounded_by_half_scale(orc):
    s, _ = orc.params_from_absmax(np.float32(2.0), 127)
    xs = np.float32(-1.9) + np.float32(0.013) * np.arange(0, 293, dtype=np.float32)
    for x in xs:
        y = orc.dequantize(orc.quantize(x, s, 0, -127, 127), s, 0)
        assert abs(float(y) - float(x)) <= s / 2 + 1e-7


def test_error_bound_and_grid_membership_random(orc):
    """|y - x| <= scale/2 inside the window; every y is an integer multiple of scale."""
    rng = np.random.default_rng(3)
    for scheme in (0, 1):
        for bits in (8, 4):
            x = (rng.standard_normal(4096) * 0.7 + (0.3 if scheme else 0)).astype(np.float32)
            r = orc.fake_quant_int(x, 64, 64, bits, scheme, 1)
            y = r["y"].reshape(64, 64).astype(np.float64)
            s = r["scale"].astype(np.float64)[:, None]
            k = y / s
            assert np.all(np.abs(k - np.round(k)) < 1e-3)
            bits_mask = np.unpackbits(r["mask"].view(np.uint8), bitorder="little")[:4096].reshape(64, 64)
            inside = bits_mask.astype(bool)
            err = np.abs(y - x.reshape(64, 64))
            assert np.all(err[inside] <= (s / 2 * (1 + 1e-6) + 1e-12).repeat(64, 1)[inside])


def test_idempotent(orc):
    rng = np.random.default_rng(4)
    x = rng.standard_normal(1000).astype(np.float32)
    for scheme in (0, 1):
        for bits in (8, 4):
            r1 = orc.fake_quant_int(x, 1, 1000, bits, scheme, 0)
            r2 = orc.fake_quant_int(r1["y"], 1, 1000, bits, scheme, 0, scale=r1["scale"],
                                    zero_point=r1["zero_point"])
            assert np.array_equal(r1["y"], r2["y"])


def test_per_channel_worked_example(orc):
    x = np.array([[0.0, 0.5, 1.0], [0.0, 50.0, 100.0]], np.float32)
    r = orc.fake_quant_int(x, 2, 3, 8, 0, 1)
    assert abs(r["scale"][0] - 1 / 127) < 1e-6 and abs(r["scale"][1] - 100 / 127) < 1e-6
    assert r["scale"][1] > 10 * r["scale"][0]
    err = np.abs(r["y"].reshape(2, 3) - x)
    assert np.all(err <= r["scale"][:, None] / 2 + 1e-9)


@pytest.mark.parametrize("scheme,bits", [(0, 8), (1, 8), (0, 4), (1, 4)])
def test_units_equal_independent_slices(orc, scheme, bits):
    """Each row / group is calibrated from its own slice only: per-row (per-group)
    results equal the per-tensor results of each row (group) taken alone."""
    rng = np.random.default_rng(9)
    rows, cols, group = 6, 96, 32
    x = (rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-3, 1, (rows, 1)))).astype(np.float32)
    for gran, L in ((1, cols), (2, group)):
        r = orc.fake_quant_int(x, rows, cols, bits, scheme, gran, group)
        flat = x.reshape(-1)
        for u in range(rows * cols // L):
            one = orc.fake_quant_int(flat[u * L:(u + 1) * L].copy(), 1, L, bits, scheme, 0)
            assert r["scale"][u] == one["scale"][0]
            assert r["zero_point"][u] == one["zero_point"][0]
            assert np.array_equal(r["y"][u * L:(u + 1) * L], one["y"])


def test_brute_force_codes_tiny_inputs_power_of_two_scale(orc):
    """With a power-of-two scale x/scale is exact; the code must be the integer
    nearest to x/scale with ties to even, clamped to the window (checked with
    exact rationals), and the zero point is added after rounding."""
    # symmetric int8: absmax = 127/8 -> scale = 1/8 exactly
    s, _ = orc.params_from_absmax(np.float32(127 / 8), 127)
    assert s == 0.125
    # affine int8: [min, max] = [-3.0625, 12.875] -> range 255/16, scale 1/16, zp = -79 (odd)
    sa, za, flag = orc.params_affine(np.float32(-3.0625), np.float32(12.875), -128, 127)
    assert flag == 0 and sa == 0.0625 and za == -79
    for scale, zp, qmin, qmax in ((0.125, 0, -127, 127), (0.0625, -79, -128, 127)):
        for kk in range(-300, 300):
            for frac in (Fraction(0), Fraction(1, 2), Fraction(1, 4), Fraction(3, 4)):
                xr = (kk + frac) * Fraction(scale)
                x = np.float32(float(xr))
                assert Fraction(float(x)) == xr
                # brute force over every code
                best = None
                for q in range(qmin, qmax + 1):
                    d = abs(xr - (q - zp) * Fraction(scale))
                    key = (d, (q - zp) % 2)
                    if best is None or key < best[0]:
                        best = (key, q)
                assert orc.quantize(x, scale, zp, qmin, qmax) == best[1], (float(xr), scale, zp)


def test_code_form_differs_only_at_ties_with_odd_zero_point(orc):
    """The module's code adds zp before rounding; with an odd zp that moves exact
    ties to the other neighbour.  The documented form is taken (see the oracle)."""
    scale, zp = 0.0625, -79
    diffs = 0
    for kk in range(-40, 40):
        x = np.float32((kk + 0.5) * scale)
        a = orc.quantize(x, scale, zp, -128, 127, True)
        b = orc.quantize(x, scale, zp, -128, 127, False)
        if a != b:
            diffs += 1
            assert abs(a - b) == 1
        assert orc.quantize(np.float32(kk * scale + 0.01), scale, zp, -128, 127, True) == \
            orc.quantize(np.float32(kk * scale + 0.01), scale, zp, -128, 127, False)
    assert diffs > 0


def test_degenerate_and_nonfinite_flags(orc):
    z = np.zeros(3, np.float32)
    for scheme in (0, 1):
        r = orc.fake_quant_int(z, 1, 3, 8, scheme, 0)
        assert r["flags"] & orc.FLAG_DEGENERATE
        assert np.all(r["y"] == 0) and np.all(r["mask"] == 0) and np.all(r["codes"] == 0)
    x = np.array([1.0, np.nan, 2.0], np.float32)
    r = orc.fake_quant_int(x, 1, 3, 8, 0, 0)
    assert r["flags"] == orc.FLAG_NONFINITE
    # given params: NaN -> code 0, +-inf -> clamp ends, mask 0 for all three
    x = np.array([np.nan, np.inf, -np.inf, 0.5], np.float32)
    r = orc.fake_quant_int(x, 1, 4, 8, 1, 0, scale=np.array([0.01], np.float32),
                           zero_point=np.array([3], np.int32))
    assert list(r["codes"]) == [0, 127, -128, 53]
    assert r["mask"][0] == 0b1000


def test_ste_worked_example(orc):
    rows = {r[0]: [float(v) for v in r[1:]] for r in golden_lines("ste_example.txt")}
    x = np.array(rows["x"], np.float32)
    g = np.array(rows["grad"], np.float32)
    # window [-1, 1]: int8 symmetric with scale 1/127 has real_max = 127 * fl(1/127) = 1 in fp32
    s = np.float32(np.float32(1.0) / np.float32(127.0))
    assert np.float32(127.0) * s == np.float32(1.0)
    r = orc.fake_quant_int(x, 1, 5, 8, 0, 0, scale=np.array([s]), zero_point=np.array([0]))
    dx = orc.ste_backward(g, r["mask"])
    assert list(dx) == rows["expected"]


def test_ste_is_bit_copy_and_positive_zero(orc):
    rng = np.random.default_rng(2)
    g = rng.standard_normal(100).astype(np.float32)
    g[3] = -0.0
    mask = rng.integers(0, 1 << 32, size=4, dtype=np.uint64).astype(np.uint32)
    dx = orc.ste_backward(g, mask)
    bits = np.unpackbits(mask.view(np.uint8), bitorder="little")[:100].astype(bool)
    assert np.array_equal(dx.view(np.uint32)[bits], g.view(np.uint32)[bits])
    assert np.all(dx.view(np.uint32)[~bits] == 0)


def test_bf16_output_rounding_matches_torch(orc):
    rng = np.random.default_rng(8)
    x = torch.from_numpy(rng.standard_normal(4096).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    rb = orc.fake_quant_int(xb, 1, 4096, 8, 0, 0)
    rf = orc.fake_quant_int(x.float().numpy(), 1, 4096, 8, 0, 0)
    assert rb["scale"][0] == rf["scale"][0]
    want = torch.from_numpy(rf["y"]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(rb["y"], want)


def test_stats_match_numpy(orc):
    rng = np.random.default_rng(12)
    x = rng.standard_normal((8, 100)).astype(np.float32)
    x[2, 5] = np.nan
    x[3, 7] = np.inf
    r = orc.fake_quant_int(x, 8, 100, 8, 1, 1)
    for row in range(8):
        v = x[row][np.isfinite(x[row])]
        rmin, rmax = min(v.min(), 0.0), max(v.max(), 0.0)
        if row in (2, 3):
            assert r["flags"] & orc.FLAG_NONFINITE
            continue
        assert r["scale"][row] == np.float32(np.float32(rmax - rmin) / np.float32(255))


def test_o64_agrees_with_o32_within_tolerance(orc):
    from tolerance import int_check

    rng = np.random.default_rng(13)
    x = (rng.standard_normal((16, 256)) * 0.5 + 0.1).astype(np.float32)
    for scheme, bits in ((0, 8), (1, 8), (0, 4), (1, 4)):
        r32 = orc.fake_quant_int(x, 16, 256, bits, scheme, 1)
        r64 = orc.fake_quant_int_f64(x, 16, 256, bits, scheme, 1)
        ok, nt = int_check(r32["y"].reshape(16, 256).astype(np.float64), r64["y"].reshape(16, 256),
                           x.astype(np.float64), r64["scale"][:, None], False)
        assert ok and nt <= 2


# ---------------------------------------------------------------------------
# two-level 4-bit (double quant)
# ---------------------------------------------------------------------------
def decode_nibbles(data: np.ndarray, n: int) -> np.ndarray:
    """Even element -> high nibble, odd -> low nibble, two's complement."""
    hi = (data >> 4) & 0xF
    lo = data & 0xF
    nib = np.empty(2 * data.size, np.int64)
    nib[0::2], nib[1::2] = hi, lo
    nib = nib[:n]
    return np.where(nib >= 8, nib - 16, nib)


def test_q4_nibble_order_and_codes(orc):
    x = np.array([7.0, 1.0, -7.0, 2.0, -3.0], np.float32)  # absmax 7 -> scale 1
    r = orc.quant4_double(x)
    assert list(r["data"]) == [0x71, 0x92, 0xD0]
    assert list(decode_nibbles(r["data"], 5)) == [7, 1, -7, 2, -3]


def test_q4_exact_ties_round_half_away_from_zero(orc):
    # absmax 7 -> scale exactly 1, so every x below is its own quotient; the
    # block code rounds like Rust's f32::round (half away from zero), unlike
    # the integer grid's ties-to-even
    x = np.array([7.0, 2.5, -2.5, 0.5, -0.5, 6.5, -6.5, 1.5], np.float32)
    r = orc.quant4_double(x)
    assert list(decode_nibbles(r["data"], 8)) == [7, 3, -3, 1, -1, 7, -7, 2]


def test_q4_accounting(orc):
    rows = {r[0]: r[1:] for r in golden_lines("double_quant_accounting.txt")}
    n = 1 << 28
    dbits = orc.q4d_memory_bytes(n) * 8 / n
    want, tol = map(float, rows["double_bits_per_param"])
    assert abs(dbits - want) <= tol
    single = (n // 2 + 4 * (n // 64)) * 8 / n
    assert single == float(rows["single_bits_per_param"][0])
    sav = single - dbits
    want, tol = map(float, rows["savings_bits_per_param_nominal"])
    assert abs(sav - want) <= tol
    n2 = 65536
    sav2 = (4 * (n2 // 64) - (n2 // 64 + 4 * ((n2 // 64 + 255) // 256))) * 8 / n2
    assert sav2 > float(rows["savings_bits_per_param_min"][0])
    m, nb, ns = map(int, rows["small_input"])
    r = orc.quant4_double(np.array([1.0, -2.0, 3.0, -4.0], np.float32))
    assert r["qscales"].size == nb and r["super_scales"].size == ns
    assert orc.dequant4_double(r["data"], r["qscales"], r["super_scales"], m).size == m


def test_q4_super_is_max_scale_and_maps_to_255(orc):
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(64 * 700) * 0.02).astype(np.float32)
    r = orc.quant4_double(x)
    single = orc.quant4_single(x)
    sc = single["scales"]
    for sb in range(r["super_scales"].size):
        blk = sc[sb * 256:(sb + 1) * 256]
        assert r["super_scales"][sb] == blk.max()
        assert r["qscales"][sb * 256 + int(np.argmax(blk))] == 255
        rs = np.array([orc.reconstruct_scale(int(q), float(r["super_scales"][sb]))
                       for q in r["qscales"][sb * 256:(sb + 1) * 256]])
        bound = r["super_scales"][sb] / 510 + 4 * np.spacing(np.float32(r["super_scales"][sb]))
        assert np.all(np.abs(rs - blk) <= bound)
    assert np.array_equal(single["data"], r["data"])


def test_q4_zeros(orc):
    r = orc.quant4_double(np.zeros(128, np.float32), roundtrip=True)
    assert np.all(r["y"] == 0) and not np.any(np.signbit(r["y"]))
    assert r["super_scales"][0] == np.float32(1e-8)


def test_q4_double_within_1pct_of_single_sin(orc):
    vals = (np.sin(np.arange(4096, dtype=np.float32) * np.float32(0.1)) * np.float32(2.0)).astype(np.float32)
    s = orc.quant4_single(vals)
    sd = orc.dequant4_single(s["data"], s["scales"], 4096)
    d = orc.quant4_double(vals, roundtrip=True)["y"]
    assert np.all(np.abs(sd - d) <= np.abs(sd) * 0.01 + 1e-6)


def test_q4_scale_reconstruction_within_1pct(orc):
    vals = (np.sin(np.arange(4096, dtype=np.float32) * np.float32(0.05)) * np.float32(5.0)).astype(np.float32)
    s = orc.quant4_single(vals)["scales"]
    r = orc.quant4_double(vals)
    rec = np.array([orc.reconstruct_scale(int(q), float(r["super_scales"][i // 256]))
                    for i, q in enumerate(r["qscales"])])
    assert np.all(np.abs(s - rec) <= np.abs(s) * 0.01 + 1e-8)


def test_q4_property_cases(orc):
    rng = np.random.default_rng(22)
    for _ in range(100):
        n = int(rng.integers(64, 1024))
        n -= n % 64
        mag = float(rng.uniform(0.1, 10.0))
        vals = (np.sin(np.arange(n, dtype=np.float32) * np.float32(0.1)) * np.float32(mag)).astype(np.float32)
        s = orc.quant4_single(vals)
        sd = orc.dequant4_single(s["data"], s["scales"], n)
        d = orc.quant4_double(vals, roundtrip=True)["y"]
        assert d.size == n
        assert np.all(np.abs(sd - d) <= np.abs(sd) * 0.01 + 1e-5)
    for n in rng.integers(1, 2048, size=40):
        r = orc.quant4_double(np.arange(n, dtype=np.float32) * np.float32(0.1), roundtrip=True)
        assert r["y"].size == n
    for n in (64 * 257, 64 * 300, 8128):
        nb = (n + 63) // 64
        single = (n + 1) // 2 + 4 * nb
        assert orc.q4d_memory_bytes(n) < single or nb <= 256


def test_q4_tail_blocks_and_odd_length(orc):
    rng = np.random.default_rng(23)
    for n in (1, 2, 63, 65, 127, 16383, 16385, 64 * 256 + 1):
        x = rng.standard_normal(n).astype(np.float32)
        r = orc.quant4_double(x, roundtrip=True)
        assert r["data"].size == (n + 1) // 2
        if n % 2:
            assert r["data"][-1] & 0x0F == 0
        # each block's absmax element reconstructs within the scale error
        codes = decode_nibbles(r["data"], n)
        assert np.all((codes >= -8) & (codes <= 7))
        y2 = orc.dequant4_double(r["data"], r["qscales"], r["super_scales"], n)
        assert np.array_equal(y2, r["y"])
