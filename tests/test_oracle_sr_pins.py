"""Pins for the oracle's stochastic rounding (the QAT module's
RoundingMode::Stochastic) and its counter-based draws (Philox-4x32-10).

The generator is checked against an independent library implementation
(triton's Philox, run by its CPU interpreter); the rounding against the
module's own stochastic tests (unbiasedness within 8 sigma over 400,000
draws, stability of exact grid values) and against exact counting over the
draw grid.  CPU only.
"""
import numpy as np
import pytest

F32 = np.float32


# ---------------------------------------------------------------------------
# the generator
# ---------------------------------------------------------------------------
_TRITON_PHILOX = r"""
import json, sys
import numpy as np
import torch
import triton
import triton.language as tl


@triton.jit
def philox_blocks(out_ptr, seed, base, N: tl.constexpr):
    idx = tl.arange(0, N)
    offs = idx.to(tl.uint64) + base
    a, b, c, d = tl.randint4x(seed, offs)
    tl.store(out_ptr + idx * 4 + 0, a)
    tl.store(out_ptr + idx * 4 + 1, b)
    tl.store(out_ptr + idx * 4 + 2, c)
    tl.store(out_ptr + idx * 4 + 3, d)


res = []
for seed, base in json.loads(sys.argv[1]):
    out = torch.zeros(16 * 4, dtype=torch.int32)
    philox_blocks[(1,)](out, seed, base, 16)
    res.append(out.numpy().view(np.uint32).tolist())
print(json.dumps(res))
"""


def test_philox_matches_triton_library(orc):
    """triton's Philox-4x32 (randint4x: counter (lo, hi of offset, 0, 0), key
    (lo, hi of seed), 10 rounds), run by triton's CPU interpreter in a child
    process, against the oracle's implementation."""
    pytest.importorskip("triton")
    import json
    import os
    import subprocess
    import sys

    rng = np.random.default_rng(5)
    cases = [(0, 0), (1, 0), (0x123456789, 5), ((1 << 63) - 1, (1 << 40) + 7)]
    cases += [(int(rng.integers(0, 1 << 62)), int(rng.integers(0, 1 << 50))) for _ in range(4)]
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, "-c", _TRITON_PHILOX, json.dumps(cases)], env=env,
                       capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + r.stderr.strip().splitlines()[-1])
    words = json.loads(r.stdout.strip().splitlines()[-1])
    for (seed, base), w in zip(cases, words):
        lib_words = np.array(w, np.uint32).reshape(16, 4)
        for k in range(16):
            j = base + k
            ours = orc.philox4x32_10([j & 0xFFFFFFFF, j >> 32, 0, 0],
                                     [seed & 0xFFFFFFFF, seed >> 32])
            assert np.array_equal(ours, lib_words[k]), (seed, j, ours, lib_words[k])


def test_draws_are_dyadic_and_follow_the_counter_layout(orc):
    seed, off = 0xDEADBEEF12345678, 1000
    u = orc.sr_uniform(seed, off, 64)
    k = u.astype(np.float64) * 2.0 ** 23
    assert np.all(k == np.floor(k)) and np.all((k >= 0) & (k < 2 ** 23))
    # element i draws word i % 4 of block offset + i // 4, bits 31..9
    for i in (0, 1, 2, 3, 4, 37, 63):
        j = off + i // 4
        w = orc.philox4x32_10([j & 0xFFFFFFFF, j >> 32, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert u[i] == F32((int(w[i % 4]) >> 9) * 2.0 ** -23)
    # shifting the offset by one block shifts the draws by four elements
    assert np.array_equal(orc.sr_uniform(seed, off + 1, 60), u[4:])


def test_draws_are_uniform(orc):
    u = orc.sr_uniform(99, 0, 40000)
    hist, _ = np.histogram(u, bins=20, range=(0.0, 1.0))
    expect = u.size / 20
    chi2 = float(((hist - expect) ** 2 / expect).sum())
    assert chi2 < 60.0  # 19 degrees of freedom; 60 is far beyond the 0.9999 quantile
    assert abs(float(u.mean()) - 0.5) < 6 * (1 / np.sqrt(12 * u.size))


# ---------------------------------------------------------------------------
# the rounding rule
# ---------------------------------------------------------------------------
def test_round_up_exactly_when_draw_below_fraction(orc):
    # r = 1 + m 2^-23 (exact in binary32): the draws k 2^-23 with k < m round
    # up, the others down, so over the whole draw grid the mean is r exactly
    for m in (1, 3, 1 << 20, (1 << 23) - 1):
        r = F32(1.0 + m * 2.0 ** -23)
        assert float(r) == 1.0 + m * 2.0 ** -23
        assert orc.sr_round(float(r), (m - 1) * 2.0 ** -23) == 2.0
        assert orc.sr_round(float(r), m * 2.0 ** -23) == 1.0
        assert orc.sr_round(float(r), 0.0) == 2.0
    # negative values round towards floor or floor + 1
    assert orc.sr_round(-2.25, 0.74) == -2.0 and orc.sr_round(-2.25, 0.75) == -3.0
    # integers never move; NaN stays NaN; infinities stay infinite
    for u in (0.0, 0.5, 1.0 - 2.0 ** -23):
        assert orc.sr_round(5.0, u) == 5.0 and orc.sr_round(-7.0, u) == -7.0
        assert np.isnan(orc.sr_round(float("nan"), u))
        assert orc.sr_round(float("inf"), u) == float("inf")


def test_int_stochastic_rounding_is_unbiased(orc):
    # the module's example: from_absmax(12.7) int8 gives scale 0.1, a value
    # 70% of the way from 3.0 to 3.1, 400,000 draws, mean within 8 sigma
    s, flag = orc.params_from_absmax(12.7, 127)
    assert flag == 0
    value = F32(F32(3.0) + F32(0.7) * F32(s))
    n = 400_000
    x = np.full(n, value, F32)
    r = orc.fake_quant_int_sr(x, 1, n, 8, 0, 0, seed=12345, offset=0, scale=[s])
    lower, upper = orc.dequantize(30, s, 0), orc.dequantize(31, s, 0)
    y = r["y"].astype(np.float64)
    assert np.all((y == lower) | (y == upper))
    assert (y == lower).any() and (y == upper).any()
    assert abs(y.mean() - float(value)) < 8 * s / np.sqrt(n)
    # codes are 30 or 31 and the STE window is that of nearest rounding
    assert set(np.unique(r["codes"])) == {30, 31}
    assert np.array_equal(r["mask"], orc.fake_quant_int(x, 1, n, 8, 0, 0, scale=[s])["mask"])


def test_int_stochastic_rounding_keeps_exact_grid_values(orc):
    # scale 0.125 (a power of two): 5 * 0.125 is exact, x / scale = 5 exactly
    x = np.full(1000, F32(0.625), F32)
    for scheme, zp in ((0, None), (1, [3])):
        r = orc.fake_quant_int_sr(x, 1, 1000, 8, scheme, 0, seed=99, offset=0, scale=[0.125],
                                  zero_point=zp)
        assert np.all(r["y"] == F32(0.625))
        assert np.all(r["codes"] == 5 + (zp[0] if zp else 0))


def test_int_stochastic_rounding_calibrated_and_clamped(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 256)).astype(F32)
    for bits in (8, 4):
        for scheme in (0, 1):
            ref = orc.fake_quant_int(x, 4, 256, bits, scheme, 1)
            r = orc.fake_quant_int_sr(x, 4, 256, bits, scheme, 1, seed=7, offset=11)
            # same calibration and window; every y on the unit's grid within one
            # step of the nearest-rounded value
            assert np.array_equal(r["scale"], ref["scale"])
            assert np.array_equal(r["zero_point"], ref["zero_point"])
            assert np.array_equal(r["mask"], ref["mask"])
            s = np.repeat(ref["scale"], 256).astype(np.float64)
            d = np.abs(r["y"].astype(np.float64) - ref["y"].astype(np.float64)) / s
            # (a y step equals s up to the binary32 rounding of y: < 2^-24 |y| / s)
            assert np.all((np.abs(d) < 2e-5) | (np.abs(d - 1.0) < 2e-5))
            # the element-wise rule with the element's own draw
            u = orc.sr_uniform(7, 11, x.size)
            qmin, qmax = orc.q_range(bits, scheme)
            for i in range(0, x.size, 37):
                row = i // 256
                q = orc.quantize_sr(float(x.flat[i]), float(ref["scale"][row]),
                                    int(ref["zero_point"][row]), qmin, qmax, float(u[i]))
                assert r["y"][i] == F32(orc.dequantize(q, float(ref["scale"][row]),
                                                       int(ref["zero_point"][row])))


def test_int_stochastic_rounding_offset_shift(orc):
    # the draws of a call depend only on (seed, offset + i // 4): a call on the
    # tail starting at element 4k with offset k reproduces the full call's tail
    rng = np.random.default_rng(8)
    x = rng.standard_normal(4096).astype(F32)
    full = orc.fake_quant_int_sr(x, 1, 4096, 4, 0, 0, seed=5, offset=0, scale=[0.3])
    tail = orc.fake_quant_int_sr(x[1024:], 1, 3072, 4, 0, 0, seed=5, offset=256, scale=[0.3])
    assert np.array_equal(full["y"][1024:], tail["y"])


# ---------------------------------------------------------------------------
# FP8
# ---------------------------------------------------------------------------
def test_fp8_stochastic_rounding_brackets_and_is_unbiased(orc):
    n = 400_000
    for fmt, t, lo, hi in ((0, 1.1, 1.0, 1.125), (1, 1.1, 1.0, 1.25),
                           (0, 2.0 ** -10, 0.0, 2.0 ** -9),       # E4M3 subnormal step
                           (0, -100.0, -104.0, -96.0)):
        x = np.full(n, F32(t), F32)
        r = orc.fake_quant_fp8_sr(x, fmt, seed=2024, offset=3, scale=1.0)
        y = r["y"].astype(np.float64)
        assert np.all((y == lo) | (y == hi)), (fmt, t)
        step = hi - lo
        assert abs(y.mean() - float(F32(t))) < 8 * step / np.sqrt(n), (fmt, t)
        assert np.all(r["mask"] == 0xFFFFFFFF)


def test_fp8_stochastic_rounding_fixed_points_and_specials(orc):
    x = np.array([1.125, -448.0, 460.0, 1e9, -np.inf, np.nan, -0.0, 0.0, 2.0 ** -9], F32)
    for seed in range(50):
        r = orc.fake_quant_fp8_sr(np.repeat(x, 4), 0, seed=seed, offset=0, scale=1.0)
        y = r["y"].reshape(-1, 4)
        assert np.all(y[0] == 1.125) and np.all(y[1] == -448.0)
        assert np.all(y[2] == 448.0) and np.all(y[3] == 448.0) and np.all(y[4] == -448.0)
        assert np.all(np.isnan(y[5]))
        assert np.all(np.signbit(y[6])) and np.all(y[6] == 0) and not np.any(np.signbit(y[7]))
        assert np.all(y[8] == 2.0 ** -9)
        codes = r["codes"].reshape(-1, 4)
        assert np.all(codes[5] == 0x7F) and np.all(codes[6] == 0x80)
