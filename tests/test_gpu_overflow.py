"""GPU parity where a quotient x / s overflows binary32.

QuantParams::quantize rounds the real quotient and then clamps it to
[qmin, qmax], so an element far beyond a clipped, rounded or percentile range
takes the end code of its sign, whatever its size (the oracle's IEEE quotient
is then +-inf and clamps the same way).  These cases put elements at every
magnitude from 2^-30 to past 2^128 times the unit's scale, so that the
reciprocal path's quotient crosses 2^22 (where rint by the magic constant is
no longer exact) and overflow, in every granularity, both schemes, both
roundings, fp32 and bf16; every output is compared bit for bit."""
import numpy as np
import pytest
import torch

from test_gpu_calib_options import run_opts
from test_gpu_percentile import run_pct

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
# (granularity, rows, cols, group): per tensor; groups of 128 / 32 (lanes of
# a warp); rows of 4096 (a block per row) and of 40 (the per-unit fallback);
# columns, staged (cols % 32 == 0) and not
CASES = [(0, 3, 1025, 0), (2, 6, 512, 128), (2, 4, 96, 32), (1, 5, 4096, 0), (1, 4, 40, 0),
         (3, 200, 256, 0), (3, 9, 33, 0)]
BIG = 1e30


def spread(rows, cols, seed, dtype, big=BIG):
    """Values +-m * big * 2^-k, k uniform in [0, 160], m in [1, 2); every
    unit holds +big (first row, every 32nd column), so a unit's absmax is about
    big and its scale (with a clip c) about c * big / qmax."""
    rng = np.random.default_rng(seed)
    k = rng.integers(0, 161, size=(rows, cols)).astype(np.float64)
    m = rng.uniform(1.0, 2.0, size=(rows, cols))
    sgn = rng.choice([-1.0, 1.0], size=(rows, cols))
    a = (sgn * m * big * 2.0 ** (-k)).astype(np.float32)
    a[:, ::32] = np.float32(big)
    a[0, :] = np.float32(big)
    a[rows // 2, cols // 2] = np.float32(-big)
    t = torch.from_numpy(a)
    return t.to(dtype) if dtype != torch.float32 else t


# clip 1e-37 puts the scale near 2^-30 (inside the reciprocal's safe range)
# and the quotient of BIG near 2^130; 2^-60 gives quotients up to about 2^67,
# finite but far past 2^22; 1e-3 stays well inside binary32
CLIPS = (1e-37, 2.0 ** -60, 1e-3)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_clip_overflow_every_path(qat, orc, dt, scheme):
    for i, (gran, r, c, g) in enumerate(CASES):
        x = spread(r, c, 4000 + i, DT[dt])
        for bits_ in (8, 4):
            for clip in CLIPS:
                run_opts(qat, orc, x, r, c, bits_, scheme, gran, g, clip, False)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_clip_overflow_with_fp16_scales(qat, orc, dt, scheme):
    """A binary16 scale after the clip.  A binary16 scale is at least 2^-24,
    so only values near binary32's top can overflow the quotient: with
    big = 1e38 a clip of 1e-40 (a binary32 subnormal) gives a scale near 8e-5
    and quotients up to about 2^141; 1e-36 a scale near 0.8 and quotients just
    below overflow."""
    for i, (gran, r, c, g) in enumerate(CASES):
        x = spread(r, c, 4100 + i, DT[dt], big=1e38)
        for bits_ in (8, 4):
            for clip in (1e-40, 1e-36):
                run_opts(qat, orc, x, r, c, bits_, scheme, gran, g, clip, True)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_clip_overflow_stochastic(qat, orc, dt, scheme):
    for i, (gran, r, c, g) in enumerate(CASES):
        x = spread(r, c, 4200 + i, DT[dt])
        for clip in (1e-37, 2.0 ** -60):
            run_opts(qat, orc, x, r, c, 8 if i % 2 else 4, scheme, gran, g, clip, False,
                     sr=(0xC0FFEE, 9))


def tiny_bulk_with_outliers(n, seed):
    """Bulk ~ 1e-20 N(0, 1); 0.05% of the elements are outliers +-1e-20 2^k
    with k up to 170 (about 1.5e31), beyond the 0.001 / 0.999 quantiles."""
    rng = np.random.default_rng(seed)
    a = (rng.standard_normal(n) * 1e-20).astype(np.float32)
    idx = rng.choice(n, size=max(4, n // 2000), replace=False)
    k = rng.integers(20, 171, size=idx.size).astype(np.float64)
    sgn = rng.choice([-1.0, 1.0], size=idx.size)
    a[idx] = (sgn * 1e-20 * 2.0 ** k).astype(np.float32)
    a[idx[0]] = np.float32(1e30)
    a[idx[1]] = np.float32(-1e30)
    return a


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_percentile_outliers_overflow(qat, orc, dt, scheme):
    for j, n in enumerate((4097, 200_000, (1 << 20) + 13)):
        t = torch.from_numpy(tiny_bulk_with_outliers(n, 4300 + j))
        x = t.to(DT[dt]) if dt != "f32" else t
        for bits_ in (8, 4):
            o = run_pct(qat, orc, x, bits_, scheme, 0.001)
            assert o["flags"] == 0
        run_pct(qat, orc, x, 8, scheme, 0.001, sr=(0xABCDEF, 123))
