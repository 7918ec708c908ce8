"""GPU parity of stochastic rounding: the CUDA library's *_sr entry points
against the oracle's, element by element (bit patterns), on the same seeded
inputs and the same (seed, offset).  Every kernel path is exercised: per
tensor (calibrated and given parameters), per group (lanes of a warp), per
row (a block per row), the per-unit fallback, scales outside the
reciprocal's safe range, and FP8 with specials.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import Poisoned, assert_same, bits, oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
SEEDS = [(0, 0), (0x9E3779B97F4A7C15, 12345), (7, (1 << 40) - 3)]


def make_input(rows, cols, dtype, seed, specials=False):
    rng = np.random.default_rng(seed)
    sig = np.exp(rng.uniform(np.log(0.01), np.log(3.0), size=(rows, 1))).astype(np.float32)
    a = (rng.standard_normal((rows, cols)).astype(np.float32) * sig
         + rng.uniform(-0.3, 0.3, size=(rows, 1)).astype(np.float32))
    flat = a.reshape(-1)
    flat[rng.integers(0, flat.size, size=max(1, flat.size // 97))] = 0.0
    flat[rng.integers(0, flat.size, size=max(1, flat.size // 211))] = -0.0
    if specials and flat.size > 8:
        flat[3], flat[5], flat[7] = np.inf, -np.inf, np.nan
    t = torch.from_numpy(a)
    return t.to(dtype) if dtype != torch.float32 else t


def run_int_sr(qat, orc, x, rows, cols, bits_, scheme, gran, group, seed, offset, scale=None,
               zp=None):
    dev = "cuda"
    n = rows * cols
    units = orc.n_units(rows, cols, gran, group)
    xd = x.to(dev).contiguous()
    y = Poisoned(n, x.dtype)
    codes = Poisoned(n if bits_ == 8 else (n + 1) // 2, torch.int8 if bits_ == 8 else torch.uint8)
    mask = Poisoned((n + 31) // 32, torch.int32)
    given = scale is not None
    if given:
        sc = torch.tensor(np.asarray(scale, np.float32), device=dev)
        zpt = torch.tensor(np.asarray(zp, np.int32), device=dev) if zp is not None else None
    else:
        sc = torch.empty(units, dtype=torch.float32, device=dev)
        zpt = torch.empty(units, dtype=torch.int32, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(max(qat.qat_workspace_bytes(rows, cols, gran, group), 16), dtype=torch.uint8,
                     device=dev)
    qat.qat_fake_quant_int_sr(xd, rows, cols, bits_, scheme, gran, group, given, sc, zpt, seed,
                              offset, y.t, codes.t, mask.t, flags, ws)
    torch.cuda.synchronize()
    assert y.canary_ok() and codes.canary_ok() and mask.canary_ok()
    o = orc.fake_quant_int_sr(oracle_input(x), rows, cols, bits_, scheme, gran, group, seed=seed,
                              offset=offset, scale=scale, zero_point=zp)
    tag = (f"{x.dtype} bits={bits_} scheme={scheme} gran={gran} ({rows},{cols}) g={group} "
           f"seed={seed:#x} offset={offset}")
    assert_same(bits(y.t), o["y"], "y " + tag)
    assert_same(bits(codes.t), o["codes"].view(np.uint8), "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    if not given:
        assert_same(bits(sc), o["scale"], "scale " + tag)
    assert int(flags.item()) == o["flags"], tag


# (granularity, rows, cols, group): per tensor; groups of 128 / 32 (lanes of a
# warp); rows of 4096 / 96 / 8192 (a block per row); rows of 40 and groups of
# 100 (the per-unit fallback); ragged tails throughout
SHAPES = [(0, 3, 1025, 0), (0, 7, 9999, 0), (2, 6, 512, 128), (2, 4, 96, 32), (1, 5, 4096, 0),
          (1, 7, 96, 0), (1, 2, 8192, 0), (1, 4, 40, 0), (2, 4, 300, 100)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("scheme", [0, 1])
def test_int_sr_calibrated(qat, orc, dt, bits_, scheme):
    for i, (gran, r, c, g) in enumerate(SHAPES):
        x = make_input(r, c, DT[dt], seed=700 + i)
        for seed, off in SEEDS:
            run_int_sr(qat, orc, x, r, c, bits_, scheme, gran, g, seed, off)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_int_sr_given_params_and_unsafe_scales(qat, orc, dt, scheme):
    rng = np.random.default_rng(71)
    for bits_ in (8, 4):
        x = make_input(3, 1000, DT[dt], seed=710, specials=True)
        run_int_sr(qat, orc, x, 3, 1000, bits_, scheme, 0, 0, 5, 77, scale=[0.013],
                   zp=[2] if scheme else None)
        # per row, one scale outside [2^-80, 2^100] (IEEE division path), one invalid
        r, c = 6, 160
        x = make_input(r, c, DT[dt], seed=711, specials=True)
        sc = rng.uniform(0.001, 0.05, size=r).astype(np.float32)
        sc[1] = np.float32(1e-30)
        sc[2] = -1.0
        zp = rng.integers(-3, 3, size=r).astype(np.int32) if scheme else None
        run_int_sr(qat, orc, x, r, c, bits_, scheme, 1, 0, 9, 1 << 33, scale=sc, zp=zp)


def test_int_sr_is_unbiased_on_device(qat):
    """The module's example on the GPU path: scale 0.1, a value 70% of the way
    between two levels, 400,000 draws; mean within 8 sigma, only the two levels."""
    n = 400_000
    s = np.float32(12.7) / np.float32(127)
    value = np.float32(np.float32(3.0) + np.float32(0.7) * s)
    x = torch.full((n,), float(value), dtype=torch.float32, device="cuda")
    r = __import__("fake_quant_numerics_gb300").fake_quant_int(
        x, 8, "symmetric", "tensor", scale=torch.tensor([s]), rounding="stochastic", seed=12345)
    y = r.y.double().cpu().numpy()
    lo, hi = float(np.float32(30) * s), float(np.float32(31) * s)
    assert np.all((y == lo) | (y == hi))
    assert abs(y.mean() - float(value)) < 8 * float(s) / np.sqrt(n)


def run_fp8_sr(qat, orc, x, fmt, seed, offset, scale=None, with_codes=True):
    n = x.numel()
    xd = x.cuda().contiguous()
    y = Poisoned(n, x.dtype)
    codes = Poisoned(n, torch.uint8) if with_codes else None
    mask = Poisoned((n + 31) // 32, torch.int32)
    s = torch.tensor([0.0 if scale is None else scale], dtype=torch.float32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(qat.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device="cuda")
    qat.qat_fake_quant_fp8_sr(xd, n, fmt, scale is not None, s, seed, offset, y.t,
                              codes.t if with_codes else None, mask.t, flags, ws)
    torch.cuda.synchronize()
    assert y.canary_ok() and (codes is None or codes.canary_ok()) and mask.canary_ok()
    o = orc.fake_quant_fp8_sr(oracle_input(x), fmt, seed=seed, offset=offset, scale=scale)
    tag = f"fp8 fmt={fmt} {x.dtype} n={n} seed={seed:#x} offset={offset} scale={scale}"
    assert_same(bits(y.t), o["y"], "y " + tag)
    if with_codes:
        assert_same(bits(codes.t), o["codes"], "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    assert_same(bits(s), np.array([o["scale"]], np.float32), "scale " + tag)
    assert int(flags.item()) == o["flags"], tag


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_fp8_sr(qat, orc, fmt, dt):
    rng = np.random.default_rng(720 + fmt)
    for n in (1, 33, 1023, 5000, 65536 + 17):
        a = (rng.standard_t(3, size=n) * 0.5).astype(np.float32)
        k = max(1, n // 50)
        idx = rng.integers(0, n, size=k)
        a[idx] = rng.choice(np.array([0.0, -0.0, 1e6, -1e6, np.inf, -np.inf, np.nan,
                                      2.0 ** -130, -(2.0 ** -130)], np.float32), size=k)
        t = torch.from_numpy(a)
        x = t.to(DT[dt]) if dt != "f32" else t
        for seed, off in SEEDS[:2]:
            run_fp8_sr(qat, orc, x, fmt, seed, off)                   # amax scale
            run_fp8_sr(qat, orc, x, fmt, seed, off, scale=1.0)        # the unscaled cast
            run_fp8_sr(qat, orc, x, fmt, seed, off, scale=1e-30)      # outside the safe range
            run_fp8_sr(qat, orc, x, fmt, seed, off, with_codes=False)  # y and mask only
        run_fp8_sr(qat, orc, x, fmt, 3, 4, scale=0.0)                 # zero scale
        run_fp8_sr(qat, orc, x, fmt, 3, 4, scale=-1.0)                # invalid given scales
        run_fp8_sr(qat, orc, x, fmt, 3, 4, scale=float("inf"), with_codes=False)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_fp8_sr_at_the_normal_boundary(qat, orc, fmt, dt):
    """Whole vectors of quotients just above, at and just below 2^emin (the
    smallest normal of the format), where the kernel switches between the
    bit rule for normal targets and the general rule; given scales that are
    not powers of two, and the amax scale."""
    emin = -6 if fmt == 0 else -14
    rng = np.random.default_rng(740 + fmt)
    n = 4096 + 5
    for s in (0.3, 1.7e-3, 3.0e4):
        edge = np.float64(s) * 2.0 ** emin
        rel = rng.choice(np.array([-2.0 ** -8, -2.0 ** -20, 0.0, 2.0 ** -20, 2.0 ** -8, 1.0, 7.5]),
                         size=n)
        a = (edge * (1.0 + rel) * rng.choice(np.array([-1.0, 1.0]), size=n)).astype(np.float32)
        t = torch.from_numpy(a)
        x = t.to(DT[dt]) if dt != "f32" else t
        for seed, off in SEEDS[:2]:
            run_fp8_sr(qat, orc, x, fmt, seed, off, scale=s)
        run_fp8_sr(qat, orc, x, fmt, 5, 0)
