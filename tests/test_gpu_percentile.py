"""GPU parity of percentile calibration (qat_fake_quant_int_percentile: the
module's per_tensor_percentile by a radix select of the two nearest-rank
quantiles) against the oracle, bit for bit: y, codes, mask, scale, zero
point and flags, nearest and stochastic rounding, sizes from one element to
full size, heavy duplicates, signed zeros, constant and non-finite tensors."""
import numpy as np
import pytest
import torch

from gpu_helpers import Poisoned, assert_same, bits, oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
FRACS = [0.0, 0.001, 0.02, 0.25, 0.4999]


def run_pct(qat, orc, x, bits_, scheme, c, sr=None):
    n = x.numel()
    xd = x.cuda().contiguous()
    y = Poisoned(n, x.dtype)
    codes = Poisoned(n if bits_ == 8 else (n + 1) // 2, torch.int8 if bits_ == 8 else torch.uint8)
    mask = Poisoned((n + 31) // 32, torch.int32)
    sc = Poisoned(1, torch.float32)
    zp = Poisoned(1, torch.int32)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(qat.qat_percentile_workspace_bytes(), dtype=torch.uint8, device="cuda")
    ws.fill_(0x5A)
    seed, off = sr if sr else (0, 0)
    qat.qat_fake_quant_int_percentile(xd, n, bits_, scheme, c, sr is not None, seed, off, sc.t,
                                      zp.t, y.t, codes.t, mask.t, flags, ws)
    torch.cuda.synchronize()
    o = orc.fake_quant_int_percentile(oracle_input(x), bits_, scheme, c, stochastic=sr is not None,
                                      seed=seed, offset=off)
    tag = f"{x.dtype} n={n} bits={bits_} scheme={scheme} c={c} sr={sr}"
    for b in (y, codes, mask, sc, zp):
        assert b.canary_ok(), tag
    yo = o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"]
    assert_same(bits(y.t), yo, "y " + tag)
    assert_same(bits(codes.t), o["codes"].view(np.uint8), "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    assert_same(bits(sc.t), o["scale"].view(np.uint32), "scale " + tag)
    if scheme == 1:
        assert int(zp.t.item()) == int(o["zero_point"][0]), tag
    assert int(flags.item()) == o["flags"], tag
    return o


def heavy(n, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_t(2, size=n).astype(np.float32)
    a[rng.integers(0, n, size=max(1, n // 50))] *= np.float32(100.0)   # outliers
    return a


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_percentile_sizes_and_fractions(qat, orc, dt, scheme):
    for i, n in enumerate((1, 2, 7, 1000, 4097, 65536 + 13, 1 << 20)):
        t = torch.from_numpy(heavy(n, 3000 + i))
        x = t.to(DT[dt]) if dt != "f32" else t
        for c in FRACS:
            run_pct(qat, orc, x, 8 if i % 2 else 4, scheme, c)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_percentile_large_equal_bins(qat, orc, dt):
    """The low quantile inside a run of 65536 (then 65537) equal values, the
    high one among spread values; then both quantiles in runs of about
    175,000 equal values."""
    rng = np.random.default_rng(3150)
    n = 200000
    for k in (65536, 65537):
        a = np.concatenate([np.full(k, -5.0, np.float32),
                            rng.uniform(1.0, 1000.0, size=n - k).astype(np.float32)])
        rng.shuffle(a)
        t = torch.from_numpy(a)
        x = t.to(DT[dt]) if dt != "f32" else t
        for scheme in (0, 1):
            run_pct(qat, orc, x, 8, scheme, 0.001)
    a = rng.choice(np.array([-2.0, -0.5, -0.0, 0.0, 0.25, 3.0], np.float32), size=1 << 20)
    t = torch.from_numpy(a)
    x = t.to(DT[dt]) if dt != "f32" else t
    for c in (0.1, 0.3):
        run_pct(qat, orc, x, 8, 1, c)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_percentile_duplicates_and_signed_zeros(qat, orc, dt):
    rng = np.random.default_rng(3100)
    # few distinct values (long runs of equal keys), zeros of both signs
    a = rng.choice(np.array([-2.0, -0.5, -0.0, 0.0, 0.25, 3.0], np.float32), size=50000)
    t = torch.from_numpy(a)
    x = t.to(DT[dt]) if dt != "f32" else t
    for scheme in (0, 1):
        for c in (0.0, 0.1, 0.3, 0.45):
            run_pct(qat, orc, x, 8, scheme, c)
    # all zeros of one sign or the other, negative-only
    for a in (np.full(3000, -0.0, np.float32), np.zeros(3000, np.float32),
              -np.abs(heavy(3000, 3101))):
        t = torch.from_numpy(a.copy())
        x = t.to(DT[dt]) if dt != "f32" else t
        for scheme in (0, 1):
            run_pct(qat, orc, x, 4, scheme, 0.05)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_percentile_errors_and_stochastic(qat, orc, dt):
    a = heavy(20000, 3200)
    a[777] = np.nan
    t = torch.from_numpy(a)
    x = t.to(DT[dt]) if dt != "f32" else t
    for scheme in (0, 1):
        o = run_pct(qat, orc, x, 8, scheme, 0.01)
        assert o["flags"] & orc.FLAG_NONFINITE
    a = heavy(20000, 3201)
    a[5] = np.inf
    t = torch.from_numpy(a)
    x = t.to(DT[dt]) if dt != "f32" else t
    run_pct(qat, orc, x, 8, 0, 0.0)
    t = torch.from_numpy(heavy(30000, 3202))
    x = t.to(DT[dt]) if dt != "f32" else t
    for scheme in (0, 1):
        for bits_ in (8, 4):
            run_pct(qat, orc, x, bits_, scheme, 0.02, sr=(0x9E3779B97F4A7C15, 4321))


def test_percentile_full_size(qat, orc):
    """A 16M-element fp32 tensor (the w2 weights' size), every output compared."""
    t = torch.from_numpy(heavy(1 << 24, 3300))
    for scheme, bits_ in ((0, 8), (1, 4)):
        run_pct(qat, orc, t, bits_, scheme, 0.001)


def test_percentile_named_op_and_arguments(qat, orc):
    import fake_quant_numerics_gb300 as fq
    data = np.concatenate([np.arange(100) / 100.0, [1000.0]]).astype(np.float32)
    r = fq.fake_quant_int_percentile(torch.from_numpy(data).cuda(), 8, "symmetric", 0.02)
    assert float(r.scale.item()) == float(np.float32(np.float32(0.98) / np.float32(127)))
    x = torch.zeros(64, device="cuda")
    with pytest.raises(fq.QatError):
        fq.fake_quant_int_percentile(x, 8, "symmetric", 0.5)
