"""GPU parity: the CUDA library against the CPU oracle, element by element,
on seeded inputs that span several tiles, ragged tails, every kernel path
(per-tensor two-pass, fused per-group lanes, fused per-row blocks, the
per-unit fallback, given parameters) and the degenerate cases.

Every comparison is of bit patterns (codes, packed bytes, masks, scales, zero
points, fake-quant outputs).  Output buffers carry canaries to catch writes
past their end.
"""
import ctypes
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from gpu_helpers import Poisoned, assert_same, bits, oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
SCHEMES = {"sym": 0, "affine": 1}
GRAN = {"tensor": 0, "row": 1, "group": 2}


def make_input(rows, cols, dtype, seed, specials=False, zero_unit=None, nan_unit=None, L=None):
    rng = np.random.default_rng(seed)
    sig = np.exp(rng.uniform(np.log(0.01), np.log(3.0), size=(rows, 1))).astype(np.float32)
    a = (rng.standard_normal((rows, cols)).astype(np.float32) * sig
         + rng.uniform(-0.3, 0.3, size=(rows, 1)).astype(np.float32))
    flat = a.reshape(-1)
    if flat.size:
        flat[rng.integers(0, flat.size, size=max(1, flat.size // 97))] = 0.0
        flat[rng.integers(0, flat.size, size=max(1, flat.size // 211))] = -0.0
    if zero_unit is not None and L:
        flat[zero_unit * L:(zero_unit + 1) * L] = 0.0
    if nan_unit is not None and L and nan_unit * L + (L // 3) < flat.size:
        flat[nan_unit * L + (L // 3)] = np.nan
    if specials and flat.size > 8:
        flat[3] = np.inf
        flat[5] = -np.inf
        flat[7] = np.nan
    t = torch.from_numpy(a)
    return t.to(dtype) if dtype != torch.float32 else t


def run_int(qat, orc, x, rows, cols, bits_, scheme, gran, group=0, scale=None, zp=None):
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
        scp = Poisoned(units, torch.float32)
        zpp = Poisoned(units, torch.int32)
        sc, zpt = scp.t, zpp.t
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = qat.qat_workspace_bytes(rows, cols, gran, group)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    qat.qat_fake_quant_int(xd, rows, cols, bits_, scheme, gran, group, given, sc, zpt, y.t, codes.t,
                           mask.t, flags, ws)
    torch.cuda.synchronize()
    for b, name in ((y, "y"), (codes, "codes"), (mask, "mask")):
        assert b.canary_ok(), f"write past the end of {name}"
    if not given:
        assert scp.canary_ok() and zpp.canary_ok()
    o = orc.fake_quant_int(oracle_input(x), rows, cols, bits_, scheme, gran, group,
                           scale=scale, zero_point=zp)
    tag = f"{x.dtype} bits={bits_} scheme={scheme} gran={gran} shape=({rows},{cols}) group={group}"
    assert_same(bits(y.t), o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"], "y " + tag)
    assert_same(bits(codes.t), o["codes"].view(np.uint8), "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    if not given:
        assert_same(bits(sc), o["scale"].view(np.uint32), "scale " + tag)
        if scheme == 1:
            assert_same(zpt.cpu().numpy(), o["zero_point"], "zero point " + tag)
    assert int(flags.item()) == o["flags"], f"flags {tag}: {int(flags.item())} vs {o['flags']}"
    return o


TENSOR_SHAPES = [(1, 1), (1, 31), (1, 1023), (3, 1025), (1, 16385), (7, 9999)]
# (5000, 96): every block of the per-row kernel takes many rows; (2, 16384):
# the largest rows of the per-row kernel (8 vectors per thread for f32)
ROW_SHAPES = [(3, 64), (2, 256), (5, 4096), (3, 8192), (7, 96), (4, 40), (3, 1000), (2, 33),
              (1, 32768), (2, 16384), (5000, 96)]
GROUP_SHAPES = [(8, 512, 128), (3, 384, 128), (5, 96, 32), (4, 300, 100), (2, 1024, 1024),
                (4, 64, 16), (6, 256, 256), (2, 2048, 512)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("scheme", ["sym", "affine"])
def test_int_per_tensor(qat, orc, dt, bits_, scheme):
    for i, (r, c) in enumerate(TENSOR_SHAPES):
        x = make_input(r, c, DT[dt], seed=100 + i)
        run_int(qat, orc, x, r, c, bits_, SCHEMES[scheme], 0)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("scheme", ["sym", "affine"])
def test_int_per_row(qat, orc, dt, bits_, scheme):
    for i, (r, c) in enumerate(ROW_SHAPES):
        x = make_input(r, c, DT[dt], seed=200 + i, zero_unit=1 if r > 2 else None,
                       nan_unit=2 if r > 3 else None, L=c)
        run_int(qat, orc, x, r, c, bits_, SCHEMES[scheme], 1)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("scheme", ["sym", "affine"])
def test_int_per_group(qat, orc, dt, bits_, scheme):
    for i, (r, c, g) in enumerate(GROUP_SHAPES):
        x = make_input(r, c, DT[dt], seed=300 + i, zero_unit=1, nan_unit=3, L=g)
        run_int(qat, orc, x, r, c, bits_, SCHEMES[scheme], 2, g)


def plant_nonfinite(x, L):
    """Units of L elements with infinities placed where the statistics fold
    meets them in different ways: a lone +Inf or -Inf first, mid-vector or
    last; both signs; a whole unit of +Inf; a NaN beside an Inf; finite units
    between them (the fold keeps its running min / max across vectors)."""
    a = x.float().numpy().reshape(-1).copy()
    units = a.size // L
    plan = [(1, [(0, np.inf)]), (2, [(L // 2 + 3, -np.inf)]), (4, [(L - 1, np.inf)]),
            (5, [(5, np.inf), (L - 9, -np.inf)]), (7, "all"), (8, [(1, np.nan), (L - 2, np.inf)]),
            (10, [(L // 3, -np.inf)])]
    for u, spots in plan:
        if u >= units:
            continue
        if spots == "all":
            a[u * L:(u + 1) * L] = np.inf
        else:
            for off, v in spots:
                a[u * L + off] = v
    t = torch.from_numpy(a.reshape(x.shape))
    return t.to(x.dtype) if x.dtype != torch.float32 else t


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", ["sym", "affine"])
def test_int_infinities_in_units(qat, orc, dt, scheme):
    """Per-row and per-group calibration with infinities in some units: those
    units are flagged and their outputs zero, the others unchanged."""
    for gran, shapes in ((1, [(12, 256), (11, 4096), (12, 1000)]),
                         (2, [(3, 1536, 128), (2, 1408, 64), (12, 96, 32)])):
        for i, shp in enumerate(shapes):
            r, c = shp[0], shp[1]
            g = shp[2] if gran == 2 else 0
            L = g if gran == 2 else c
            x = plant_nonfinite(make_input(r, c, DT[dt], seed=900 + 10 * gran + i), L)
            for bits_ in (8, 4):
                o = run_int(qat, orc, x, r, c, bits_, SCHEMES[scheme], gran, g)
                assert o["flags"] & orc.FLAG_NONFINITE


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits_", [8, 4])
def test_int_affine_zero_window_ends(qat, orc, dt, bits_):
    """Affine units whose window ends at 0 (all values >= 0 gives zp = qmin and
    wlo = +0; all values <= 0 gives zp = qmax and whi = +0) holding both signed
    zeros: -0 and +0 are inside the window."""
    rng = np.random.default_rng(61)
    for gran, (r, c, g) in ((0, (1, 4096, 0)), (1, (4, 4096, 0)), (1, (4, 96, 0)),
                            (2, (4, 512, 128)), (2, (4, 512, 64))):
        a = np.abs(rng.standard_normal((r, c)).astype(np.float32)) + np.float32(0.01)
        if gran == 0:
            a = a if rng.integers(2) else -a
        else:
            a[1::2] *= -1  # odd rows non-positive, even rows non-negative
        flat = a.reshape(-1)
        flat[rng.integers(0, flat.size, size=flat.size // 9)] = -0.0
        flat[rng.integers(0, flat.size, size=flat.size // 9)] = 0.0
        x = torch.from_numpy(a)
        x = x.to(DT[dt]) if dt != "f32" else x
        run_int(qat, orc, x, r, c, bits_, 1, gran, g)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", ["sym", "affine"])
def test_int_given_params(qat, orc, dt, scheme):
    """Given parameters: NaN -> code 0, +-Inf -> clamp ends, invalid units flagged."""
    sch = SCHEMES[scheme]
    rng = np.random.default_rng(7)
    for bits_ in (8, 4):
        # per tensor
        x = make_input(3, 1000, DT[dt], seed=400, specials=True)
        run_int(qat, orc, x, 3, 1000, bits_, sch, 0, scale=[0.013], zp=[3] if sch else None)
        # per row with one invalid unit of each kind
        r, c = 6, 160
        x = make_input(r, c, DT[dt], seed=401, specials=True)
        sc = rng.uniform(0.001, 0.05, size=r).astype(np.float32)
        zp = rng.integers(-5, 5, size=r).astype(np.int32)
        sc[1] = 0.0
        sc[2] = -1.0
        sc[3] = np.inf
        if sch:
            zp[4] = 500
        run_int(qat, orc, x, r, c, bits_, sch, 1, scale=sc, zp=zp if sch else None)
        # per group
        x = make_input(4, 256, DT[dt], seed=402, specials=True)
        g = 64
        sc = rng.uniform(0.001, 0.05, size=16).astype(np.float32)
        zp = rng.integers(-5, 5, size=16).astype(np.int32)
        run_int(qat, orc, x, 4, 256, bits_, sch, 2, g, scale=sc, zp=zp if sch else None)


def test_int_degenerate_whole_tensor(qat, orc):
    for dt in ("f32", "bf16"):
        z = torch.zeros(2, 512, dtype=DT[dt])
        for scheme in (0, 1):
            for gran, g in ((0, 0), (1, 0), (2, 128)):
                o = run_int(qat, orc, z, 2, 512, 8, scheme, gran, g)
                assert o["flags"] & orc.FLAG_DEGENERATE


# ---------------------------------------------------------------------------
# FP8
# ---------------------------------------------------------------------------
def run_fp8(qat, orc, x, fmt, scale=None, want_codes=True):
    dev = "cuda"
    n = x.numel()
    xd = x.to(dev).contiguous().reshape(-1)
    y = Poisoned(n, x.dtype)
    codes = Poisoned(n, torch.uint8) if want_codes else None
    mask = Poisoned((n + 31) // 32, torch.int32)
    s = torch.tensor([0.0 if scale is None else scale], dtype=torch.float32, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(qat.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device=dev)
    qat.qat_fake_quant_fp8(xd, n, fmt, scale is not None, s, y.t, codes.t if codes else None, mask.t,
                           flags, ws)
    torch.cuda.synchronize()
    assert y.canary_ok() and mask.canary_ok() and (codes is None or codes.canary_ok())
    o = orc.fake_quant_fp8(oracle_input(x), fmt, scale=scale)
    tag = f"fp8 fmt={fmt} {x.dtype} n={n} scale={scale}"
    assert_same(bits(y.t), o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"], "y " + tag)
    if codes is not None:
        assert_same(bits(codes.t), o["codes"], "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    assert bits(s)[0] == np.float32(o["scale"]).view(np.uint32), tag
    assert int(flags.item()) == o["flags"], tag
    return o


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_workload_like_small(qat, orc, fmt):
    from fake_quant_numerics_gb300 import workloads as W

    for rows, cols in ((64, 1024), (3, 777), (1, 5)):
        a = W.cfg3(rows=rows, cols=cols, seed=11 + rows)
        run_fp8(qat, orc, a, fmt)
        run_fp8(qat, orc, a.float(), fmt)


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_all_fp16_and_bf16_values_unscaled(qat, orc, fmt):
    with np.errstate(invalid="ignore"):
        xs = torch.from_numpy(np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float32))
    run_fp8(qat, orc, xs, fmt, scale=1.0)
    bf = torch.from_numpy(np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.int16)).view(
        torch.bfloat16)
    run_fp8(qat, orc, bf, fmt, scale=1.0)


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_all_fp32_bit_patterns_unscaled(qat, orc, fmt):
    """Every one of the 2^32 fp32 bit patterns through the hardware cast path,
    against the oracle's restatement of the rounding rule (scale 1)."""
    chunk = 1 << 26
    n = chunk
    x = torch.empty(n, dtype=torch.int32, device="cuda")
    y = torch.empty(n, dtype=torch.float32, device="cuda")
    codes = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, dtype=torch.float32, device="cuda")
    pool = ThreadPoolExecutor(max_workers=16)

    def oracle_part(xs):
        return orc.fake_quant_fp8(xs, fmt, scale=1.0, want_mask=False)

    for c0 in range(0, 1 << 32, chunk):
        base = np.arange(c0, c0 + chunk, dtype=np.uint64).astype(np.uint32)
        x.copy_(torch.from_numpy(base.view(np.int32)))
        qat.qat_fake_quant_fp8(x.view(torch.float32), n, fmt, True, s, y, codes, None, None, None)
        xs = base.view(np.float32)
        parts = list(pool.map(oracle_part, np.array_split(xs, 16)))
        gy, gc = bits(y), bits(codes)
        assert_same(gy, np.concatenate([p["y"] for p in parts]).view(np.uint32), f"y chunk {c0:#x}")
        assert_same(gc, np.concatenate([p["codes"] for p in parts]), f"codes chunk {c0:#x}")
    pool.shutdown()


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_random_scales_random_bit_patterns(qat, orc, fmt):
    """Given scales across the whole fast range and its edges, each over 2^20
    random fp32 bit patterns plus values placed on and next to the cast's
    rounding boundaries (scaled FP8 midpoints +- a few ulps)."""
    rng = np.random.default_rng(31 + fmt)
    scales = [float(np.float32(2.0 ** e * m)) for e, m in
              zip(rng.integers(-80, 100, size=10), rng.uniform(1, 2, size=10))]
    scales += [float(np.float32(v)) for v in (2.0 ** -80, 2.0 ** 100, 1 - 2 ** -24, 1.9999999, 3.0,
                                              448 / 7, 2.0 ** -81, 2.0 ** 101)]
    probe = np.concatenate([[0.0], np.geomspace(2.0 ** -20, 6.0e4, 400_000)]).astype(np.float32)
    grid = np.unique(np.abs(orc.fake_quant_fp8(probe, fmt, scale=1.0)["y"].astype(np.float64)))
    mids = (grid[:-1] + grid[1:]) / 2
    for sc in scales:
        bits_ = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
        x = bits_.view(np.float32).copy()
        near = (mids * sc).astype(np.float32)
        near = np.concatenate([near, -near])
        for d in (-2, -1, 0, 1, 2):
            x[: near.size] = (near.view(np.int32) + d).view(np.float32)
            run_fp8(qat, orc, torch.from_numpy(x.copy()), fmt, scale=sc, want_codes=True)


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_zero_and_invalid_scale(qat, orc, fmt):
    x = make_input(2, 300, torch.float32, seed=5, specials=True)
    for s in (0.0, -1.0, float("nan"), float("inf"), 2.5e-3):
        run_fp8(qat, orc, x, fmt, scale=s)
    z = torch.zeros(1000)
    z[17] = float("nan")
    o = run_fp8(qat, orc, z, fmt)
    assert o["scale"] == 0.0


# ---------------------------------------------------------------------------
# STE backward
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_ste_backward(qat, orc, dt):
    rng = np.random.default_rng(9)
    for n in (1, 31, 32, 33, 1000, 1024, 1025, 70001):
        g = torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(DT[dt])
        m = rng.integers(0, 1 << 32, size=(n + 31) // 32, dtype=np.uint64).astype(np.uint32)
        dx = Poisoned(n, DT[dt])
        qat.qat_ste_backward(g.cuda(), n, torch.from_numpy(m.view(np.int32)).cuda(), dx.t)
        torch.cuda.synchronize()
        assert dx.canary_ok()
        assert_same(bits(dx.t), orc.ste_backward(oracle_input(g), m), f"ste {dt} n={n}")


# ---------------------------------------------------------------------------
# statistics
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_amax_stats(qat, orc, dt):
    cases = [(0, 3, 1025, 0), (0, 1, 1, 0), (1, 5, 4096, 0), (1, 3, 96, 0), (1, 4, 40, 0),
             (1, 5000, 96, 0), (1, 2, 16384, 0),
             (2, 8, 512, 128), (2, 4, 300, 100), (2, 3, 64, 32)]
    for i, (gran, r, c, g) in enumerate(cases):
        x = make_input(r, c, DT[dt], seed=500 + i, specials=True)
        units = orc.n_units(r, c, gran, g)
        L = r * c if gran == 0 else (c if gran == 1 else g)
        a, mn, mx = (Poisoned(units, torch.float32) for _ in range(3))
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.empty(max(qat.qat_workspace_bytes(r, c, gran, g), 16), dtype=torch.uint8,
                         device="cuda")
        qat.qat_amax_stats(x.cuda(), r, c, gran, g, a.t, mn.t, mx.t, flags, ws)
        torch.cuda.synchronize()
        omn, omx, oa, bad = orc.unit_stats(oracle_input(x), L)
        tag = f"stats {dt} gran={gran} ({r},{c}) g={g}"
        assert_same(bits(a.t), oa.view(np.uint32), "absmax " + tag)
        assert_same(bits(mn.t), omn.view(np.uint32), "min " + tag)
        assert_same(bits(mx.t), omx.view(np.uint32), "max " + tag)
        assert int(flags.item()) == (8 if bad.sum() else 0), tag
        assert a.canary_ok() and mn.canary_ok() and mx.canary_ok()


# ---------------------------------------------------------------------------
# two-level 4-bit
# ---------------------------------------------------------------------------
Q4_SIZES = [1, 2, 63, 64, 65, 127, 16383, 16384, 16385, 3 * 16384 + 100, 64 * 256 * 5 + 7, 1 << 20]


def run_q4(qat, orc, x: np.ndarray):
    n = x.size
    nd, nb, ns = orc.q4_sizes(n)
    xd = torch.from_numpy(x).cuda()
    data, qs, sup = Poisoned(nd, torch.uint8), Poisoned(nb, torch.uint8), Poisoned(ns, torch.float32)
    yrt = Poisoned(n, torch.float32)
    qat.qat_quant4_double(xd, n, data.t, qs.t, sup.t, yrt.t)
    y2 = Poisoned(n, torch.float32)
    qat.qat_dequant4_double(data.t, qs.t, sup.t, n, y2.t)
    data_b, qs_b, sup_b = Poisoned(nd, torch.uint8), Poisoned(nb, torch.uint8), Poisoned(ns, torch.float32)
    qat.qat_quant4_double(xd, n, data_b.t, qs_b.t, sup_b.t, None)
    torch.cuda.synchronize()
    for b in (data, qs, sup, yrt, y2, data_b, qs_b, sup_b):
        assert b.canary_ok()
    o = orc.quant4_double(x, roundtrip=True)
    tag = f"q4 n={n}"
    assert_same(bits(data.t), o["data"], "data " + tag)
    assert_same(bits(qs.t), o["qscales"], "qscales " + tag)
    assert_same(bits(sup.t), o["super_scales"].view(np.uint32), "supers " + tag)
    assert_same(bits(yrt.t), o["y"].view(np.uint32), "fused round trip " + tag)
    assert_same(bits(y2.t), o["y"].view(np.uint32), "dequant " + tag)
    assert_same(bits(data_b.t), o["data"], "data (no round trip) " + tag)
    assert_same(bits(qs_b.t), o["qscales"], "qscales (no round trip) " + tag)


def test_q4_double_sizes(qat, orc):
    rng = np.random.default_rng(13)
    for n in Q4_SIZES:
        run_q4(qat, orc, (rng.standard_normal(n) * 0.02).astype(np.float32))


def test_q4_double_specials(qat, orc):
    rng = np.random.default_rng(14)
    x = (rng.standard_normal(5 * 16384 + 33) * np.exp(rng.uniform(-20, 5, size=1))).astype(np.float32)
    x[:64] = 0.0                      # an all-zero block
    x[64:128] = -0.0
    x[200] = np.nan                   # NaN inside a block
    x[300] = np.inf                   # an infinite block scale
    x[16384:16384 * 2] = 0.0          # an all-zero super-block (super = 1e-8)
    x[40000:40064] = rng.standard_normal(64).astype(np.float32) * np.float32(2 ** -140)  # subnormals
    x[50000] = 3e38
    run_q4(qat, orc, x)
    run_q4(qat, orc, np.zeros(128, np.float32))
    run_q4(qat, orc, (np.sin(np.arange(4096, dtype=np.float32) * np.float32(0.1)) * 2).astype(np.float32))


def test_q4_double_exact_ties(qat, orc):
    """Blocks whose absmax is 7 * 2^k give the scale 2^k exactly, so x / s of
    half-integer multiples of 2^k are exact ties, which the codes round half
    away from zero; one block also holds a NaN, one a negative absmax."""
    rng = np.random.default_rng(15)
    nblk = 3 * 256 + 5
    x = np.empty(nblk * 64, np.float32)
    halves = np.arange(-13, 14, dtype=np.float32) / 2  # -6.5 .. 6.5 in steps of 1/2
    for b in range(nblk):
        k = int(rng.integers(-30, 30))
        blk = rng.choice(halves, size=64) * np.float32(2.0 ** k)
        blk[rng.integers(64)] = np.float32(7 * 2.0 ** k) * (1 if b % 5 else -1)
        blk[rng.integers(64, size=3)] = [0.0, -0.0, np.float32(2.0 ** k)]
        x[b * 64:(b + 1) * 64] = blk
    x[64 * 7 + 9] = np.nan
    run_q4(qat, orc, x)


# ---------------------------------------------------------------------------
# binding behaviour
# ---------------------------------------------------------------------------
def test_pointer_inside_an_element_is_rejected(qat):
    """A pointer that does not hold whole elements is refused before any
    launch (views at element offsets are accepted; tests/test_gpu_unaligned.py)."""
    import ctypes

    from fake_quant_numerics_gb300 import _lib

    lib = _lib.load()
    x = torch.randn(1000, device="cuda")
    y = torch.empty_like(x)
    s = torch.empty(1, device="cuda")
    ws = torch.empty(1 << 14, dtype=torch.uint8, device="cuda")
    c0 = lib.qat_kernel_launch_count()
    st = lib.qat_fake_quant_int(ctypes.c_void_p(x.data_ptr() + 2), _lib.F32, 1, 999, 8, 0, 0, 0,
                                0, ctypes.c_void_p(s.data_ptr()), None,
                                ctypes.c_void_p(y.data_ptr()), None, None, None,
                                ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
    assert st == _lib.QAT_ERR_MISALIGNED
    assert lib.qat_kernel_launch_count() == c0


def test_named_ops_and_launch_count(qat, orc):
    x = torch.randn(3, 4096, device="cuda")
    c0 = qat.qat_kernel_launch_count()
    r = qat.fake_quant_int(x, bits=8, scheme="symmetric", granularity="tensor")
    assert qat.qat_kernel_launch_count() - c0 == 1  # statistics and map in one launch
    r2 = qat.fake_quant_int(x[:, 1:], bits=8)  # non-contiguous input is copied first
    torch.cuda.synchronize()
    assert r2.y.shape == (3, 4095)
    # autograd wrapper: forward = fake quant, backward = STE
    xr = x.clone().requires_grad_(True)
    out = qat.FakeQuantSTE.apply(xr, 8, "symmetric", "row", 0)
    out.backward(torch.ones_like(out))
    m = np.unpackbits(bits(qat.fake_quant_int(x, 8, "symmetric", "row").mask).view(np.uint8),
                      bitorder="little")[: x.numel()]
    assert np.array_equal((xr.grad.reshape(-1).cpu().numpy() == 1.0), m.astype(bool))
    with pytest.raises(qat.QatDataError):
        qat.fake_quant_int(torch.zeros(64, device="cuda"), check=True)
    _ = r


def test_binding_dimension_mismatch(qat):
    """The binding's DIMENSION_MISMATCH (raised before any launch): a given
    parameter array whose length is not the unit count, an affine call given
    scales without zero points, and an STE mask of the wrong length."""
    from fake_quant_numerics_gb300 import _lib as L

    x = torch.randn(4, 64, device="cuda")
    c0 = qat.qat_kernel_launch_count()
    for kw in (dict(granularity="row", scale=torch.ones(3, device="cuda")),
               dict(granularity="group", group=32, scale=torch.ones(4, device="cuda")),
               dict(granularity="row", scheme="affine", scale=torch.ones(4, device="cuda")),
               dict(granularity="row", scheme="affine", scale=torch.ones(4, device="cuda"),
                    zero_point=torch.zeros(5, dtype=torch.int32, device="cuda"))):
        with pytest.raises(qat.QatError) as e:
            qat.fake_quant_int(x, 8, **kw)
        assert e.value.status == L.QAT_ERR_DIMENSION_MISMATCH, kw
    with pytest.raises(qat.QatError) as e:
        qat.fake_quant_backward(torch.randn(256, device="cuda"),
                                torch.zeros(7, dtype=torch.int32, device="cuda"))
    assert e.value.status == L.QAT_ERR_DIMENSION_MISMATCH
    assert qat.qat_kernel_launch_count() == c0
