"""GPU parity of tensors at element offsets: views such as x[k:] whose data
pointer holds whole elements but is off the 32-byte grid of the vector
kernels.  x, y, grad and grad_in at offsets 1-7 (fp32) and 1-15 (bf16),
against the oracle bit for bit: integer fake quant per tensor, per row and per
group (calibrated or given parameters, nearest or stochastic rounding,
calibration options), FP8 (amax-scaled or given scale, nearest or
stochastic), the STE backward, the statistics, and the two-level 4-bit
quantize (x, the fused round trip's y) and dequantize (y)."""
import numpy as np
import pytest
import torch

from gpu_helpers import Poisoned, assert_same, bits, oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
OFFSETS = {"f32": range(1, 8), "bf16": range(1, 16)}


def at_offset(t: torch.Tensor, off: int) -> torch.Tensor:
    """A CUDA view of t's values starting `off` elements into a fresh buffer."""
    buf = torch.empty(t.numel() + off + 16, dtype=t.dtype, device="cuda")
    v = buf[off:off + t.numel()]
    v.copy_(t.reshape(-1).to("cuda"))
    return v


def empty_at(n, dtype, off):
    return torch.empty(n + off + 16, dtype=dtype, device="cuda")[off:off + n]


def make(rows, cols, dt, seed):
    rng = np.random.default_rng(seed)
    a = (rng.standard_normal((rows, cols)) * rng.uniform(0.05, 2.0, size=(rows, 1))).astype(np.float32)
    a.reshape(-1)[rng.integers(0, a.size, size=max(1, a.size // 50))] = 0.0
    t = torch.from_numpy(a)
    return t.to(DT[dt]) if dt != "f32" else t


def run_int_at(qat, orc, x, rows, cols, bits_, scheme, gran, group, xoff, yoff, sr=None,
               clip=1.0, given=False):
    n = rows * cols
    units = orc.n_units(rows, cols, gran, group)
    xd = at_offset(x, xoff)
    y = empty_at(n, x.dtype, yoff)
    codes = Poisoned(n if bits_ == 8 else (n + 1) // 2, torch.int8 if bits_ == 8 else torch.uint8)
    mask = Poisoned((n + 31) // 32, torch.int32)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(qat.qat_workspace_bytes(rows, cols, gran, group), 16), dtype=torch.uint8,
                     device="cuda")
    if given:
        o0 = orc.fake_quant_int(oracle_input(x), rows, cols, bits_, scheme, gran, group)
        sc = torch.from_numpy(o0["scale"].copy()).cuda()
        zp = torch.from_numpy(o0["zero_point"].copy()).cuda() if scheme else None
    else:
        sc = torch.empty(units, device="cuda")
        zp = torch.empty(units, dtype=torch.int32, device="cuda")
    seed, off = sr if sr else (0, 0)
    if clip != 1.0:
        qat.qat_fake_quant_int_opts(xd, rows, cols, bits_, scheme, gran, group,
                                    qat.calib_options(clip), sr is not None, seed, off, sc, zp, y,
                                    codes.t, mask.t, flags, ws)
    elif sr is not None:
        qat.qat_fake_quant_int_sr(xd, rows, cols, bits_, scheme, gran, group, given, sc, zp, seed,
                                  off, y, codes.t, mask.t, flags, ws)
    else:
        qat.qat_fake_quant_int(xd, rows, cols, bits_, scheme, gran, group, given, sc, zp, y,
                               codes.t, mask.t, flags, ws)
    torch.cuda.synchronize()
    if given:
        o = orc.fake_quant_int(oracle_input(x), rows, cols, bits_, scheme, gran, group,
                               scale=o0["scale"], zero_point=o0["zero_point"] if scheme else None)
        if sr is not None:
            o = orc.fake_quant_int_sr(oracle_input(x), rows, cols, bits_, scheme, gran, group,
                                      seed=seed, offset=off, scale=o0["scale"],
                                      zero_point=o0["zero_point"] if scheme else None)
    elif clip != 1.0 or sr is not None:
        o = orc.fake_quant_int_opts(oracle_input(x), rows, cols, bits_, scheme, gran, group,
                                    clip=clip, stochastic=sr is not None, seed=seed, offset=off)
    else:
        o = orc.fake_quant_int(oracle_input(x), rows, cols, bits_, scheme, gran, group)
    tag = (f"{x.dtype} bits={bits_} scheme={scheme} gran={gran} ({rows},{cols}) g={group} "
           f"xoff={xoff} yoff={yoff} sr={sr} clip={clip} given={given}")
    assert codes.canary_ok() and mask.canary_ok(), tag
    assert_same(bits(y), o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"], "y " + tag)
    assert_same(bits(codes.t), o["codes"].view(np.uint8), "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    if not given:
        assert_same(bits(sc), o["scale"].view(np.uint32), "scale " + tag)
        if scheme:
            assert_same(zp.cpu().numpy(), o["zero_point"], "zp " + tag)
    assert int(flags.item()) == o["flags"], tag


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_int_at_element_offsets(qat, orc, dt):
    for k, off in enumerate(OFFSETS[dt]):
        for gran, r, c, g in ((0, 3, 1000 + k, 0), (1, 5, 512, 0), (2, 4, 384, 128)):
            x = make(r, c, dt, 7000 + 10 * k + gran)
            bits_ = 8 if (k + gran) % 2 else 4
            scheme = (k + gran) % 2
            run_int_at(qat, orc, x, r, c, bits_, scheme, gran, g, off, 0)
            run_int_at(qat, orc, x, r, c, bits_, 1 - scheme, gran, g, 0, off)  # y off the grid


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_int_at_offsets_stochastic_options_given(qat, orc, dt):
    for gran, r, c, g in ((0, 2, 3001, 0), (1, 3, 256, 0), (2, 2, 512, 64)):
        x = make(r, c, dt, 7100 + gran)
        run_int_at(qat, orc, x, r, c, 4, 1, gran, g, 3, 5, sr=(0xFEED, 11))
        run_int_at(qat, orc, x, r, c, 8, 0, gran, g, 1, 1, clip=0.6)
        run_int_at(qat, orc, x, r, c, 8, 1, gran, g, 2, 0, given=True)
        run_int_at(qat, orc, x, r, c, 4, 0, gran, g, 0, 3, given=True, sr=(77, 5))


def run_fp8_at(qat, orc, x, fmt, xoff, yoff, scale=None, sr=None):
    n = x.numel()
    xd = at_offset(x, xoff)
    y = empty_at(n, x.dtype, yoff)
    codes = Poisoned(n, torch.uint8)
    mask = Poisoned((n + 31) // 32, torch.int32)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.tensor([scale if scale is not None else 0.0], dtype=torch.float32, device="cuda")
    ws = torch.empty(qat.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device="cuda")
    if sr is None:
        qat.qat_fake_quant_fp8(xd, n, fmt, scale is not None, sc, y, codes.t, mask.t, flags, ws)
        o = orc.fake_quant_fp8(oracle_input(x), fmt, scale=scale)
    else:
        qat.qat_fake_quant_fp8_sr(xd, n, fmt, scale is not None, sc, sr[0], sr[1], y, codes.t,
                                  mask.t, flags, ws)
        o = orc.fake_quant_fp8_sr(oracle_input(x), fmt, seed=sr[0], offset=sr[1], scale=scale)
    torch.cuda.synchronize()
    tag = f"{x.dtype} fmt={fmt} xoff={xoff} yoff={yoff} scale={scale} sr={sr}"
    yo = o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"]
    assert_same(bits(y), yo, "y " + tag)
    assert_same(bits(codes.t), o["codes"], "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    assert_same(bits(sc), np.array([o["scale"]], np.float32).view(np.uint32), "scale " + tag)
    assert int(flags.item()) == o["flags"], tag


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_fp8_at_element_offsets(qat, orc, dt):
    rng = np.random.default_rng(7200)
    a = (rng.standard_t(3, size=20_011) * 0.5).astype(np.float32)
    a[[3, 50, 900]] = [np.nan, np.inf, -0.0]
    a[1000:1010] = 1e6
    t = torch.from_numpy(a)
    x = t.to(DT[dt]) if dt != "f32" else t
    for k, off in enumerate(OFFSETS[dt]):
        fmt = k % 2
        run_fp8_at(qat, orc, x, fmt, off, 0)
        run_fp8_at(qat, orc, x, 1 - fmt, 0, off, scale=0.01)
    run_fp8_at(qat, orc, x, 0, 1, 3, sr=(5, 9))
    run_fp8_at(qat, orc, x, 1, 3, 0, scale=0.5, sr=(6, 1))
    run_fp8_at(qat, orc, x, 0, 2, 2, scale=0.0)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_ste_and_stats_at_element_offsets(qat, orc, dt):
    n = 10_007
    x = make(1, n, dt, 7300)
    g = make(1, n, dt, 7301)
    o = orc.fake_quant_int(oracle_input(x), 1, n, 8, 0, 0)
    mask = torch.from_numpy(o["mask"].view(np.int32).copy()).cuda()
    for off in OFFSETS[dt]:
        gd = at_offset(g, off)
        dx = empty_at(n, g.dtype, (off * 3) % (8 if dt == "f32" else 16))
        qat.qat_ste_backward(gd, n, mask, dx)
        torch.cuda.synchronize()
        assert_same(bits(dx), orc.ste_backward(oracle_input(g), o["mask"]), f"ste off={off}")
    # statistics per tensor and per row at an offset
    xd = at_offset(x, 1)
    for gran, rows, cols in ((0, 1, n), (1, 1, n)):
        am = torch.empty(1, device="cuda")
        mn = torch.empty(1, device="cuda")
        mx = torch.empty(1, device="cuda")
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.empty(max(qat.qat_workspace_bytes(rows, cols, gran, 0), 16), dtype=torch.uint8,
                         device="cuda")
        qat.qat_amax_stats(xd, rows, cols, gran, 0, am, mn, mx, flags, ws)
        torch.cuda.synchronize()
        ref = np.asarray(x.float().reshape(-1).numpy(), np.float64)
        assert am.item() == np.abs(ref).max() and mn.item() == ref.min() and mx.item() == ref.max()


def test_per_column_off_the_grid_is_refused(qat):
    """Per-column calls copy rows into shared memory with bulk copies that need
    16-byte addresses: a view off the grid is refused before any launch (the
    named ops copy such a view first)."""
    from fake_quant_numerics_gb300 import QatError

    x = torch.randn(64 * 64 + 1, device="cuda")[1:]
    y = torch.empty(64 * 64, device="cuda")
    sc = torch.empty(64, device="cuda")
    ws = torch.empty(qat.qat_workspace_bytes(64, 64, 3, 0), dtype=torch.uint8, device="cuda")
    c0 = qat.qat_kernel_launch_count()
    with pytest.raises(QatError, match="misaligned"):
        qat.qat_fake_quant_int(x, 64, 64, 8, 0, 3, 0, False, sc, None, y, None, None, None, ws)
    assert qat.qat_kernel_launch_count() == c0
    r = qat.fake_quant_int(x.view(64, 64), 8, "symmetric", "column")  # copied, then quantized
    torch.cuda.synchronize()
    assert r.y.shape == (64, 64)


def test_q4_double_at_element_offsets(qat, orc):
    """x and the fused round trip's y of quantize_4bit_double, and y of
    dequantize_4bit_double, at fp32 offsets 1-7; a ragged tail and a full
    super-block or more."""
    rng = np.random.default_rng(7400)
    for k, off in enumerate(range(1, 8)):
        n = 16384 * (1 + k % 3) + 37 * k + 5
        a = (rng.standard_normal(n) * 0.02).astype(np.float32)
        a[rng.integers(0, n, size=3)] = 0.0
        xd = at_offset(torch.from_numpy(a), off)
        nd, nb, ns = orc.q4_sizes(n)
        data = Poisoned(nd, torch.uint8)
        qs = Poisoned(nb, torch.uint8)
        sup = Poisoned(ns, torch.float32)
        yr = empty_at(n, torch.float32, (off * 3) % 8)
        qat.qat_quant4_double(xd, n, data.t, qs.t, sup.t, yr)
        y = empty_at(n, torch.float32, (off + 4) % 8)
        qat.qat_dequant4_double(data.t, qs.t, sup.t, n, y)
        torch.cuda.synchronize()
        o = orc.quant4_double(a, roundtrip=True)
        tag = f"n={n} off={off}"
        assert data.canary_ok() and qs.canary_ok() and sup.canary_ok(), tag
        assert_same(bits(data.t), o["data"], "data " + tag)
        assert_same(bits(qs.t), o["qscales"], "qscales " + tag)
        assert_same(bits(sup.t), o["super_scales"].view(np.uint32), "supers " + tag)
        assert_same(bits(yr), o["y"].view(np.uint32), "round trip " + tag)
        assert_same(bits(y), o["y"].view(np.uint32), "dequant " + tag)
