"""GPU parity of the calibration options (qat_fake_quant_int_opts: the clip
factor and binary16 scales) against the oracle, bit for bit, on every device
path: per tensor, per group (lanes of a warp), per row (a block per row and
the per-unit fallback), per column (staged and the unit fallback), nearest
and stochastic rounding, and the degenerate binary16 scales."""
import numpy as np
import pytest
import torch

from gpu_helpers import Poisoned, assert_same, bits, oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
# (granularity, rows, cols, group): tensor; groups of 128 / 32; rows of 4096
# (a block per row) and 40 (fallback); columns, staged (cols % 32 == 0) and not
CASES = [(0, 3, 1025, 0), (2, 6, 512, 128), (2, 4, 96, 32), (1, 5, 4096, 0), (1, 4, 40, 0),
         (3, 200, 256, 0), (3, 9, 33, 0)]


def make_input(rows, cols, dtype, seed, tails=True):
    rng = np.random.default_rng(seed)
    a = rng.standard_t(3, size=(rows, cols)).astype(np.float32) * np.float32(0.3)
    a += rng.uniform(-0.2, 0.2, size=(rows, 1)).astype(np.float32)
    t = torch.from_numpy(a)
    return t.to(dtype) if dtype != torch.float32 else t


def run_opts(qat, orc, x, rows, cols, bits_, scheme, gran, group, clip, fp16, sr=None):
    n = rows * cols
    units = orc.n_units(rows, cols, gran, group)
    xd = x.cuda().contiguous()
    y = Poisoned(n, x.dtype)
    codes = Poisoned(n if bits_ == 8 else (n + 1) // 2, torch.int8 if bits_ == 8 else torch.uint8)
    mask = Poisoned((n + 31) // 32, torch.int32)
    sc = Poisoned(units, torch.float32)
    zp = Poisoned(units, torch.int32)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(qat.qat_workspace_bytes(rows, cols, gran, group), 16), dtype=torch.uint8,
                     device="cuda")
    seed, off = sr if sr else (0, 0)
    qat.qat_fake_quant_int_opts(xd, rows, cols, bits_, scheme, gran, group,
                                qat.calib_options(clip, fp16), sr is not None, seed, off, sc.t,
                                zp.t, y.t, codes.t, mask.t, flags, ws)
    torch.cuda.synchronize()
    o = orc.fake_quant_int_opts(oracle_input(x), rows, cols, bits_, scheme, gran, group, clip=clip,
                                fp16=fp16, stochastic=sr is not None, seed=seed, offset=off)
    tag = (f"{x.dtype} bits={bits_} scheme={scheme} gran={gran} ({rows},{cols}) g={group} "
           f"clip={clip} fp16={fp16} sr={sr}")
    for b in (y, codes, mask, sc, zp):
        assert b.canary_ok(), tag
    yo = o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"]
    assert_same(bits(y.t), yo, "y " + tag)
    assert_same(bits(codes.t), o["codes"].view(np.uint8), "codes " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    assert_same(bits(sc.t), o["scale"].view(np.uint32), "scale " + tag)
    if scheme == 1:
        assert_same(zp.t.cpu().numpy(), o["zero_point"], "zero point " + tag)
    assert int(flags.item()) == o["flags"], tag
    return o


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_clip_and_fp16_every_path(qat, orc, dt, scheme):
    for i, (gran, r, c, g) in enumerate(CASES):
        x = make_input(r, c, DT[dt], seed=2000 + i)
        for bits_ in (8, 4):
            for clip, fp16 in ((1.0, True), (0.7, False), (0.3, True), (0.5, False)):
                run_opts(qat, orc, x, r, c, bits_, scheme, gran, g, clip, fp16)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("scheme", [0, 1])
def test_clip_and_fp16_stochastic(qat, orc, dt, scheme):
    for i, (gran, r, c, g) in enumerate(CASES):
        x = make_input(r, c, DT[dt], seed=2100 + i)
        run_opts(qat, orc, x, r, c, 4, scheme, gran, g, 0.6, True, sr=(0x5EED, 77))


def test_fp16_scales_out_of_range_are_degenerate(qat, orc):
    """Scales that round to binary16 zero (tiny values) or infinity (huge
    ones) are degenerate units."""
    for scale_of in (1e-12, 1e9):
        x = (make_input(4, 256, torch.float32, seed=2200) * scale_of).to(torch.float32)
        for gran, g in ((0, 0), (2, 64), (1, 0), (3, 0)):
            o = run_opts(qat, orc, x, 4, 256, 8, 0, gran, g, 1.0, True)
            assert o["flags"] & orc.FLAG_DEGENERATE


def test_named_op_options(qat, orc):
    import fake_quant_numerics_gb300 as fq
    x = make_input(8, 512, torch.float32, seed=2300)
    r = fq.fake_quant_int(x.cuda(), 4, "symmetric", "group", 128, clip=0.5, scale_fp16=True)
    o = orc.fake_quant_int_opts(x.numpy().reshape(-1), 8, 512, 4, 0, 2, 128, clip=0.5, fp16=True)
    assert_same(bits(r.y).reshape(-1), o["y"].view(np.uint32), "named op y")
    with pytest.raises(fq.QatError):
        fq.qat_fake_quant_int_opts(x.cuda(), 8, 512, 8, 0, 0, 0, fq.calib_options(1.5), False, 0,
                                   0, torch.empty(1, device="cuda"), None,
                                   torch.empty(8 * 512, device="cuda"), None, None,
                                   torch.zeros(1, dtype=torch.int32, device="cuda"),
                                   torch.empty(16384, dtype=torch.uint8, device="cuda"))
