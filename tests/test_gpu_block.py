"""GPU parity of block-scaled floating-point fake quant (qat_fake_quant_block:
MX formats with E8M0 scales, NVFP4 with E4M3 scales under an FP32 tensor
scale, exact FP32 scales) against the oracle, bit for bit: y, element codes,
block scales, tensor scale, mask and flags, every element format, blocks of
16 and 32, fp32 and bf16 inputs, with NaN, Inf, zeros, subnormal and
all-zero blocks."""
import numpy as np
import pytest
import torch

from gpu_helpers import Poisoned, assert_same, bits, oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
ELEM_BITS = {0: 8, 1: 8, 2: 6, 3: 6, 4: 4}


def make_input(n, seed, specials=True):
    rng = np.random.default_rng(seed)
    a = (rng.standard_t(5, size=n) * 0.02).astype(np.float32)
    # blocks of very different magnitude, an all-zero block, tiny values
    nb = n // 32
    a.reshape(nb, 32)[:, :] *= np.exp(rng.uniform(-12, 12, size=(nb, 1))).astype(np.float32)
    if specials and n >= 256:
        a[32:64] = 0.0
        a[70] = np.nan
        a[75] = np.inf
        a[80] = -np.inf
        a[100] = -0.0
        a[130:140] = np.float32(1e-40)  # binary32 subnormals
        a[200:224] = np.float32(3e38)
    return a


def run_block(qat, orc, x, fmt, block, kind):
    n = x.numel()
    xd = x.cuda().contiguous()
    y = Poisoned(n, x.dtype)
    ncodes = n // 2 if ELEM_BITS[fmt] == 4 else n
    codes = Poisoned(ncodes, torch.uint8)
    bs = Poisoned(n // block, torch.float32 if kind == 2 else torch.uint8)
    mask = Poisoned((n + 31) // 32, torch.int32)
    g = Poisoned(1, torch.float32)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(qat.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device="cuda")
    qat.qat_fake_quant_block(xd, n, fmt, block, kind, g.t, y.t, codes.t, bs.t, mask.t, flags, ws)
    torch.cuda.synchronize()
    o = orc.fake_quant_block(oracle_input(x), fmt, block, kind)
    tag = f"{x.dtype} n={n} fmt={fmt} block={block} kind={kind}"
    for b in (y, codes, bs, mask, g):
        assert b.canary_ok(), tag
    yo = o["y"].view(np.uint32) if x.dtype == torch.float32 else o["y"]
    assert_same(bits(y.t), yo, "y " + tag)
    oc = o["codes"]
    if ELEM_BITS[fmt] == 4:  # two codes per byte, element 2j in the high nibble
        oc = ((oc[0::2] & 0xF) << 4 | (oc[1::2] & 0xF)).astype(np.uint8)
    assert_same(bits(codes.t), oc, "codes " + tag)
    ob = o["bscales"].view(np.uint32) if kind == 2 else o["bscales"]
    assert_same(bits(bs.t), ob, "block scales " + tag)
    assert_same(bits(mask.t), o["mask"], "mask " + tag)
    assert_same(bits(g.t), np.array([o["tensor_scale"]], np.float32), "tensor scale " + tag)
    assert int(flags.item()) == o["flags"], tag


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
def test_block_formats(qat, orc, dt, fmt):
    for i, n in enumerate((32, 256, 4096, 1 << 16)):
        t = torch.from_numpy(make_input(n, 4000 + i + 10 * fmt))
        x = t.to(DT[dt]) if dt != "f32" else t
        for block in (16, 32):
            for kind in (0, 1, 2):
                run_block(qat, orc, x, fmt, block, kind)


def test_block_all_zero_and_named_ops(qat, orc):
    import fake_quant_numerics_gb300 as fq
    z = torch.zeros(1024)
    for kind in (0, 1, 2):
        run_block(qat, orc, z, 4, 16, kind)
    x = torch.from_numpy(make_input(1 << 14, 4100, specials=False))
    r = fq.fake_quant_block(x.cuda(), "e2m1", 16, "e4m3")
    o = orc.fake_quant_block(x.numpy(), 4, 16, 1)
    assert_same(bits(r.y), o["y"].view(np.uint32), "nvfp4 named op")
    with pytest.raises(ValueError):
        fq.fake_quant_block(torch.zeros(40, device="cuda"), "e2m1", 16, "e4m3")
