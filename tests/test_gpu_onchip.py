"""The single-launch per-tensor path and the bounded device waits.

A calibrated per-tensor integer call whose tensor fits in the registers of
the resident blocks runs as one cooperative kernel (statistics, a grid
barrier, then the map from registers); larger tensors take the two-pass path.
Parity is bit for bit against the oracle on both sides of that threshold,
with special values; the launch count shows which path ran.  The barrier and
the per-column kernels' staged-copy waits are bounded: with the testing hook
qat_debug_set_wait_limit(0) every such wait gives up at once, the call
reports QAT_FLAG_DEVICE_TIMEOUT, and the next call (default limit) is exact
again, so the context stays usable."""
import numpy as np
import pytest
import torch

from fake_quant_numerics_gb300 import _lib
from gpu_helpers import assert_same, bits
from test_gpu_parity import make_input, run_int

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
# (rows, cols): one element to the w1 size (one launch), a size that takes 2
# or 4 vectors per thread, and one beyond every resident grid (two launches)
SHAPES = [(1, 1), (1, 7), (1, 33), (1, 1000), (1, 4097), (3, 65549), (1, 1 << 20),
          (1, 3_000_001), (3, 4_000_000)]
BEYOND = 12_000_000  # > 152 SMs x 4 blocks x 512 threads x 4 vectors x 8 fp32


def launches(qat, fn):
    c0 = qat.qat_kernel_launch_count()
    fn()
    torch.cuda.synchronize()
    return qat.qat_kernel_launch_count() - c0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("scheme", [0, 1])
def test_onchip_parity_both_sides_of_the_threshold(qat, orc, dt, bits_, scheme):
    for i, (r, c) in enumerate(SHAPES):
        x = make_input(r, c, DT[dt], seed=6000 + i, specials=(i == 4))
        nl = launches(qat, lambda: run_int(qat, orc, x, r, c, bits_, scheme, 0))
        if r * c <= (1 << 20):
            assert nl == 1, (r, c, nl)
        else:
            assert nl in (1, 2), (r, c, nl)


def test_onchip_beyond_the_resident_grid_takes_two_launches(qat, orc):
    x = make_input(1, BEYOND, torch.float32, seed=6100)
    assert launches(qat, lambda: run_int(qat, orc, x, 1, BEYOND, 8, 0, 0)) == 2


@pytest.mark.parametrize("scheme", [0, 1])
def test_onchip_degenerate_and_nonfinite(qat, orc, scheme):
    """A NaN anywhere makes the tensor a failed calibration (codes 0, y +0,
    mask 0, the flag); all zeros is degenerate; +-inf alone is non-finite."""
    n = 300_001
    for case in ("nan", "zeros", "inf"):
        a = np.random.default_rng(6200).standard_normal(n).astype(np.float32)
        if case == "nan":
            a[n // 2] = np.nan
        elif case == "zeros":
            a[:] = 0.0
        else:
            a[7] = -np.inf
        for dt in ("f32", "bf16"):
            t = torch.from_numpy(a.copy())
            x = t.to(DT[dt]) if dt != "f32" else t
            o = run_int(qat, orc, x, 1, n, 8, scheme, 0)
            assert o["flags"] != 0


def test_onchip_call_replayed_in_a_cuda_graph(qat, orc):
    """The clear of the barrier counter and the cooperative kernel captured
    in one graph: every replay on new contents of x is exact."""
    n = (1 << 20) + 5
    dev = "cuda"
    x = torch.zeros(n, device=dev)
    y = torch.empty(n, device=dev)
    codes = torch.empty(n, dtype=torch.int8, device=dev)
    mask = torch.empty((n + 31) // 32, dtype=torch.int32, device=dev)
    sc = torch.empty(1, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(qat.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device=dev)

    def call():
        qat.qat_fake_quant_int(x, 1, n, 8, 0, 0, 0, False, sc, None, y, codes, mask, flags, ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for seed in (1, 2, 3):
        a = (np.random.default_rng(6300 + seed).standard_normal(n) * seed).astype(np.float32)
        x.copy_(torch.from_numpy(a))
        flags.zero_()
        g.replay()
        torch.cuda.synchronize()
        o = orc.fake_quant_int(a, 1, n, 8, 0, 0)
        assert_same(bits(y), o["y"].view(np.uint32), f"y replay {seed}")
        assert_same(bits(codes), o["codes"].view(np.uint8), f"codes replay {seed}")
        assert_same(bits(mask), o["mask"], f"mask replay {seed}")
        assert_same(bits(sc), o["scale"].view(np.uint32), f"scale replay {seed}")
        assert int(flags.item()) == 0


def _wait_limit(polls):
    _lib.load().qat_debug_set_wait_limit(polls)


@pytest.mark.parametrize("case", ["tensor", "column"])
def test_bounded_wait_runs_out_and_the_context_stays_usable(qat, orc, case):
    """Every bounded wait given no polls: the grid barrier of the single-launch
    per-tensor path, or the staged-copy waits of the per-column statistics and
    map kernels (each block first drains the copies it issued).  The call
    returns OK with QAT_FLAG_DEVICE_TIMEOUT; the same call with the default
    limit is then exact."""
    rows, cols, gran = (1, 1 << 20, 0) if case == "tensor" else (512, 256, 3)
    n = rows * cols
    x = make_input(rows, cols, torch.float32, seed=6400)
    xd = x.cuda()
    dev = "cuda"
    units = 1 if gran == 0 else cols
    y = torch.empty(n, device=dev)
    codes = torch.empty(n, dtype=torch.int8, device=dev)
    mask = torch.empty((n + 31) // 32, dtype=torch.int32, device=dev)
    sc = torch.empty(units, device=dev)
    zp = torch.empty(units, dtype=torch.int32, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(qat.qat_workspace_bytes(rows, cols, gran, 0), dtype=torch.uint8, device=dev)
    try:
        _wait_limit(0)
        qat.qat_fake_quant_int(xd, rows, cols, 8, 1, gran, 0, False, sc, zp, y, codes, mask, flags,
                               ws)
        torch.cuda.synchronize()
        assert int(flags.item()) & _lib.FLAG_DEVICE_TIMEOUT
    finally:
        _wait_limit(-1)
    o = run_int(qat, orc, x, rows, cols, 8, 1, gran)
    assert not (o["flags"] & _lib.FLAG_DEVICE_TIMEOUT)
