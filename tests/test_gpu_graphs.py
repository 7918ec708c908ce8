"""Calls whose kernels are chained by programmatic dependent launch, captured
in a CUDA graph and replayed on new contents of x: every replay must equal
the oracle bit for bit.  The chains: per-tensor FP8 (statistics, map),
per-tensor int beyond the single-read size (statistics, map), percentile
calibration (reset, three passes, map), per-column (reset, statistics, map)
and NVFP4 (statistics, block map)."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_same, bits

pytestmark = pytest.mark.gpu


def replay_check(make_call, fill, oracle, outputs, seeds=(1, 2, 3)):
    """make_call() issues the call on the current stream; fill(seed) writes new
    inputs in place and returns their host copy; oracle(host) returns the
    expected outputs (same order as `outputs`)."""
    fill(0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        make_call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        make_call()
    for seed in seeds:
        host = fill(seed)
        g.replay()
        torch.cuda.synchronize()
        for k, (got, want) in enumerate(zip(outputs, oracle(host))):
            assert_same(bits(got), want, f"output {k} replay {seed}")


def test_fp8_and_large_int_per_tensor_in_a_graph(qat, orc):
    n = 12_000_000 + 7  # beyond the single-read per-tensor path
    x = torch.empty(n, device="cuda")
    y = torch.empty(n, device="cuda")
    m = torch.empty((n + 31) // 32, dtype=torch.int32, device="cuda")
    codes = torch.empty(n, dtype=torch.int8, device="cuda")
    sc = torch.empty(1, device="cuda")
    fl = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(qat.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device="cuda")

    def fill(seed):
        a = (np.random.default_rng(8000 + seed).standard_normal(n) * (seed + 1)).astype(np.float32)
        x.copy_(torch.from_numpy(a))
        return a

    replay_check(lambda: qat.qat_fake_quant_fp8(x, n, 0, False, sc, y, None, m, fl, ws), fill,
                 lambda a: (lambda o: (o["y"].view(np.uint32), o["mask"],
                                       np.array([o["scale"]], np.float32).view(np.uint32)))(
                     orc.fake_quant_fp8(a, 0)), (y, m, sc))
    replay_check(lambda: qat.qat_fake_quant_int(x, 1, n, 8, 1, 0, 0, False, sc, None, y, codes, m,
                                                fl, ws), fill,
                 lambda a: (lambda o: (o["y"].view(np.uint32), o["codes"].view(np.uint8),
                                       o["mask"]))(orc.fake_quant_int(a, 1, n, 8, 1, 0)),
                 (y, codes, m))


def test_percentile_and_columns_in_a_graph(qat, orc):
    rows, cols = 512, 1024
    n = rows * cols
    x = torch.empty(n, device="cuda")
    y = torch.empty(n, device="cuda")
    m = torch.empty(n // 32, dtype=torch.int32, device="cuda")
    sc = torch.empty(cols, device="cuda")
    zp = torch.empty(cols, dtype=torch.int32, device="cuda")
    fl = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsp = torch.empty(qat.qat_percentile_workspace_bytes(), dtype=torch.uint8, device="cuda")
    wsc = torch.empty(qat.qat_workspace_bytes(rows, cols, 3, 0), dtype=torch.uint8, device="cuda")

    def fill(seed):
        rng = np.random.default_rng(8100 + seed)
        a = (rng.standard_t(3, size=n) * (0.5 + seed)).astype(np.float32)
        x.copy_(torch.from_numpy(a))
        return a

    replay_check(lambda: qat.qat_fake_quant_int_percentile(x, n, 8, 0, 0.001, False, 0, 0, sc[:1],
                                                           None, y, None, m, fl, wsp), fill,
                 lambda a: (lambda o: (o["y"].view(np.uint32), o["mask"]))(
                     orc.fake_quant_int_percentile(a, 8, 0, 0.001)), (y, m))
    replay_check(lambda: qat.qat_fake_quant_int(x, rows, cols, 8, 1, 3, 0, False, sc, zp, y, None,
                                                m, fl, wsc), fill,
                 lambda a: (lambda o: (o["y"].view(np.uint32), o["mask"],
                                       o["scale"].view(np.uint32)))(
                     orc.fake_quant_int(a, rows, cols, 8, 1, 3)), (y, m, sc))


def test_nvfp4_in_a_graph(qat, orc):
    n = 1 << 20
    x = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    codes = torch.empty(n // 2, dtype=torch.uint8, device="cuda")
    bs = torch.empty(n // 16, dtype=torch.uint8, device="cuda")
    m = torch.empty(n // 32, dtype=torch.int32, device="cuda")
    g = torch.empty(1, device="cuda")
    fl = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(qat.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device="cuda")

    def fill(seed):
        rng = np.random.default_rng(8200 + seed)
        a = torch.from_numpy((rng.standard_t(5, size=n) * 0.02 * (seed + 1)).astype(np.float32))
        xb = a.to(torch.bfloat16)
        x.copy_(xb)
        return xb.view(torch.int16).numpy().view(np.uint16)

    def expect(a):
        o = orc.fake_quant_block(a, 4, 16, 1)
        oc = o["codes"]
        packed = ((oc[0::2] & 0xF) << 4 | (oc[1::2] & 0xF)).astype(np.uint8)  # 2j high
        return o["y"], packed, o["bscales"], o["mask"]

    replay_check(lambda: qat.qat_fake_quant_block(x, n, 4, 16, 1, g, y, codes, bs, m, fl, ws), fill,
                 expect, (y, codes, bs, m))
