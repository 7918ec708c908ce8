"""The bench's end-to-end leg pipelines its steps (two device buffer sets,
copies in, calls and copies out on three streams): the outputs it copies back
must be exactly those of the same calls made directly."""
import argparse
import os
import sys

import numpy as np
import pytest
import torch

from gpu_helpers import bits

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_pipelined_e2e_outputs_equal_the_direct_calls(qat):
    import bench

    dev = torch.device("cuda", torch.cuda.current_device())
    inputs = bench.make_inputs(1 / 64)
    suite = bench.Suite(dev, qat, inputs)
    calls = suite.calls()
    for c in calls:
        c()
    torch.cuda.synchronize()
    direct = [bits(t) for t in suite.outputs_for_host()]
    n1, n2, n3, n4, n5 = suite.n
    wb = bench.workload_bytes(n1, suite.r2, suite.c2, n3, suite.r4, suite.c4, n5)
    args = argparse.Namespace(steps=3, e2e_steps=3, only="")
    keep = {}
    r = bench.run_e2e(args, suite, calls, sum(b for _, _, b, _ in wb), keep=keep)
    assert r["value"] > 0 and r["h2d_bytes_per_step"] > 0 and r["d2h_bytes_per_step"] > 0
    for k, (a, h) in enumerate(zip(direct, keep["host_out"])):
        assert np.array_equal(a, bits(h)), f"output {k} differs"
