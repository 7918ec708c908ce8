"""GPU parity of the QAT optimizer step (qat_optimizer_step) against the
oracle: master, moments, view, codes, mask, scale, zero point and flags bit
for bit over consecutive steps, for every view target and both roundings.
"""
import numpy as np
import pytest
import torch

import fake_quant_numerics_gb300 as fq
from gpu_helpers import assert_same, bits

pytestmark = pytest.mark.gpu

F32 = np.float32
TARGETS = [(8, 0, 0), (8, 1, 0), (4, 0, 0), (4, 1, 0), (0, 0, 0), (0, 0, 1)]  # (bits, scheme, fmt)


def assert_state(gpu_t, ref, what):
    """Optimizer state (master, moments): bit patterns, except that a NaN
    matches any NaN (arithmetic NaN payloads are not canonicalised in state)."""
    g = bits(gpu_t).view(np.float32)
    both_nan = np.isnan(g) & np.isnan(ref)
    assert_same(np.where(both_nan, np.float32(0), g), np.where(both_nan, np.float32(0), ref), what)


def gpu_state(w, m, v):
    return [torch.from_numpy(a.copy()).cuda() for a in (w, m, v)]


def run_steps(orc, n, bits_, scheme, fmt, stochastic, wd, seed, steps=3):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal(n) * 0.05).astype(F32)
    m = (rng.standard_normal(n) * 1e-3).astype(F32)
    v = (rng.random(n) * 1e-5).astype(F32)
    W, M, V = gpu_state(w, m, v)
    lr, b1, b2, eps = 1e-3, 0.9, 0.999, 1e-8
    for t in range(1, steps + 1):
        g = (rng.standard_normal(n) * 1e-2).astype(F32)
        off = 1000 * t
        o = orc.qat_optimizer_step(w, g, m, v, lr=lr, beta1=b1, beta2=b2, eps=eps,
                                   weight_decay=wd, step=t, bits=bits_, scheme=scheme, fmt=fmt,
                                   stochastic=stochastic, seed=seed, offset=off)
        target = {8: "int8", 4: "int4"}.get(bits_, "e4m3" if fmt == 0 else "e5m2")
        r = fq.optimizer_step(W, torch.from_numpy(g).cuda(), M, V, t, lr, (b1, b2), eps, wd,
                              target=target, scheme=("affine" if scheme else "symmetric"),
                              rounding="stochastic" if stochastic else "nearest", seed=seed,
                              offset=off, want_codes=True, want_mask=True)
        torch.cuda.synchronize()
        tag = f"n={n} bits={bits_} scheme={scheme} fmt={fmt} sr={stochastic} wd={wd} step={t}"
        assert_state(W, o["w"], "master " + tag)
        assert_state(M, o["m"], "exp_avg " + tag)
        assert_state(V, o["v"], "exp_avg_sq " + tag)
        assert_same(bits(r.view), o["view"], "view " + tag)
        assert_same(bits(r.codes)[:o["codes"].size], o["codes"].view(np.uint8), "codes " + tag)
        assert_same(bits(r.mask), o["mask"], "mask " + tag)
        assert_same(bits(r.scale), np.array([o["scale"]], F32), "scale " + tag)
        if bits_ and scheme:
            assert int(r.zero_point.item()) == o["zero_point"], tag
        assert int(r.flags.item()) == o["flags"], tag
        w, m, v = o["w"], o["m"], o["v"]


@pytest.mark.parametrize("bits_,scheme,fmt", TARGETS)
def test_optimizer_step_parity(orc, bits_, scheme, fmt):
    for i, n in enumerate((1, 7, 1000, 1024, 33333, (1 << 20) + 5)):
        for stochastic in (False, True):
            run_steps(orc, n, bits_, scheme, fmt, stochastic, wd=0.01 if i % 2 else 0.0,
                      seed=900 + i)


def test_optimizer_step_nonfinite_master_flags_int_view(orc):
    n = 5000
    rng = np.random.default_rng(9)
    w = (rng.standard_normal(n) * 0.05).astype(F32)
    z = np.zeros(n, F32)
    g = (rng.standard_normal(n) * 1e-2).astype(F32)
    g[1234] = np.nan
    W, M, V = gpu_state(w, z, z)
    r = fq.optimizer_step(W, torch.from_numpy(g).cuda(), M, V, 1, 1e-3, want_codes=True,
                          want_mask=True)
    torch.cuda.synchronize()
    o = orc.qat_optimizer_step(w, g, z, z, lr=1e-3, step=1, bits=8)
    assert o["flags"] & 1 and int(r.flags.item()) == o["flags"]
    assert_state(W, o["w"], "master with NaN")
    assert_same(bits(r.view), o["view"], "view of a flagged master")
    with pytest.raises(fq.QatDataError):
        fq.raise_on_flags(r.flags)
