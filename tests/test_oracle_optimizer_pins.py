"""Pins for the oracle's QAT optimizer step (QatOptimizer::step: Adam/AdamW
update of the master weights, then the fake-quant view re-derived from them).

The update is checked against an independent library implementation of the
same algorithm (torch.optim.Adam / AdamW in float64), against Adam's closed
form for a first step, and against the decoupled weight decay alone; the view
against the module's own optimizer tests (the view tracks the master, lies on
the grid, the master stays off it).  CPU only.
"""
import numpy as np
import pytest
import torch

F32 = np.float32


def ulp(a):
    return np.spacing(np.abs(np.asarray(a, F32))).astype(np.float64)


def test_module_example_int8_view_tracks_master(orc):
    # the module's qat_master_update_keeps_fp32_master_and_quantized_view_tracks_it
    w0 = np.array([0.12, -0.37, 0.88, -0.05, 0.51], F32)
    g = np.array([0.1, -0.2, 0.05, 0.3, -0.15], F32)
    z = np.zeros(5, F32)
    r = orc.qat_optimizer_step(w0, g, z, z, lr=0.1, bits=8, scheme=0)
    assert np.any(np.abs(r["w"] - w0) > 1e-9)  # the master moved
    ref = orc.fake_quant_int(r["w"], 1, 5, 8, 0, 0)  # independent fake quant of the master
    assert np.array_equal(r["view"], ref["y"]) and r["scale"] == ref["scale"][0]
    # the view is on the grid: every element is RN(k * scale) for an integer k
    codes = np.round(r["view"].astype(np.float64) / float(r["scale"])).astype(F32)
    assert np.array_equal(r["view"], codes * r["scale"])
    off = r["w"].astype(np.float64) / float(r["scale"])
    assert np.any(np.abs(off - np.round(off)) > 1e-6)  # the master is not


def test_module_example_fp8_view_tracks_master(orc):
    # the module's qat_fp8_target_tracks_master: the view is the unscaled cast
    w0 = np.array([0.3, -1.2, 4.0, -0.01, 2.5], F32)
    g = np.array([0.2, 0.1, -0.3, 0.4, -0.05], F32)
    z = np.zeros(5, F32)
    r = orc.qat_optimizer_step(w0, g, z, z, lr=0.05, bits=0, fmt=0)
    ref = orc.fake_quant_fp8(r["w"], 0, scale=1.0)
    assert np.array_equal(r["view"], ref["y"]) and r["scale"] == 1.0
    assert np.array_equal(r["codes"], ref["codes"])


@pytest.mark.parametrize("wd", [0.0, 0.01])
def test_update_matches_torch_adam(orc, wd):
    """Five steps against torch.optim.Adam (wd = 0) / AdamW in float64."""
    rng = np.random.default_rng(31)
    # the oracle's hyper-parameters are binary32: hand torch the same values
    n, lr, b1, b2, eps = (4096,) + tuple(float(F32(h)) for h in (1e-3, 0.9, 0.999, 1e-8))
    wd = float(F32(wd))
    w = (rng.standard_normal(n) * 0.05).astype(F32)
    m = np.zeros(n, F32)
    v = np.zeros(n, F32)
    p = torch.nn.Parameter(torch.from_numpy(w.astype(np.float64)))
    opt = (torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd) if wd
           else torch.optim.Adam([p], lr=lr, betas=(b1, b2), eps=eps))
    for t in range(1, 6):
        g = (rng.standard_normal(n) * 1e-2).astype(F32)
        bc1, bc2 = orc.bias_corrections(b1, b2, t)
        w, m, v = orc.adam_update(w, g, m, v, lr, b1, b2, eps, wd, bc1, bc2)
        p.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
        st = opt.state[p]
        ref_w = p.detach().numpy()
        # binary32 state: a few ulps of the weight per step, plus the update's
        # relative rounding (< 1e-5 of lr)
        assert np.all(np.abs(w - ref_w) <= 4 * t * ulp(ref_w) + 1e-5 * lr * t), t
        # the moments: binary32 roundings of terms of the size of the largest
        # moment (beta1 m and (1 - beta1) g can cancel, so no relative bound)
        mr, vr = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        assert np.all(np.abs(m - mr) <= 1e-6 * np.abs(mr).max())
        assert np.all(np.abs(v - vr) <= 1e-6 * np.abs(vr).max())


def test_first_step_closed_form(orc):
    # from zero moments with eps = 0: m_hat = g, v_hat = g^2, so the update is
    # lr * sign(g) (up to the roundings of the moments and the bias corrections)
    rng = np.random.default_rng(32)
    w = rng.standard_normal(1000).astype(F32)
    g = (rng.standard_normal(1000) * 0.3).astype(F32)
    g[g == 0] = F32(0.1)
    z = np.zeros(1000, F32)
    bc1, bc2 = orc.bias_corrections(0.9, 0.999, 1)
    w1, _, _ = orc.adam_update(w, g, z, z, 0.01, 0.9, 0.999, 0.0, 0.0, bc1, bc2)
    step = w.astype(np.float64) - w1.astype(np.float64)
    assert np.all(np.abs(step - 0.01 * np.sign(g)) <= ulp(w1) + 1e-7)


def test_decoupled_weight_decay_alone(orc):
    # zero gradient and moments: the Adam term is 0 / (0 + eps) = 0 and the
    # step is the decay w - (lr wd) w alone, exactly
    w = np.array([1.0, -3.5, 1e-3, 0.0, -0.0, 7e-30, 123.0], F32)
    z = np.zeros(w.size, F32)
    bc1, bc2 = orc.bias_corrections(0.9, 0.999, 3)
    w1, m1, v1 = orc.adam_update(w, z, z, z, 0.1, 0.9, 0.999, 1e-8, 0.2, bc1, bc2)
    assert np.array_equal(w1, w - F32(F32(0.1) * F32(0.2)) * w)
    assert np.all(m1 == 0) and np.all(v1 == 0)
    w2, _, _ = orc.adam_update(w, z, z, z, 0.1, 0.9, 0.999, 1e-8, 0.0, bc1, bc2)
    assert np.array_equal(w2, w)  # no decay, no gradient: no change


def test_view_targets_and_rounding(orc):
    rng = np.random.default_rng(33)
    n = 3000
    w = (rng.standard_normal(n) * 0.1).astype(F32)
    g = (rng.standard_normal(n) * 0.01).astype(F32)
    m = (rng.standard_normal(n) * 0.001).astype(F32)
    v = (rng.random(n) * 1e-4).astype(F32)
    for bits, scheme in ((8, 0), (8, 1), (4, 0), (4, 1)):
        for sr in (False, True):
            r = orc.qat_optimizer_step(w, g, m, v, lr=1e-3, weight_decay=0.01, step=7, bits=bits,
                                       scheme=scheme, stochastic=sr, seed=11, offset=5)
            if sr:
                ref = orc.fake_quant_int_sr(r["w"], 1, n, bits, scheme, 0, seed=11, offset=5)
            else:
                ref = orc.fake_quant_int(r["w"], 1, n, bits, scheme, 0)
            assert np.array_equal(r["view"], ref["y"]) and np.array_equal(r["mask"], ref["mask"])
            assert r["scale"] == ref["scale"][0] and r["zero_point"] == ref["zero_point"][0]
    for fmt in (0, 1):
        r = orc.qat_optimizer_step(w, g, m, v, lr=1e-3, step=2, bits=0, fmt=fmt, stochastic=True,
                                   seed=3, offset=0)
        ref = orc.fake_quant_fp8_sr(r["w"], fmt, seed=3, offset=0, scale=1.0)
        assert np.array_equal(r["view"], ref["y"])
