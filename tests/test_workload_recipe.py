"""The synthetic input recipe (the five workloads' generators) has the
structure the benchmark and the parity tests claim: distribution parameters,
the outlier columns and special values of the activations, exact bf16
subnormals, and determinism in the seed.  Reduced shapes; CPU only."""
import numpy as np
import torch

from fake_quant_numerics_gb300 import workloads as W


def test_cfg1_standard_normal_pair():
    x, g = W.cfg1(n=1 << 16)
    assert x.dtype == g.dtype == torch.float32 and x.shape == g.shape == (1 << 16,)
    for t in (x, g):
        a = t.numpy().astype(np.float64)
        assert abs(a.mean()) < 0.03 and abs(a.std() - 1.0) < 0.03
    assert not torch.equal(x, g)                  # separate streams


def test_cfg2_row_scales_log_uniform():
    w = W.cfg2(rows=512, cols=1024).numpy().astype(np.float64)
    s = w.std(axis=1)
    # sigma_r in [0.01, 1] (sample std within a few percent of it)
    assert s.min() > 0.01 * 0.9 and s.max() < 1.0 * 1.1
    # log-uniform: about a third of the rows in each decade third
    ls = np.log10(s)
    assert 0.25 < np.mean(ls < -4 / 3) < 0.42 and 0.25 < np.mean(ls > -2 / 3) < 0.42


def test_cfg3_outlier_columns_and_specials():
    rows, cols = 512, 1000
    t = W.cfg3(rows=rows, cols=cols)
    assert t.dtype == torch.bfloat16 and t.shape == (rows, cols)
    bits = W.bf16_bits(t).reshape(rows, cols)
    a = t.float().numpy()
    n = rows * cols
    exp = (bits >> 7) & 0xFF
    man = bits & 0x7F
    nan = (exp == 0xFF) & (man != 0)
    inf = (exp == 0xFF) & (man == 0)
    sub = (exp == 0) & (man != 0)
    big = np.abs(a) == np.float32(999424.0)       # 1e6 rounded to bf16
    neg0 = bits == 0x8000
    # 0.1% of the positions are specials, every kind present
    n_sp = int(round(n * 0.001))
    assert nan.sum() + inf.sum() + sub.sum() + big.sum() <= n_sp
    for m in (nan, inf, sub, big, neg0):
        assert m.sum() > 0
    assert (inf & (a > 0)).sum() > 0 and (inf & (a < 0)).sum() > 0
    # subnormals are exact: m * 2^-133, m in [1, 127]
    assert np.array_equal(a[sub], man[sub].astype(np.float32) * np.float32(2.0 ** -133)
                          * np.where(bits[sub] >> 15, -1, 1).astype(np.float32))
    # 1% of the columns (10 here) carry x50 values: their median |x| stands out
    fin = np.where(np.isfinite(a) & ~big, np.abs(a), np.nan)
    med = np.nanmedian(fin, axis=0)
    hot = med > 10 * np.median(med)
    assert hot.sum() == int(round(cols * 0.01))
    assert 30 < np.median(med[hot]) / np.median(med[~hot]) < 70


def test_cfg4_laplace_weights_and_grads():
    w, g = W.cfg4(rows=256, cols=1024)
    assert w.dtype == g.dtype == torch.bfloat16
    wa = w.float().numpy().astype(np.float64)
    ga = g.float().numpy().astype(np.float64)
    assert abs(np.abs(wa).mean() - 0.02) < 0.001          # Laplace(0, b): E|x| = b
    assert abs(ga.std() - np.sqrt(1e-3)) < 0.001


def test_cfg5_scale_and_determinism():
    x = W.cfg5(n=1 << 16).numpy().astype(np.float64)
    assert abs(x.std() - 0.02) < 0.001
    assert torch.equal(W.cfg5(n=4096), W.cfg5(n=4096))
    assert not torch.equal(W.cfg5(n=4096), W.cfg5(n=4096, seed=99))
    a, b = W.cfg3(rows=64, cols=256), W.cfg3(rows=64, cols=256)
    assert np.array_equal(W.bf16_bits(a), W.bf16_bits(b))
