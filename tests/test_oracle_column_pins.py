"""Pins for per-column channels (the QAT module's per_channel_params /
fake_quant_int_per_channel with axis 1): the module's per-channel example
transposed, and the identity per-column(x) = per-row(x transposed).  CPU only.
"""
import numpy as np

F32 = np.float32
PER_ROW, PER_COLUMN = 1, 3


def test_module_per_channel_example_along_columns(orc):
    # the module's per_channel_scales_differ_and_error_respects_each_scale,
    # with the channels as columns: [[0, 0], [0.5, 50], [1, 100]]
    x = np.array([[0.0, 0.0], [0.5, 50.0], [1.0, 100.0]], F32)
    r = orc.fake_quant_int(x, 3, 2, 8, 0, PER_COLUMN)
    s = r["scale"]
    assert s.size == 2 and s[1] > 10 * s[0]
    assert abs(float(s[0]) - 1 / 127) < 1e-6 and abs(float(s[1]) - 100 / 127) < 1e-6
    err = np.abs(r["y"].reshape(3, 2).astype(np.float64) - x)
    assert np.all(err <= s.astype(np.float64)[None, :] / 2 + 1e-7)
    mn, mx, am, bad = orc.column_stats(x, 3, 2)
    assert list(am) == [1.0, 100.0] and list(mn) == [0.0, 0.0] and not bad.any()


def test_per_column_equals_per_row_of_the_transpose(orc):
    rng = np.random.default_rng(41)
    for rows, cols in ((7, 33), (64, 96), (5, 1)):
        x = (rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-3, 1, size=(1, cols)))).astype(F32)
        x[rng.integers(rows), rng.integers(cols)] = 0.0
        for bits in (8, 4):
            for scheme in (0, 1):
                c = orc.fake_quant_int(x, rows, cols, bits, scheme, PER_COLUMN, want_codes=False)
                t = orc.fake_quant_int(np.ascontiguousarray(x.T), cols, rows, bits, scheme, PER_ROW,
                                       want_codes=False)
                assert np.array_equal(c["scale"], t["scale"])
                assert np.array_equal(c["zero_point"], t["zero_point"])
                assert np.array_equal(c["y"].reshape(rows, cols), t["y"].reshape(cols, rows).T)
                mc = np.unpackbits(c["mask"].view(np.uint8), bitorder="little")[:rows * cols]
                mt = np.unpackbits(t["mask"].view(np.uint8), bitorder="little")[:rows * cols]
                assert np.array_equal(mc.reshape(rows, cols), mt.reshape(cols, rows).T)


def test_per_column_flags_only_the_bad_column(orc):
    x = np.ones((4, 3), F32)
    x[:, 1] = 0.0          # degenerate column
    x[2, 2] = np.nan       # non-finite column
    r = orc.fake_quant_int(x, 4, 3, 8, 0, PER_COLUMN)
    y = r["y"].reshape(4, 3)
    assert np.all(y[:, 0] == 1.0) and np.all(y[:, 1] == 0.0) and np.all(y[:, 2] == 0.0)
    assert r["flags"] == 1 | 2
