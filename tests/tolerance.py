"""Tolerance of an fp32 (or bf16) fake-quant output against the binary64
evaluation of the same formulas.

Derivation (int grids): y = k * scale with k an integer, |k| <= 255.  In fp32
the scale carries up to two roundings (range subtraction, division), each
<= 2^-24 relative, and the product one more, so for a given k
|y32 - y64| <= 3 * 2^-24 * |y64| (+ half an output ulp when the output is bf16).
A stated floor of 1e-6 * scale is kept on top.  Where x/scale lies so close to a
half-integer that the fp32 and f64 quotients can round to different integers,
k may differ by one: such "tie-adjacent" elements may differ by one grid step
(plus the output rounding of that neighbour) and are counted separately.
With bf16 inputs exact rational ties (x / scale = k + 1/2 exactly, e.g.
x = absmax / 2 in int4) are common, so the count is reported, not bounded
tightly.
"""
import numpy as np

U24 = 2.0 ** -24


def half_ulp_bf16(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def int_check(y_out, y64, x, scale64, out_bf16: bool):
    """Returns (ok, n_tie_adjacent).  All arrays float64, broadcast-compatible."""
    q = x / scale64
    frac = np.abs(q - np.floor(q) - 0.5)
    tie = frac <= 4 * U24 * np.abs(q) + 2.0 ** -23
    tol = 1e-6 * scale64 + 3 * U24 * np.abs(y64)
    if out_bf16:
        tol = tol + half_ulp_bf16(y64)
    d = np.abs(y_out - y64)
    ok_main = d <= tol
    tol_tie = scale64 + tol
    if out_bf16:
        tol_tie = tol_tie + half_ulp_bf16(y_out)
    ok_tie = d <= tol_tie
    ok = np.where(tie, ok_tie, ok_main)
    return bool(np.all(ok)), int(np.count_nonzero(tie & ~ok_main))
