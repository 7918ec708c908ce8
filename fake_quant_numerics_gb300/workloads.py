"""Seeded synthetic inputs for the five fake-quant workloads.

This module only draws random numbers; it holds none of the quantization
arithmetic, so the CUDA library's tests, the CPU oracle and the benchmark can
all take their inputs from it.  Every generator is a pure function of its seed
and shape (numpy ``default_rng`` / PCG64 streams, keyed by ``[seed, stream]``).

bf16 tensors are drawn in fp32 and rounded once to bf16 (round to nearest
even, via torch's CPU conversion); they are returned as torch ``bfloat16``
tensors whose raw ``uint16`` bits are what the oracle reads.

Workloads (full sizes; every generator also takes smaller shapes with the same
distribution, for parity tests and the CPU baseline):

1. per-tensor symmetric int8, fwd + STE bwd: x fp32 [1,048,576] ~ N(0,1),
   upstream grad fp32 ~ N(0,1).
2. per-row affine int8 and symmetric int4: fp32 weight [4096, 4096], row r
   ~ N(0, sigma_r^2) with sigma_r log-uniform in [0.01, 1].
3. per-tensor amax-scaled FP8 (E4M3 and E5M2): bf16 activations [8192, 8192]
   ~ 0.5 * Student-t(nu=3), 1% of the columns scaled x50 (outlier channels),
   0.1% of the positions replaced by specials drawn uniformly from
   {+0, -0, +sub, -sub, +1e6, -1e6, +Inf, -Inf, NaN} (sub = an fp32/bf16
   subnormal m * 2^-133, m uniform in [1, 127]).
4. per-group (128 along the last dim) symmetric int4: bf16 weight
   [14336, 4096] ~ Laplace(0, 0.02); bf16 upstream grad ~ N(0, 1e-3)
   (variance 1e-3).
5. QLoRA two-level 4-bit: fp32 flat [268,435,456] ~ N(0, 0.02^2).
"""
from __future__ import annotations

import numpy as np
import torch

FULL_SHAPES = {
    1: (1, 1 << 20),
    2: (4096, 4096),
    3: (8192, 8192),
    4: (14336, 4096),
    5: (1, 268_435_456),
}
SEEDS = {1: 0, 2: 1, 3: 2, 4: 3, 5: 4}
GROUP = 128


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """fp32 numpy -> torch.bfloat16 (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a CPU bf16 tensor."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def cfg1(n: int = 1 << 20, seed: int = SEEDS[1]):
    x = _rng(seed, 0).standard_normal(n, dtype=np.float32)
    g = _rng(seed, 1).standard_normal(n, dtype=np.float32)
    return torch.from_numpy(x), torch.from_numpy(g)


def cfg2(rows: int = 4096, cols: int = 4096, seed: int = SEEDS[2]):
    r = _rng(seed, 0)
    sigma = np.exp(r.uniform(np.log(0.01), np.log(1.0), size=(rows, 1))).astype(np.float32)
    w = r.standard_normal((rows, cols), dtype=np.float32) * sigma
    return torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32))


SPECIAL_KINDS = ("+0", "-0", "+sub", "-sub", "+1e6", "-1e6", "+inf", "-inf", "nan")


def cfg3(rows: int = 8192, cols: int = 8192, seed: int = SEEDS[3], outlier_frac: float = 0.01,
         special_frac: float = 0.001):
    r = _rng(seed, 0)
    a = (0.5 * r.standard_t(3.0, size=(rows, cols))).astype(np.float32)
    n_out = int(round(cols * outlier_frac))
    out_cols = r.permutation(cols)[:n_out]
    a[:, out_cols] *= np.float32(50.0)
    flat = a.reshape(-1)
    n_sp = int(round(flat.size * special_frac))
    if n_sp:
        pos = r.choice(flat.size, size=n_sp, replace=False)
        kind = r.integers(0, len(SPECIAL_KINDS), size=n_sp)
        m = r.integers(1, 128, size=n_sp).astype(np.float32)
        sub = m * np.float32(2.0 ** -133)
        vals = np.select(
            [kind == 0, kind == 1, kind == 2, kind == 3, kind == 4, kind == 5, kind == 6, kind == 7],
            [np.float32(0.0), np.float32(-0.0), sub, -sub, np.float32(1e6), np.float32(-1e6),
             np.float32(np.inf), np.float32(-np.inf)],
            default=np.float32(np.nan)).astype(np.float32)
        # np.select drops the sign of -0.0 through the default broadcast; set it explicitly
        vals[kind == 1] = np.float32(-0.0)
        flat[pos] = vals
    return to_bf16(a)


def cfg4(rows: int = 14336, cols: int = 4096, seed: int = SEEDS[4]):
    r = _rng(seed, 0)
    w = r.laplace(0.0, 0.02, size=(rows, cols)).astype(np.float32)
    g = (_rng(seed, 1).standard_normal((rows, cols), dtype=np.float32)
         * np.float32(np.sqrt(1e-3)))
    return to_bf16(w), to_bf16(g)


def cfg5(n: int = 268_435_456, seed: int = SEEDS[5]):
    x = _rng(seed, 0).standard_normal(n, dtype=np.float32)
    x *= np.float32(0.02)
    return torch.from_numpy(x)
