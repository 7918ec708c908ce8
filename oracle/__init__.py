"""CPU oracle for the fake-quant / STE / 4-bit double-quant path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never calls it and shares no code with it.

The arithmetic lives in ``qat_oracle.c`` (plain single-threaded loops, binary32
with no FMA contraction, plus a binary64 twin); this module only compiles it
with gcc and marshals numpy arrays through ctypes.  bf16 data is passed as its
raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qat_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fno-strict-aliasing",
           "-shared", "-fPIC"]

F32, BF16 = 0, 1
SYM, AFFINE = 0, 1
PER_TENSOR, PER_ROW, PER_GROUP, PER_COLUMN = 0, 1, 2, 3
E4M3, E5M2 = 0, 1
FLAG_NONFINITE, FLAG_DEGENERATE, FLAG_BAD_PARAMS, FLAG_NONFINITE_INPUT = 1, 2, 4, 8
FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}

_lib = None


def build(force: bool = False) -> str:
    """Compile ``qat_oracle.c`` into ``liboracle.so`` next to it (gcc)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        L.or_fake_quant_int.argtypes = [vp, i32, i64, i64, i32, i32, i32, i64, i32, vp, vp, vp, vp,
                                        vp, vp, i32]
        L.or_fake_quant_fp8.argtypes = [vp, i32, i64, i32, i32, vp, vp, vp, vp, vp]
        L.or_ste_backward.argtypes = [vp, i32, i64, vp, vp]
        L.or_quant4_double.argtypes = [vp, i64, vp, vp, vp, vp]
        L.or_dequant4_double.argtypes = [vp, vp, vp, i64, vp]
        L.or_quant4_single.argtypes = [vp, i64, vp, vp]
        L.or_dequant4_single.argtypes = [vp, vp, i64, vp]
        L.or_q4d_memory_bytes.argtypes = [i64]
        L.or_q4d_memory_bytes.restype = i64
        L.or_fp8_cast.argtypes = [f32, i32]
        L.or_fp8_cast.restype = f32
        L.or_fp8_encode.argtypes = [f32, i32]
        L.or_fp8_encode.restype = ctypes.c_uint8
        L.or_quantize.argtypes = [f32, f32, i32, i32, i32, i32]
        L.or_quantize.restype = i32
        L.or_dequantize.argtypes = [i32, f32, i32]
        L.or_dequantize.restype = f32
        L.or_q_range.argtypes = [i32, i32, vp, vp]
        L.or_params_from_absmax.argtypes = [f32, i32, vp]
        L.or_params_affine.argtypes = [f32, f32, i32, i32, vp, vp]
        L.or_reconstruct_scale.argtypes = [ctypes.c_uint8, f32]
        L.or_reconstruct_scale.restype = f32
        L.or64_fake_quant_int.argtypes = [vp, i32, i64, i64, i32, i32, i32, i64, vp, vp, vp]
        L.or64_fake_quant_fp8.argtypes = [vp, i32, i64, i32, vp, vp]
        L.or_unit_stats.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp]
        L.or_unit_stats_strided.argtypes = [vp, i32, i64, i64, i64, vp, vp, vp, vp]
        u64 = ctypes.c_uint64
        L.or_philox4x32_10.argtypes = [vp, vp, vp]
        L.or_sr_uniform.argtypes = [u64, u64, i64]
        L.or_sr_uniform.restype = f32
        L.or_sr_round.argtypes = [f32, f32]
        L.or_sr_round.restype = f32
        L.or_quantize_sr.argtypes = [f32, f32, i32, i32, i32, f32]
        L.or_quantize_sr.restype = i32
        L.or_fp8_cast_sr.argtypes = [f32, i32, f32]
        L.or_fp8_cast_sr.restype = f32
        L.or_fake_quant_int_sr.argtypes = [vp, i32, i64, i64, i32, i32, i32, i64, i32, vp, vp, u64,
                                           u64, vp, vp, vp, vp]
        L.or_fake_quant_fp8_sr.argtypes = [vp, i32, i64, i32, i32, vp, u64, u64, vp, vp, vp, vp]
        L.or_adam_update.argtypes = [vp, vp, vp, vp, i64, f32, f32, f32, f32, f32, f32, f32]
        L.or_qat_optimizer_step.argtypes = [vp, vp, vp, vp, i64, f32, f32, f32, f32, f32, f32, f32,
                                            i32, i32, i32, i32, u64, u64, vp, vp, vp, vp, vp, vp]
        L.or_elem_round.argtypes = [f32, i32]
        L.or_elem_round.restype = f32
        L.or_elem_encode.argtypes = [f32, i32]
        L.or_elem_encode.restype = ctypes.c_uint8
        L.or_elem_decode.argtypes = [ctypes.c_uint8, i32]
        L.or_elem_decode.restype = f32
        L.or_fake_quant_block.argtypes = [vp, i32, i64, i32, i64, i32, vp, vp, vp, vp, vp, vp]
        L.or_round_fp16.argtypes = [f32]
        L.or_round_fp16.restype = f32
        L.or_fake_quant_int_opts.argtypes = [vp, i32, i64, i64, i32, i32, i32, i64, f32, i32, i32,
                                             u64, u64, vp, vp, vp, vp, vp, vp]
        f64 = ctypes.c_double
        L.or_percentile_minmax.argtypes = [vp, i32, i64, f64, vp, vp, vp]
        L.or_fake_quant_int_percentile.argtypes = [vp, i32, i64, i32, i32, f64, i32, u64, u64, vp,
                                                   vp, vp, vp, vp, vp]
    return _lib


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:
        return BF16
    raise TypeError("oracle inputs are float32 arrays or uint16 bf16 bit patterns")


def unit_stats(x: np.ndarray, L: int):
    """(min, max, absmax, nonfinite count) of each run of L elements (finite values only)."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    u = x.size // L if L else 0
    out = np.zeros((u, 3), np.float32)
    bad = np.zeros(u, np.int64)
    mn, mx, am, nb = ctypes.c_float(), ctypes.c_float(), ctypes.c_float(), ctypes.c_int64()
    for k in range(u):
        lib().or_unit_stats(_p(x), dt, k * L, L, ctypes.byref(mn), ctypes.byref(mx), ctypes.byref(am),
                            ctypes.byref(nb))
        out[k] = (mn.value, mx.value, am.value)
        bad[k] = nb.value
    return out[:, 0], out[:, 1], out[:, 2], bad


def column_stats(x: np.ndarray, rows: int, cols: int):
    """(min, max, absmax, nonfinite count) of each column of a row-major
    [rows, cols] tensor (finite values only)."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    out = np.zeros((cols, 3), np.float32)
    bad = np.zeros(cols, np.int64)
    mn, mx, am, nb = ctypes.c_float(), ctypes.c_float(), ctypes.c_float(), ctypes.c_int64()
    for c in range(cols):
        lib().or_unit_stats_strided(_p(x), dt, c, rows, cols, ctypes.byref(mn), ctypes.byref(mx),
                                    ctypes.byref(am), ctypes.byref(nb))
        out[c] = (mn.value, mx.value, am.value)
        bad[c] = nb.value
    return out[:, 0], out[:, 1], out[:, 2], bad


def q_range(bits: int, scheme: int):
    lo, hi = ctypes.c_int32(), ctypes.c_int32()
    st = lib().or_q_range(bits, scheme, ctypes.byref(lo), ctypes.byref(hi))
    if st:
        raise ValueError(f"unsupported: bits={bits} scheme={scheme} (status {st})")
    return lo.value, hi.value


def params_from_absmax(absmax: float, qmax: int):
    s = ctypes.c_float()
    flag = lib().or_params_from_absmax(absmax, qmax, ctypes.byref(s))
    return s.value, flag


def params_affine(mn: float, mx: float, qmin: int, qmax: int):
    s, z = ctypes.c_float(), ctypes.c_int32()
    flag = lib().or_params_affine(mn, mx, qmin, qmax, ctypes.byref(s), ctypes.byref(z))
    return s.value, z.value, flag


def quantize(x: float, scale: float, zp: int, qmin: int, qmax: int, doc_form: bool = True) -> int:
    return lib().or_quantize(x, scale, zp, qmin, qmax, int(doc_form))


def dequantize(q: int, scale: float, zp: int) -> float:
    return lib().or_dequantize(q, scale, zp)


def n_units(rows: int, cols: int, granularity: int, group: int = 0) -> int:
    if granularity == PER_TENSOR:
        return 1 if rows * cols > 0 else 0
    if granularity == PER_ROW:
        return rows
    if granularity == PER_COLUMN:
        return cols if rows > 0 else 0
    return rows * cols // group


def fake_quant_int(x: np.ndarray, rows: int, cols: int, bits: int, scheme: int, granularity: int,
                   group: int = 0, scale=None, zero_point=None, want_y=True, want_codes=True,
                   want_mask=True, doc_form: bool = True):
    """Returns dict(y, codes, mask, scale, zero_point, flags)."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    n = rows * cols
    u = n_units(rows, cols, granularity, group) if (granularity != PER_GROUP or group > 0) else 0
    given = scale is not None
    sc = np.ascontiguousarray(scale, dtype=np.float32).copy() if given else np.zeros(max(u, 1), np.float32)
    zp = (np.ascontiguousarray(zero_point, dtype=np.int32).copy() if zero_point is not None
          else np.zeros(max(u, 1), np.int32))
    y = np.empty(n, dtype=x.dtype) if want_y else None
    codes = None
    if want_codes:
        codes = np.empty(n, np.int8) if bits == 8 else np.empty((n + 1) // 2, np.uint8)
    mask = np.empty((n + 31) // 32, np.uint32) if want_mask else None
    flags = ctypes.c_int32(0)
    st = lib().or_fake_quant_int(_p(x), dt, rows, cols, bits, scheme, granularity, group, int(given),
                                 _p(sc), _p(zp), _p(y), _p(codes), _p(mask), ctypes.byref(flags),
                                 int(doc_form))
    if st:
        raise ValueError(f"oracle fake_quant_int status {st}")
    return dict(y=y, codes=codes, mask=mask, scale=sc[:u], zero_point=zp[:u], flags=flags.value)


def philox4x32_10(counter, key) -> np.ndarray:
    """One Philox-4x32-10 block: counter (4 x uint32), key (2 x uint32) -> 4 x uint32."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib().or_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_uniform(seed: int, offset: int, n: int) -> np.ndarray:
    """The stochastic-rounding draws u_0 .. u_{n-1} of a call with (seed, offset)."""
    f = lib().or_sr_uniform
    return np.array([f(seed, offset, i) for i in range(n)], np.float32)


def sr_round(r: float, u: float) -> float:
    return lib().or_sr_round(r, u)


def quantize_sr(x: float, scale: float, zp: int, qmin: int, qmax: int, u: float) -> int:
    return lib().or_quantize_sr(x, scale, zp, qmin, qmax, u)


def fp8_cast_sr(t: float, fmt: int, u: float) -> float:
    return lib().or_fp8_cast_sr(t, fmt, u)


def fake_quant_int_sr(x: np.ndarray, rows: int, cols: int, bits: int, scheme: int,
                      granularity: int, group: int = 0, seed: int = 0, offset: int = 0,
                      scale=None, zero_point=None, want_y=True, want_codes=True, want_mask=True):
    """fake_quant_int with stochastic rounding; returns dict(y, codes, mask, scale,
    zero_point, flags)."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    n = rows * cols
    u = n_units(rows, cols, granularity, group) if (granularity != PER_GROUP or group > 0) else 0
    given = scale is not None
    sc = np.ascontiguousarray(scale, dtype=np.float32).copy() if given else np.zeros(max(u, 1), np.float32)
    zp = (np.ascontiguousarray(zero_point, dtype=np.int32).copy() if zero_point is not None
          else np.zeros(max(u, 1), np.int32))
    y = np.empty(n, dtype=x.dtype) if want_y else None
    codes = None
    if want_codes:
        codes = np.empty(n, np.int8) if bits == 8 else np.empty((n + 1) // 2, np.uint8)
    mask = np.empty((n + 31) // 32, np.uint32) if want_mask else None
    flags = ctypes.c_int32(0)
    st = lib().or_fake_quant_int_sr(_p(x), dt, rows, cols, bits, scheme, granularity, group,
                                    int(given), _p(sc), _p(zp), seed, offset, _p(y), _p(codes),
                                    _p(mask), ctypes.byref(flags))
    if st:
        raise ValueError(f"oracle fake_quant_int_sr status {st}")
    return dict(y=y, codes=codes, mask=mask, scale=sc[:u], zero_point=zp[:u], flags=flags.value)


def round_fp16(x) -> np.ndarray:
    """IEEE binary16 rounding (nearest, ties to even) of binary32 values, as binary32."""
    a = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    return np.array([lib().or_round_fp16(float(v)) for v in a], np.float32).reshape(np.shape(x))


def fake_quant_int_opts(x: np.ndarray, rows: int, cols: int, bits: int, scheme: int,
                        granularity: int, group: int = 0, clip: float = 1.0, fp16: bool = False,
                        stochastic: bool = False, seed: int = 0, offset: int = 0):
    """Calibrated fake_quant_int with the range options (clip factor in (0, 1],
    binary16 scales); returns dict(y, codes, mask, scale, zero_point, flags)."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    n = rows * cols
    u = n_units(rows, cols, granularity, group) if (granularity != PER_GROUP or group > 0) else 0
    sc = np.zeros(max(u, 1), np.float32)
    zp = np.zeros(max(u, 1), np.int32)
    y = np.empty(n, dtype=x.dtype)
    codes = np.empty(n, np.int8) if bits == 8 else np.empty((n + 1) // 2, np.uint8)
    mask = np.empty((n + 31) // 32, np.uint32)
    flags = ctypes.c_int32(0)
    st = lib().or_fake_quant_int_opts(_p(x), dt, rows, cols, bits, scheme, granularity, group,
                                      float(np.float32(clip)), int(fp16), int(stochastic), seed,
                                      offset, _p(sc), _p(zp), _p(y), _p(codes), _p(mask),
                                      ctypes.byref(flags))
    if st:
        raise ValueError(f"oracle fake_quant_int_opts status {st}")
    return dict(y=y, codes=codes, mask=mask, scale=sc[:u], zero_point=zp[:u], flags=flags.value)


ELEM_E4M3, ELEM_E5M2, ELEM_E2M3, ELEM_E3M2, ELEM_E2M1 = 0, 1, 2, 3, 4
ELEM_MAX = {0: 448.0, 1: 57344.0, 2: 7.5, 3: 28.0, 4: 6.0}
ELEM_BITS = {0: 8, 1: 8, 2: 6, 3: 6, 4: 4}
SCALE_E8M0, SCALE_E4M3, SCALE_FP32 = 0, 1, 2


def elem_round(v, fmt: int) -> np.ndarray:
    """Round-to-nearest-even with saturation on an element format's grid."""
    a = np.ascontiguousarray(v, dtype=np.float32).reshape(-1)
    return np.array([lib().or_elem_round(float(t), fmt) for t in a], np.float32).reshape(np.shape(v))


def elem_encode(v, fmt: int) -> np.ndarray:
    a = np.ascontiguousarray(v, dtype=np.float32).reshape(-1)
    return np.array([lib().or_elem_encode(float(t), fmt) for t in a], np.uint8).reshape(np.shape(v))


def elem_decode(codes, fmt: int) -> np.ndarray:
    a = np.asarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([lib().or_elem_decode(int(c), fmt) for c in a], np.float32).reshape(np.shape(codes))


def fake_quant_block(x: np.ndarray, fmt: int, block: int, kind: int):
    """Block-scaled fake quant (the teaching script's block_scaled); returns
    dict(y, codes, bscales, tensor_scale, mask, flags)."""
    x = np.ascontiguousarray(x).reshape(-1)
    n = x.size
    y = np.empty(n, dtype=x.dtype)
    codes = np.empty(n, np.uint8)
    nb = n // block if block > 0 else 0
    bs = np.empty(max(nb, 1), np.float32 if kind == SCALE_FP32 else np.uint8)
    mask = np.empty((n + 31) // 32, np.uint32)
    g, fl = ctypes.c_float(1.0), ctypes.c_int32(0)
    st = lib().or_fake_quant_block(_p(x), _dtype_code(x), n, fmt, block, kind, ctypes.byref(g),
                                   _p(y), _p(codes), _p(bs), _p(mask), ctypes.byref(fl))
    if st:
        raise ValueError(f"oracle fake_quant_block status {st}")
    return dict(y=y, codes=codes, bscales=bs[:nb], tensor_scale=np.float32(g.value), mask=mask,
                flags=fl.value)


def percentile_minmax(x: np.ndarray, clip_fraction: float):
    """(lo, hi, flags): the nearest-rank quantiles of per_tensor_percentile."""
    x = np.ascontiguousarray(x).reshape(-1)
    lo, hi, fl = ctypes.c_float(), ctypes.c_float(), ctypes.c_int32(0)
    st = lib().or_percentile_minmax(_p(x), _dtype_code(x), x.size, float(clip_fraction),
                                    ctypes.byref(lo), ctypes.byref(hi), ctypes.byref(fl))
    if st:
        raise ValueError(f"oracle percentile_minmax status {st}")
    return np.float32(lo.value), np.float32(hi.value), fl.value


def fake_quant_int_percentile(x: np.ndarray, bits: int, scheme: int, clip_fraction: float,
                              stochastic: bool = False, seed: int = 0, offset: int = 0):
    """Per-tensor fake quant calibrated by per_tensor_percentile; returns
    dict(y, codes, mask, scale, zero_point, flags)."""
    x = np.ascontiguousarray(x).reshape(-1)
    n = x.size
    s, z, fl = ctypes.c_float(), ctypes.c_int32(), ctypes.c_int32(0)
    y = np.empty(n, dtype=x.dtype)
    codes = np.empty(n, np.int8) if bits == 8 else np.empty((n + 1) // 2, np.uint8)
    mask = np.empty((n + 31) // 32, np.uint32)
    st = lib().or_fake_quant_int_percentile(_p(x), _dtype_code(x), n, bits, scheme,
                                            float(clip_fraction), int(stochastic), seed, offset,
                                            ctypes.byref(s), ctypes.byref(z), _p(y), _p(codes),
                                            _p(mask), ctypes.byref(fl))
    if st:
        raise ValueError(f"oracle fake_quant_int_percentile status {st}")
    return dict(y=y, codes=codes, mask=mask, scale=np.array([s.value], np.float32),
                zero_point=np.array([z.value], np.int32), flags=fl.value)


def fake_quant_fp8_sr(x: np.ndarray, fmt: int, seed: int = 0, offset: int = 0, scale=None,
                      want_codes=True, want_mask=True):
    """fake_quant_fp8 with stochastic rounding; returns dict(y, codes, mask, scale, flags)."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    n = x.size
    s = ctypes.c_float(0.0 if scale is None else float(scale))
    y = np.empty(n, dtype=x.dtype)
    codes = np.empty(n, np.uint8) if want_codes else None
    mask = np.empty((n + 31) // 32, np.uint32) if want_mask else None
    flags = ctypes.c_int32(0)
    st = lib().or_fake_quant_fp8_sr(_p(x), dt, n, fmt, int(scale is not None), ctypes.byref(s),
                                    seed, offset, _p(y), _p(codes), _p(mask), ctypes.byref(flags))
    if st:
        raise ValueError(f"oracle fake_quant_fp8_sr status {st}")
    return dict(y=y, codes=codes, mask=mask, scale=np.float32(s.value), flags=flags.value)


def bias_corrections(beta1: float, beta2: float, t: int):
    """1 - beta^t of step t, evaluated in binary64 as the QAT module does, then
    rounded to binary32 (the values a caller hands to the optimizer step)."""
    b1, b2 = float(np.float32(beta1)), float(np.float32(beta2))
    return np.float32(1.0 - b1 ** t), np.float32(1.0 - b2 ** t)


def adam_update(w, g, m, v, lr, beta1, beta2, eps, wd, bc1, bc2):
    """The optimizer's element loop on copies; returns (w, m, v)."""
    w, m, v = (np.array(a, np.float32).reshape(-1).copy() for a in (w, m, v))
    g = np.ascontiguousarray(g, np.float32).reshape(-1)
    lib().or_adam_update(_p(w), _p(g), _p(m), _p(v), w.size, lr, beta1, beta2, eps, wd, bc1, bc2)
    return w, m, v


def qat_optimizer_step(w, g, m, v, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                       step=1, bits=8, scheme=0, fmt=0, stochastic=False, seed=0, offset=0,
                       want_codes=True, want_mask=True):
    """One QatOptimizer::step on copies of (w, m, v): returns dict(w, m, v, view,
    codes, mask, scale, zero_point, flags); bits = 0 selects the FP8 view."""
    w, m, v = (np.array(a, np.float32).reshape(-1).copy() for a in (w, m, v))
    g = np.ascontiguousarray(g, np.float32).reshape(-1)
    n = w.size
    bc1, bc2 = bias_corrections(beta1, beta2, step)
    view = np.empty(n, np.float32)
    codes = None
    if want_codes:
        codes = (np.empty(n, np.int8) if bits == 8 else np.empty((n + 1) // 2, np.uint8) if bits == 4
                 else np.empty(n, np.uint8))
    mask = np.empty((n + 31) // 32, np.uint32) if want_mask else None
    sc, zp, flags = ctypes.c_float(0.0), ctypes.c_int32(0), ctypes.c_int32(0)
    st = lib().or_qat_optimizer_step(_p(w), _p(g), _p(m), _p(v), n, lr, beta1, beta2, eps,
                                     weight_decay, bc1, bc2, bits, scheme, fmt, int(stochastic),
                                     seed, offset, _p(view), _p(codes), _p(mask), ctypes.byref(sc),
                                     ctypes.byref(zp), ctypes.byref(flags))
    if st:
        raise ValueError(f"oracle qat_optimizer_step status {st}")
    return dict(w=w, m=m, v=v, view=view, codes=codes, mask=mask, scale=np.float32(sc.value),
                zero_point=zp.value, flags=flags.value, bias_corrections=(bc1, bc2))


def fake_quant_fp8(x: np.ndarray, fmt: int, scale=None, want_codes=True, want_mask=True):
    """Returns dict(y, codes, mask, scale, flags); ``scale`` given -> used as is."""
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    n = x.size
    s = ctypes.c_float(0.0 if scale is None else float(scale))
    y = np.empty(n, dtype=x.dtype)
    codes = np.empty(n, np.uint8) if want_codes else None
    mask = np.empty((n + 31) // 32, np.uint32) if want_mask else None
    flags = ctypes.c_int32(0)
    st = lib().or_fake_quant_fp8(_p(x), dt, n, fmt, int(scale is not None), ctypes.byref(s), _p(y),
                                 _p(codes), _p(mask), ctypes.byref(flags))
    if st:
        raise ValueError(f"oracle fake_quant_fp8 status {st}")
    return dict(y=y, codes=codes, mask=mask, scale=np.float32(s.value), flags=flags.value)


def fp8_cast(t: float, fmt: int) -> float:
    return lib().or_fp8_cast(t, fmt)


def fp8_encode(c: float, fmt: int) -> int:
    return lib().or_fp8_encode(c, fmt)


def ste_backward(g: np.ndarray, mask: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g).reshape(-1)
    dt = _dtype_code(g)
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    dx = np.empty_like(g)
    st = lib().or_ste_backward(_p(g), dt, g.size, _p(mask), _p(dx))
    if st:
        raise ValueError(f"oracle ste_backward status {st}")
    return dx


def q4_sizes(n: int):
    nb = (n + 63) // 64
    return (n + 1) // 2, nb, (nb + 255) // 256


def quant4_double(x: np.ndarray, roundtrip: bool = False):
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    n = x.size
    nd, nb, ns = q4_sizes(n)
    data = np.zeros(nd, np.uint8)
    qs = np.zeros(nb, np.uint8)
    sup = np.zeros(ns, np.float32)
    y = np.empty(n, np.float32) if roundtrip else None
    st = lib().or_quant4_double(_p(x), n, _p(data), _p(qs), _p(sup), _p(y))
    if st:
        raise ValueError(f"oracle quant4_double status {st}")
    return dict(data=data, qscales=qs, super_scales=sup, y=y)


def dequant4_double(data, qscales, super_scales, n: int) -> np.ndarray:
    data = np.ascontiguousarray(data, dtype=np.uint8)
    qscales = np.ascontiguousarray(qscales, dtype=np.uint8)
    super_scales = np.ascontiguousarray(super_scales, dtype=np.float32)
    y = np.empty(n, np.float32)
    lib().or_dequant4_double(_p(data), _p(qscales), _p(super_scales), n, _p(y))
    return y


def quant4_single(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    nd, nb, _ = q4_sizes(x.size)
    data = np.zeros(nd, np.uint8)
    sc = np.zeros(nb, np.float32)
    lib().or_quant4_single(_p(x), x.size, _p(data), _p(sc))
    return dict(data=data, scales=sc)


def dequant4_single(data, scales, n: int) -> np.ndarray:
    y = np.empty(n, np.float32)
    lib().or_dequant4_single(_p(np.ascontiguousarray(data, np.uint8)),
                             _p(np.ascontiguousarray(scales, np.float32)), n, _p(y))
    return y


def reconstruct_scale(q: int, super_scale: float) -> float:
    return lib().or_reconstruct_scale(q, super_scale)


def q4d_memory_bytes(n: int) -> int:
    return lib().or_q4d_memory_bytes(n)


def fake_quant_int_f64(x: np.ndarray, rows: int, cols: int, bits: int, scheme: int, granularity: int,
                       group: int = 0):
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    n = rows * cols
    u = max(n_units(rows, cols, granularity, group), 1)
    y = np.empty(n, np.float64)
    s = np.zeros(u, np.float64)
    z = np.zeros(u, np.int32)
    st = lib().or64_fake_quant_int(_p(x), dt, rows, cols, bits, scheme, granularity, group, _p(y),
                                   _p(s), _p(z))
    if st:
        raise ValueError(f"oracle f64 int status {st}")
    return dict(y=y, scale=s, zero_point=z)


def fake_quant_fp8_f64(x: np.ndarray, fmt: int):
    x = np.ascontiguousarray(x).reshape(-1)
    dt = _dtype_code(x)
    y = np.empty(x.size, np.float64)
    s = ctypes.c_double()
    lib().or64_fake_quant_fp8(_p(x), dt, x.size, fmt, _p(y), ctypes.byref(s))
    return dict(y=y, scale=s.value)
