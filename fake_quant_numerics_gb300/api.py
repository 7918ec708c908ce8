"""Python binding of libqat.so.

Two layers, both thin:

* ``qat_*`` functions mirror the C ABI one to one: they take torch CUDA
  tensors for every buffer, turn them into pointers, pass the current CUDA
  stream and raise :class:`QatError` on a non-OK status.  They allocate
  nothing.
* The named operations of the source module (``fake_quant_int``,
  ``fake_quant_fp8``, ``fake_quant_backward``, ``quantize_4bit_double``,
  ``dequantize_4bit_double``, ``amax_stats``) allocate the outputs with torch
  and call the ``qat_*`` layer.  Every step of the computation runs in the
  library's kernels.
"""
from __future__ import annotations

import ctypes
from typing import NamedTuple, Optional

import torch

from . import _lib
from ._lib import (AFFINE, BF16, E4M3, E5M2, F32, FLAG_BAD_PARAMS, FLAG_DEGENERATE,
                   FLAG_DEVICE_TIMEOUT, FLAG_NONFINITE_CALIB, PER_COLUMN, PER_GROUP, PER_ROW, PER_TENSOR, SYMMETRIC,
                   QatError)

_DT = {torch.float32: F32, torch.bfloat16: BF16}
_SCHEME = {"symmetric": SYMMETRIC, "sym": SYMMETRIC, "affine": AFFINE,
           SYMMETRIC: SYMMETRIC, AFFINE: AFFINE}
_GRAN = {"tensor": PER_TENSOR, "per_tensor": PER_TENSOR, "row": PER_ROW, "per_row": PER_ROW,
         "channel": PER_ROW, "group": PER_GROUP, "per_group": PER_GROUP, "column": PER_COLUMN,
         "per_column": PER_COLUMN, PER_TENSOR: PER_TENSOR, PER_ROW: PER_ROW, PER_GROUP: PER_GROUP,
         PER_COLUMN: PER_COLUMN}
_FMT = {"e4m3": E4M3, "E4M3": E4M3, "e5m2": E5M2, "E5M2": E5M2, E4M3: E4M3, E5M2: E5M2}
ERROR_FLAGS = FLAG_NONFINITE_CALIB | FLAG_DEGENERATE | FLAG_BAD_PARAMS


class QatDataError(ValueError):
    """A device-side data error (non-finite or degenerate calibration, bad parameters)."""


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libqat takes CUDA tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dt(x: torch.Tensor) -> int:
    try:
        return _DT[x.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {x.dtype} (float32 or bfloat16)") from None


def _nbytes(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.numel() * t.element_size()


# ---------------------------------------------------------------------------
# C ABI mirror
# ---------------------------------------------------------------------------
def qat_workspace_bytes(rows: int, cols: int, granularity, group: int = 0) -> int:
    return int(_lib.lib().qat_workspace_bytes(rows, cols, _GRAN[granularity], group))


def qat_amax_stats(x, rows, cols, granularity, group, absmax, minv, maxv, dev_flags, workspace,
                   stream=None):
    st = _lib.lib().qat_amax_stats(_p(x), _dt(x), rows, cols, _GRAN[granularity], group, _p(absmax),
                                   _p(minv), _p(maxv), _p(dev_flags), _p(workspace),
                                   _nbytes(workspace), _s(stream))
    _lib.check("qat_amax_stats", st)


def qat_fake_quant_int(x, rows, cols, bits, scheme, granularity, group, params_given, scale,
                       zero_point, y, codes, mask, dev_flags, workspace, stream=None):
    st = _lib.lib().qat_fake_quant_int(_p(x), _dt(x), rows, cols, bits, _SCHEME[scheme],
                                       _GRAN[granularity], group, int(params_given), _p(scale),
                                       _p(zero_point), _p(y), _p(codes), _p(mask), _p(dev_flags),
                                       _p(workspace), _nbytes(workspace), _s(stream))
    _lib.check("qat_fake_quant_int", st)


def qat_fake_quant_fp8(x, n, fmt, scale_given, scale, y, codes, mask, dev_flags, workspace,
                       stream=None):
    st = _lib.lib().qat_fake_quant_fp8(_p(x), _dt(x), n, _FMT[fmt], int(scale_given), _p(scale),
                                       _p(y), _p(codes), _p(mask), _p(dev_flags), _p(workspace),
                                       _nbytes(workspace), _s(stream))
    _lib.check("qat_fake_quant_fp8", st)


def qat_fake_quant_int_sr(x, rows, cols, bits, scheme, granularity, group, params_given, scale,
                          zero_point, seed, offset, y, codes, mask, dev_flags, workspace,
                          stream=None):
    st = _lib.lib().qat_fake_quant_int_sr(_p(x), _dt(x), rows, cols, bits, _SCHEME[scheme],
                                          _GRAN[granularity], group, int(params_given), _p(scale),
                                          _p(zero_point), int(seed), int(offset), _p(y), _p(codes),
                                          _p(mask), _p(dev_flags), _p(workspace),
                                          _nbytes(workspace), _s(stream))
    _lib.check("qat_fake_quant_int_sr", st)


def calib_options(clip: float = 1.0, scale_fp16: bool = False) -> "_lib.CalibOptions":
    """qat_calib_options: the calibrated range times clip (in (0, 1]), binary16 scales."""
    return _lib.CalibOptions(float(clip), int(bool(scale_fp16)))


def qat_fake_quant_int_opts(x, rows, cols, bits, scheme, granularity, group, options, stochastic,
                            seed, offset, scale, zero_point, y, codes, mask, dev_flags, workspace,
                            stream=None):
    opt = ctypes.byref(options) if options is not None else None
    st = _lib.lib().qat_fake_quant_int_opts(_p(x), _dt(x), rows, cols, bits, _SCHEME[scheme],
                                            _GRAN[granularity], group, opt, int(bool(stochastic)),
                                            int(seed), int(offset), _p(scale), _p(zero_point),
                                            _p(y), _p(codes), _p(mask), _p(dev_flags),
                                            _p(workspace), _nbytes(workspace), _s(stream))
    _lib.check("qat_fake_quant_int_opts", st)


_ELEM = {"e4m3": 0, "e5m2": 1, "e2m3": 2, "e3m2": 3, "e2m1": 4, 0: 0, 1: 1, 2: 2, 3: 3, 4: 4}
_BSCALE = {"e8m0": 0, "e4m3": 1, "fp32": 2, 0: 0, 1: 1, 2: 2}
_ELEM_BITS = {0: 8, 1: 8, 2: 6, 3: 6, 4: 4}


def qat_fake_quant_block(x, n, elem, block, scale_kind, tensor_scale, y, codes, block_scales,
                         mask, dev_flags, workspace, stream=None):
    st = _lib.lib().qat_fake_quant_block(_p(x), _dt(x), n, _ELEM[elem], block, _BSCALE[scale_kind],
                                         _p(tensor_scale), _p(y), _p(codes), _p(block_scales),
                                         _p(mask), _p(dev_flags), _p(workspace),
                                         _nbytes(workspace), _s(stream))
    _lib.check("qat_fake_quant_block", st)


class FakeQuantBlock(NamedTuple):
    y: torch.Tensor
    codes: Optional[torch.Tensor]
    block_scales: torch.Tensor
    tensor_scale: torch.Tensor
    mask: Optional[torch.Tensor]
    flags: torch.Tensor


def fake_quant_block(x: torch.Tensor, elem="e2m1", block: int = 16, scale="e4m3",
                     want_codes: bool = True, want_mask: bool = True) -> FakeQuantBlock:
    """Block-scaled floating-point fake quantization of x (float32 or bfloat16,
    CUDA; blocks of 16 or 32 consecutive elements).  NVFP4 is elem="e2m1",
    block=16, scale="e4m3"; MXFP4 / MXFP6 / MXFP8 are block=32, scale="e8m0"
    with elem "e2m1" / "e2m3" or "e3m2" / "e4m3" or "e5m2"."""
    x = _ready(x)
    n = x.numel()
    dev = x.device
    e, k = _ELEM[elem], _BSCALE[scale]
    if n % block:
        raise ValueError(f"{n} elements are not a whole number of blocks of {block}")
    nb = n // block
    y = torch.empty_like(x)
    codes = None
    if want_codes:
        codes = torch.empty(n // 2 if _ELEM_BITS[e] == 4 else n, dtype=torch.uint8, device=dev)
    bs = torch.empty(nb, dtype=torch.float32 if k == 2 else torch.uint8, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    mask = torch.empty((n + 31) // 32, dtype=torch.int32, device=dev) if want_mask else None
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(max(qat_workspace_bytes(1, n, PER_TENSOR, 0), 16), dtype=torch.uint8,
                     device=dev)
    qat_fake_quant_block(x, n, e, block, k, g, y, codes, bs, mask, flags, ws)
    return FakeQuantBlock(y, codes, bs, g, mask, flags)


def qat_percentile_workspace_bytes() -> int:
    return int(_lib.lib().qat_percentile_workspace_bytes())


def qat_fake_quant_int_percentile(x, n, bits, scheme, clip_fraction, stochastic, seed, offset,
                                  scale, zero_point, y, codes, mask, dev_flags, workspace,
                                  stream=None):
    st = _lib.lib().qat_fake_quant_int_percentile(_p(x), _dt(x), n, bits, _SCHEME[scheme],
                                                  float(clip_fraction), int(bool(stochastic)),
                                                  int(seed), int(offset), _p(scale),
                                                  _p(zero_point), _p(y), _p(codes), _p(mask),
                                                  _p(dev_flags), _p(workspace),
                                                  _nbytes(workspace), _s(stream))
    _lib.check("qat_fake_quant_int_percentile", st)


def fake_quant_int_percentile(x: torch.Tensor, bits: int = 8, scheme="symmetric",
                              clip_fraction: float = 0.0, want_codes: bool = True,
                              want_mask: bool = True, check: bool = False,
                              rounding: str = "nearest", seed: int = 0,
                              offset: int = 0) -> FakeQuantInt:
    """Per-tensor integer fake quantization calibrated by the nearest-rank
    quantiles at clip_fraction and 1 - clip_fraction (the module's
    per_tensor_percentile)."""
    x = _ready(x)
    n = x.numel()
    sch = _SCHEME[scheme]
    dev = x.device
    scale = torch.empty(1, dtype=torch.float32, device=dev)
    zero_point = torch.empty(1, dtype=torch.int32, device=dev) if sch == AFFINE else None
    y = torch.empty_like(x)
    codes = None
    if want_codes:
        codes = (torch.empty(n, dtype=torch.int8, device=dev) if bits == 8
                 else torch.empty((n + 1) // 2, dtype=torch.uint8, device=dev))
    mask = torch.empty((n + 31) // 32, dtype=torch.int32, device=dev) if want_mask else None
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(qat_percentile_workspace_bytes(), dtype=torch.uint8, device=dev)
    if rounding not in ("nearest", "stochastic"):
        raise ValueError(f"rounding must be 'nearest' or 'stochastic', not {rounding!r}")
    qat_fake_quant_int_percentile(x, n, bits, sch, clip_fraction, rounding == "stochastic", seed,
                                  offset, scale, zero_point, y, codes, mask, flags, ws)
    if check:
        raise_on_flags(flags, "fake_quant_int_percentile")
    return FakeQuantInt(y, codes, mask, scale, zero_point, flags)


def qat_fake_quant_fp8_sr(x, n, fmt, scale_given, scale, seed, offset, y, codes, mask, dev_flags,
                          workspace, stream=None):
    st = _lib.lib().qat_fake_quant_fp8_sr(_p(x), _dt(x), n, _FMT[fmt], int(scale_given), _p(scale),
                                          int(seed), int(offset), _p(y), _p(codes), _p(mask),
                                          _p(dev_flags), _p(workspace), _nbytes(workspace),
                                          _s(stream))
    _lib.check("qat_fake_quant_fp8_sr", st)


def adam_hparams(lr, beta1, beta2, eps, weight_decay, step):
    """qat_adam_hparams of step `step` (>= 1): the bias corrections 1 - beta^t
    evaluated in binary64 (as QatOptimizer::step does) from the binary32 betas."""
    b1, b2 = ctypes.c_float(beta1).value, ctypes.c_float(beta2).value
    return _lib.AdamHparams(lr, beta1, beta2, eps, weight_decay, 1.0 - b1 ** step, 1.0 - b2 ** step)


def qat_optimizer_step(master, grad, exp_avg, exp_avg_sq, n, hparams, bits, scheme, fmt, stochastic,
                       seed, offset, view, codes, mask, scale, zero_point, dev_flags, workspace,
                       stream=None):
    st = _lib.lib().qat_optimizer_step(_p(master), _p(grad), _p(exp_avg), _p(exp_avg_sq), n,
                                       ctypes.byref(hparams), bits, _SCHEME[scheme], _FMT[fmt],
                                       int(stochastic), int(seed), int(offset), _p(view),
                                       _p(codes), _p(mask), _p(scale), _p(zero_point),
                                       _p(dev_flags), _p(workspace), _nbytes(workspace),
                                       _s(stream))
    _lib.check("qat_optimizer_step", st)


def qat_ste_backward(grad, n, mask, grad_in, stream=None):
    st = _lib.lib().qat_ste_backward(_p(grad), _dt(grad), n, _p(mask), _p(grad_in), _s(stream))
    _lib.check("qat_ste_backward", st)


def qat_quant4_double(x, n, data, qscales, super_scales, y_roundtrip=None, stream=None):
    st = _lib.lib().qat_quant4_double(_p(x), n, _p(data), _p(qscales), _p(super_scales),
                                      _p(y_roundtrip), _s(stream))
    _lib.check("qat_quant4_double", st)


def qat_dequant4_double(data, qscales, super_scales, n, y, stream=None):
    st = _lib.lib().qat_dequant4_double(_p(data), _p(qscales), _p(super_scales), n, _p(y), _s(stream))
    _lib.check("qat_dequant4_double", st)


def qat_kernel_launch_count() -> int:
    return int(_lib.lib().qat_kernel_launch_count())


# ---------------------------------------------------------------------------
# named operations (allocate outputs)
# ---------------------------------------------------------------------------
def _ready(x: torch.Tensor) -> torch.Tensor:
    """Contiguous and 32-byte aligned (a fresh copy when it is not)."""
    x = x.contiguous()
    if x.data_ptr() % 32:
        x = x.clone()
    return x


def _shape2d(x: torch.Tensor):
    if x.dim() == 0:
        return 1, 1
    if x.dim() == 1:
        return 1, x.shape[0]
    return x.numel() // x.shape[-1], x.shape[-1]


def n_units(rows: int, cols: int, granularity, group: int = 0) -> int:
    g = _GRAN[granularity]
    if g == PER_TENSOR:
        return 1
    if g == PER_ROW:
        return rows
    if g == PER_COLUMN:
        return cols
    return rows * cols // group


def raise_on_flags(flags: torch.Tensor, what: str = "fake quant"):
    """Synchronise on the flag word and raise QatDataError for error flags
    (QatError for a device-side wait that ran out)."""
    f = int(flags.item())
    if f & FLAG_DEVICE_TIMEOUT:
        raise QatError(what, _lib.QAT_ERR_CUDA)
    if f & ERROR_FLAGS:
        parts = []
        if f & FLAG_NONFINITE_CALIB:
            parts.append("non-finite value in calibration tensor")
        if f & FLAG_DEGENERATE:
            parts.append("degenerate (zero-range) calibration")
        if f & FLAG_BAD_PARAMS:
            parts.append("invalid quantization parameters")
        raise QatDataError(f"{what}: " + "; ".join(parts))


class FakeQuantInt(NamedTuple):
    y: torch.Tensor
    codes: Optional[torch.Tensor]
    mask: Optional[torch.Tensor]
    scale: torch.Tensor
    zero_point: Optional[torch.Tensor]
    flags: torch.Tensor


class FakeQuantFp8(NamedTuple):
    y: torch.Tensor
    codes: Optional[torch.Tensor]
    mask: Optional[torch.Tensor]
    scale: torch.Tensor
    flags: torch.Tensor


class DoubleQuantized4Bit(NamedTuple):
    data: torch.Tensor              # uint8[ceil(n/2)]
    quantized_scales: torch.Tensor  # uint8[ceil(n/64)]
    super_scales: torch.Tensor      # float32[ceil(ceil(n/64)/256)]
    len: int
    y: Optional[torch.Tensor]       # fused round trip, if requested

    @property
    def num_blocks(self) -> int:
        return self.quantized_scales.numel()

    def memory_bytes(self) -> int:
        return self.quantized_scales.numel() + 4 * self.super_scales.numel() + self.data.numel()


def fake_quant_int(x: torch.Tensor, bits: int = 8, scheme="symmetric", granularity="tensor",
                   group: int = 0, scale: Optional[torch.Tensor] = None,
                   zero_point: Optional[torch.Tensor] = None, want_codes: bool = True,
                   want_mask: bool = True, check: bool = False, rounding: str = "nearest",
                   seed: int = 0, offset: int = 0, clip: float = 1.0,
                   scale_fp16: bool = False) -> FakeQuantInt:
    """Integer fake quantization of x (float32 or bfloat16, CUDA), calibrated per
    tensor / row / group / column (of the last dimension), or with the given
    per-unit scale and zero point.
    rounding="stochastic" rounds with the counter-based draws of (seed, offset).
    clip (in (0, 1]) shrinks the calibrated range; scale_fp16 rounds the
    calibrated scales to binary16 (calibrated calls only)."""
    x = _ready(x)
    rows, cols = _shape2d(x)
    n = x.numel()
    sch = _SCHEME[scheme]
    gran = _GRAN[granularity]
    if gran == PER_GROUP and (group <= 0 or cols % group):
        raise ValueError(f"group {group} must divide the last dimension {cols}")
    units = n_units(rows, cols, gran, group)
    dev = x.device
    given = scale is not None
    if given:
        scale = _ready(scale.to(device=dev, dtype=torch.float32).reshape(-1))
        if scale.numel() != units:
            raise QatError("fake_quant_int", _lib.QAT_ERR_DIMENSION_MISMATCH)
        if sch == AFFINE:
            if zero_point is None or zero_point.numel() != units:
                raise QatError("fake_quant_int", _lib.QAT_ERR_DIMENSION_MISMATCH)
            zero_point = _ready(zero_point.to(device=dev, dtype=torch.int32).reshape(-1))
    else:
        scale = torch.empty(units, dtype=torch.float32, device=dev)
        zero_point = torch.empty(units, dtype=torch.int32, device=dev) if sch == AFFINE else None
    y = torch.empty_like(x)
    codes = None
    if want_codes:
        codes = (torch.empty(n, dtype=torch.int8, device=dev) if bits == 8
                 else torch.empty((n + 1) // 2, dtype=torch.uint8, device=dev))
    mask = torch.empty((n + 31) // 32, dtype=torch.int32, device=dev) if want_mask else None
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = qat_workspace_bytes(rows, cols, gran, group)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    if rounding not in ("nearest", "stochastic"):
        raise ValueError(f"rounding must be 'nearest' or 'stochastic', not {rounding!r}")
    if clip != 1.0 or scale_fp16:
        if given:
            raise ValueError("clip and scale_fp16 apply to calibrated calls only")
        qat_fake_quant_int_opts(x, rows, cols, bits, sch, gran, group,
                                calib_options(clip, scale_fp16), rounding == "stochastic", seed,
                                offset, scale, zero_point, y, codes, mask, flags, ws)
    elif rounding == "stochastic":
        qat_fake_quant_int_sr(x, rows, cols, bits, sch, gran, group, given, scale, zero_point, seed,
                              offset, y, codes, mask, flags, ws)
    elif rounding == "nearest":
        qat_fake_quant_int(x, rows, cols, bits, sch, gran, group, given, scale, zero_point, y, codes,
                           mask, flags, ws)
    else:
        raise ValueError(f"rounding must be 'nearest' or 'stochastic', not {rounding!r}")
    if check:
        raise_on_flags(flags, "fake_quant_int")
    return FakeQuantInt(y, codes, mask, scale, zero_point, flags)


def fake_quant_fp8(x: torch.Tensor, fmt="e4m3", scale: Optional[float] = None,
                   want_codes: bool = False, want_mask: bool = True, rounding: str = "nearest",
                   seed: int = 0, offset: int = 0) -> FakeQuantFp8:
    """Per-tensor amax-scaled (or given-scale) saturating FP8 fake quantization;
    rounding="stochastic" rounds with the counter-based draws of (seed, offset).
    clip (in (0, 1]) shrinks the calibrated range; scale_fp16 rounds the
    calibrated scales to binary16 (calibrated calls only)."""
    x = _ready(x)
    n = x.numel()
    dev = x.device
    given = scale is not None
    s = torch.empty(1, dtype=torch.float32, device=dev)
    if given:
        s.fill_(float(scale))
    y = torch.empty_like(x)
    codes = torch.empty(n, dtype=torch.uint8, device=dev) if want_codes else None
    mask = torch.empty((n + 31) // 32, dtype=torch.int32, device=dev) if want_mask else None
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = None
    if not given:
        ws = torch.empty(qat_workspace_bytes(1, n, PER_TENSOR, 0), dtype=torch.uint8, device=dev)
    if rounding == "stochastic":
        qat_fake_quant_fp8_sr(x, n, fmt, given, s, seed, offset, y, codes, mask, flags, ws)
    elif rounding == "nearest":
        qat_fake_quant_fp8(x, n, fmt, given, s, y, codes, mask, flags, ws)
    else:
        raise ValueError(f"rounding must be 'nearest' or 'stochastic', not {rounding!r}")
    return FakeQuantFp8(y, codes, mask, s, flags)


class OptimizerStep(NamedTuple):
    view: torch.Tensor
    codes: Optional[torch.Tensor]
    mask: Optional[torch.Tensor]
    scale: torch.Tensor
    zero_point: Optional[torch.Tensor]
    flags: torch.Tensor


_TARGETS = {"int8": (8, E4M3), "int4": (4, E4M3), "e4m3": (0, E4M3), "fp8_e4m3": (0, E4M3),
            "e5m2": (0, E5M2), "fp8_e5m2": (0, E5M2)}


def _in_place(t: torch.Tensor, what: str) -> torch.Tensor:
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.data_ptr() % 32:
        raise ValueError(f"{what} must be a contiguous, 32-byte aligned float32 CUDA tensor "
                         "(it is updated in place)")
    return t


def optimizer_step(master: torch.Tensor, grad: torch.Tensor, exp_avg: torch.Tensor,
                   exp_avg_sq: torch.Tensor, step: int, lr: float, betas=(0.9, 0.999),
                   eps: float = 1e-8, weight_decay: float = 0.0, target: str = "int8",
                   scheme="symmetric", rounding: str = "nearest", seed: int = 0, offset: int = 0,
                   want_codes: bool = False, want_mask: bool = False,
                   check: bool = False) -> OptimizerStep:
    """One QatOptimizer::step: Adam / AdamW update of the float32 master and its
    moments in place (step t >= 1), then the fake-quant view of the new master
    (target int8 / int4 calibrated per tensor, or the unscaled e4m3 / e5m2 cast)."""
    if step < 1:
        raise ValueError("step counts from 1")
    bits, fmt = _TARGETS[target]
    master = _in_place(master, "master")
    exp_avg = _in_place(exp_avg, "exp_avg")
    exp_avg_sq = _in_place(exp_avg_sq, "exp_avg_sq")
    grad = _ready(grad.to(torch.float32))
    n = master.numel()
    if grad.numel() != n or exp_avg.numel() != n or exp_avg_sq.numel() != n:
        raise QatError("optimizer_step", _lib.QAT_ERR_DIMENSION_MISMATCH)
    dev = master.device
    view = torch.empty_like(master)
    codes = None
    if want_codes:
        codes = (torch.empty(n, dtype=torch.int8, device=dev) if bits == 8
                 else torch.empty((n + 1) // 2, dtype=torch.uint8, device=dev) if bits == 4
                 else torch.empty(n, dtype=torch.uint8, device=dev))
    mask = torch.empty((n + 31) // 32, dtype=torch.int32, device=dev) if want_mask else None
    scale = torch.empty(1, dtype=torch.float32, device=dev)
    zp = torch.empty(1, dtype=torch.int32, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(qat_workspace_bytes(1, n, PER_TENSOR, 0), dtype=torch.uint8, device=dev)
    if rounding not in ("nearest", "stochastic"):
        raise ValueError(f"rounding must be 'nearest' or 'stochastic', not {rounding!r}")
    hp = adam_hparams(lr, betas[0], betas[1], eps, weight_decay, step)
    qat_optimizer_step(master, grad, exp_avg, exp_avg_sq, n, hp, bits, scheme, fmt,
                       rounding == "stochastic", seed, offset, view, codes, mask, scale, zp, flags,
                       ws)
    if check:
        raise_on_flags(flags, "optimizer_step")
    return OptimizerStep(view, codes, mask, scale, zp if bits and _SCHEME[scheme] == AFFINE else None,
                         flags)


def fake_quant_backward(grad: torch.Tensor, mask: torch.Tensor) -> torch.Tensor:
    """Straight-through estimator: grad where the forward mask bit is set, else +0."""
    grad = _ready(grad)
    n = grad.numel()
    if mask.numel() != (n + 31) // 32:
        raise QatError("fake_quant_backward", _lib.QAT_ERR_DIMENSION_MISMATCH)
    dx = torch.empty_like(grad)
    qat_ste_backward(grad, n, _ready(mask), dx)
    return dx


def amax_stats(x: torch.Tensor, granularity="tensor", group: int = 0):
    """(absmax, min, max, flags) over the finite elements of each unit."""
    x = _ready(x)
    rows, cols = _shape2d(x)
    gran = _GRAN[granularity]
    units = n_units(rows, cols, gran, group)
    dev = x.device
    a = torch.empty(units, dtype=torch.float32, device=dev)
    mn = torch.empty_like(a)
    mx = torch.empty_like(a)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(max(qat_workspace_bytes(rows, cols, gran, group), 16), dtype=torch.uint8,
                     device=dev)
    qat_amax_stats(x, rows, cols, gran, group, a, mn, mx, flags, ws)
    return a, mn, mx, flags


def quantize_4bit_double(x: torch.Tensor, roundtrip: bool = False) -> DoubleQuantized4Bit:
    """QLoRA two-level 4-bit quantization of a float32 tensor (flattened)."""
    if x.dtype != torch.float32:
        raise TypeError("quantize_4bit_double takes float32")
    x = _ready(x.reshape(-1))
    n = x.numel()
    dev = x.device
    nb = (n + 63) // 64
    data = torch.empty((n + 1) // 2, dtype=torch.uint8, device=dev)
    qs = torch.empty(nb, dtype=torch.uint8, device=dev)
    sup = torch.empty((nb + 255) // 256, dtype=torch.float32, device=dev)
    y = torch.empty(n, dtype=torch.float32, device=dev) if roundtrip else None
    qat_quant4_double(x, n, data, qs, sup, y)
    return DoubleQuantized4Bit(data, qs, sup, n, y)


def dequantize_4bit_double(dq: DoubleQuantized4Bit) -> torch.Tensor:
    y = torch.empty(dq.len, dtype=torch.float32, device=dq.data.device)
    qat_dequant4_double(_ready(dq.data), _ready(dq.quantized_scales), dq.super_scales.contiguous(),
                        dq.len, y)
    return y


class FakeQuantSTE(torch.autograd.Function):
    """Integer fake quant whose backward is the straight-through estimator."""

    @staticmethod
    def forward(ctx, x, bits=8, scheme="symmetric", granularity="tensor", group=0):
        r = fake_quant_int(x, bits, scheme, granularity, group, want_codes=False)
        ctx.save_for_backward(r.mask)
        ctx.shape = x.shape
        return r.y.view(x.shape)

    @staticmethod
    def backward(ctx, g):
        (mask,) = ctx.saved_tensors
        return fake_quant_backward(g, mask).view(ctx.shape), None, None, None, None
