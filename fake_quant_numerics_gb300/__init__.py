"""GB300 fake-quant library: QAT fake quantization (int8/int4 symmetric and
affine per tensor / row / group, saturating FP8 E4M3/E5M2), its
straight-through-estimator backward, and the QLoRA two-level 4-bit block
format, as CUDA kernels for sm_103a behind a C ABI (include/qat.h); the
integer and FP8 maps also round stochastically with counter-based draws;
units may also be columns, and calibration takes a clip factor and binary16
scales; block-scaled floating-point formats (MX with E8M0 scales, NVFP4
with E4M3 scales under an FP32 tensor scale).
"""
from ._lib import QatError, load  # noqa: F401
from .api import (DoubleQuantized4Bit, FakeQuantBlock, FakeQuantFp8, FakeQuantInt,  # noqa: F401
                  FakeQuantSTE, fake_quant_block, qat_fake_quant_block,
                  OptimizerStep, QatDataError, adam_hparams, amax_stats, calib_options,
                  dequantize_4bit_double,
                  fake_quant_backward, optimizer_step, qat_optimizer_step,
                  fake_quant_fp8, fake_quant_int, fake_quant_int_percentile, qat_amax_stats,
                  qat_dequant4_double, qat_fake_quant_int_percentile,
                  qat_percentile_workspace_bytes,
                  qat_fake_quant_fp8, qat_fake_quant_fp8_sr, qat_fake_quant_int,
                  qat_fake_quant_int_opts, qat_fake_quant_int_sr, qat_kernel_launch_count,
                  qat_quant4_double, qat_ste_backward, qat_workspace_bytes, quantize_4bit_double,
                  raise_on_flags)
