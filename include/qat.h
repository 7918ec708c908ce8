/*
 * qat.h -- C ABI of the GB300 fake-quant library (libqat.so).
 *
 * Quantization-aware-training fake quantization and its straight-through
 * estimator, plus the QLoRA two-level 4-bit block format, as CUDA kernels for
 * sm_103a.  Sources of the operations (cited by page and item):
 *
 *   [QAT] optirs-gpu 0.3.2, src/optirs_gpu/quantization.rs -- module docs
 *         ("What fake quantization means", "Integer quantization",
 *         "fp8 quantization", "Straight-through estimator"), IntDtype::q_range,
 *         QuantParams::{from_minmax, from_absmax, quantize, dequantize,
 *         real_min, real_max}, finite_min_max, fake_quant_int,
 *         per_channel_params, fake_quant_int_per_channel,
 *         fp8_quantize_magnitude, fake_quant_fp8, fake_quant_backward.
 *   [DQ]  aprender-train 0.32.0, src/entrenar/quant/double_quant.rs --
 *         quantize_4bit_double, reconstruct_scales, dequantize_4bit_double,
 *         DoubleQuantized4Bit.
 *   [MAR] ferrum-kernels 0.8.0, src/marlin_repack.rs -- per-channel E4M3
 *         scale absmax / 448, a zero scale encodes as byte 0.
 *   [EDU] cs349e 05_quantization_basics.py, demo 3 -- groups run along the
 *         last dimension.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer.  x, y, grad, grad_in and
 *   y_roundtrip must be 32-byte aligned (each lane moves 32-byte vectors);
 *   codes, mask, data, qscales and workspace 16-byte aligned; per-unit arrays
 *   (scale, zero_point, absmax, minv, maxv, super_scales) 4-byte aligned.
 *   A violation returns QAT_ERR_MISALIGNED.  dev_flags is an int32.
 * - Tensors are row-major and contiguous; n = rows * cols.  A "unit" is the
 *   whole tensor (per tensor), one row of `cols` elements (per row, the axis-0
 *   channel of [QAT] per_channel_params) or one run of `group` consecutive
 *   elements of a row (per group; `group` must divide `cols`).
 * - Outputs y have the dtype of x; they are computed in fp32 and rounded once
 *   (round to nearest even) to bf16 when x is bf16.
 * - mask: uint32 words, bit (i % 32) of word (i / 32) is element i; bits past
 *   n in the last word are 0.  Length ceil(n / 32) words.
 * - 4-bit codes are packed two per byte: element 2j in the HIGH nibble and
 *   element 2j+1 in the LOW nibble of byte j, two's complement (the nibble
 *   order of [DQ] dequantize_4bit_double); an odd tail leaves the last low
 *   nibble 0.  Length ceil(n / 2) bytes.  8-bit codes are int8[n].
 * - Ownership: the caller owns every buffer.  The library allocates nothing,
 *   keeps no state between calls (apart from a diagnostic launch counter and a
 *   per-device SM-count cache) and is re-entrant.  All work is enqueued on
 *   `stream` and is asynchronous with respect to the host; results are valid
 *   once the stream has reached the end of the call.
 * - Synchronous errors (returned before anything is enqueued): a required
 *   pointer that is NULL or a negative size -> QAT_ERR_INVALID_ARGUMENT;
 *   a bit width other than 4 or 8, an unknown dtype / scheme / format ->
 *   QAT_ERR_UNSUPPORTED ([QAT] IntDtype::from_bits); a misaligned pointer ->
 *   QAT_ERR_MISALIGNED; a workspace smaller than qat_workspace_bytes() where
 *   the call needs one -> QAT_ERR_WORKSPACE; a failed CUDA launch ->
 *   QAT_ERR_CUDA.  n == 0 is a no-op that returns QAT_OK.
 * - Data errors are only known on the device.  Kernels OR the QAT_FLAG_* bits
 *   into *dev_flags (nullable; the caller zeroes it and reads it after the
 *   stream has passed the call).  A unit whose calibration fails, or whose
 *   given parameters are invalid, gets codes 0, y = +0 and mask bits 0; its
 *   scale is still written.
 */
#ifndef QAT_H
#define QAT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t / CUstream handle; NULL is the legacy default stream. */
typedef struct CUstream_st* qat_stream_t;

typedef enum {
  QAT_OK = 0,
  QAT_ERR_INVALID_ARGUMENT = 1, /* NULL required pointer, negative size, bad granularity/group */
  QAT_ERR_DIMENSION_MISMATCH = 2,
  QAT_ERR_UNSUPPORTED = 3,      /* bits not in {4, 8}; unknown dtype, scheme or format */
  QAT_ERR_CUDA = 4,             /* a CUDA launch or query failed */
  QAT_ERR_MISALIGNED = 5,       /* a pointer violates the alignment rule above */
  QAT_ERR_WORKSPACE = 6         /* workspace NULL or smaller than qat_workspace_bytes() */
} qat_status;

/* Device-side data flags (bitwise OR into *dev_flags). */
#define QAT_FLAG_NONFINITE_CALIB 1 /* NaN/Inf inside a unit being calibrated ([QAT] finite_min_max) */
#define QAT_FLAG_DEGENERATE 2      /* absmax == 0, zero range, or a scale that is 0 or inf
                                      ([QAT] from_absmax / from_minmax) */
#define QAT_FLAG_BAD_PARAMS 4      /* given scale not finite and > 0 (int) or not finite and >= 0
                                      (fp8), or given zero point outside [qmin, qmax] */
#define QAT_FLAG_NONFINITE_INPUT 8 /* NaN/Inf seen by an FP8 amax or by qat_amax_stats; informational */
#define QAT_FLAG_DEVICE_TIMEOUT 16 /* a kernel's bounded wait for its own staged copies ran out (an
                                      internal fault, not a data error); the call's outputs are
                                      invalid */

typedef enum { QAT_F32 = 0, QAT_BF16 = 1 } qat_dtype;
typedef enum { QAT_SYMMETRIC = 0, QAT_AFFINE = 1 } qat_scheme;
/*
 * Units of one parameter set in a row-major [rows, cols] tensor: the whole
 * tensor; each row (cols elements, [QAT] per_channel_params with the channel
 * axis first); consecutive groups of `group` elements inside a row; each
 * column (rows elements at stride cols, [QAT] per_channel_params /
 * fake_quant_int_per_channel with the channel axis 1; rows up to 2^36
 * elements long, QAT_ERR_UNSUPPORTED beyond).
 */
typedef enum {
  QAT_PER_TENSOR = 0,
  QAT_PER_ROW = 1,
  QAT_PER_GROUP = 2,
  QAT_PER_COLUMN = 3
} qat_granularity;
typedef enum { QAT_E4M3 = 0, QAT_E5M2 = 1 } qat_fp8_format;

/* Human-readable name of a status code (static string, never NULL). */
const char* qat_status_string(qat_status status);

/*
 * Bytes of device workspace a call may need: per tensor, the cross-block
 * partial statistics (16 KiB); per row / per group, five bytes per unit
 * (a dead byte and a zero point, each array rounded up to 16 bytes), used
 * only by the fallback for unit lengths the fused single-pass kernels do not
 * cover; per column, 21 bytes per column (a 16-byte statistics accumulator,
 * then the fallback's dead byte and zero point, each array rounded up to 16
 * bytes), used by every calibrated call.  The workspace is scratch: its contents on entry do not matter and
 * are overwritten.  Two calls that use the same workspace must be ordered on
 * one stream.
 */
size_t qat_workspace_bytes(int64_t rows, int64_t cols, qat_granularity granularity, int64_t group);

/*
 * Scale statistics of every unit ([QAT] finite_min_max; symmetric_from_absmax;
 * [MAR] absmax per channel): absmax = max |x|, minv / maxv = min / max, all
 * over the FINITE elements of the unit, with -0 ordered below +0.  A unit
 * without finite elements gives absmax 0, minv +inf, maxv -inf.  Outputs are
 * float[units], each nullable.  Any NaN/Inf sets QAT_FLAG_NONFINITE_INPUT.
 * workspace: qat_workspace_bytes(rows, cols, granularity, group) bytes
 * (per tensor and per column only).
 */
qat_status qat_amax_stats(const void* x, qat_dtype dtype, int64_t rows, int64_t cols,
                          qat_granularity granularity, int64_t group, float* absmax, float* minv,
                          float* maxv, int32_t* dev_flags, void* workspace, size_t workspace_bytes,
                          qat_stream_t stream);

/*
 * Integer fake quantization ([QAT] module docs "Integer quantization",
 * QuantParams::quantize / dequantize, fake_quant_int,
 * fake_quant_int_per_channel) fused with the STE window mask
 * ([QAT] real_min / real_max, fake_quant_backward).
 *
 *   bits 8 or 4; symmetric: [qmin,qmax] = [-127,127] / [-7,7], zp = 0;
 *   affine: [-128,127] / [-8,7].
 *   params_given == 0: calibrate every unit.  symmetric: scale = absmax / qmax;
 *     affine: rmin = min(min,0), rmax = max(max,0),
 *     scale = (rmax - rmin) / (qmax - qmin), zp = clamp(rne(qmin - rmin/scale)).
 *     scale[u] (and zero_point[u] if non-NULL) are written.
 *   params_given == 1: scale[u], zero_point[u] are read (zero_point may be
 *     NULL for symmetric).
 *   q = clamp(rne(x / scale) + zp, qmin, qmax)   (documented form: zp added
 *     after rounding);  y = (q - zp) * scale;
 *   mask bit = (x >= (qmin - zp) * scale) && (x <= (qmax - zp) * scale).
 *   With given parameters a NaN input gets code 0 and +-Inf the clamp ends;
 *   both get mask 0.
 * y, codes, mask are each nullable.  scale / zero_point have one entry per
 * unit.  workspace: qat_workspace_bytes(...) bytes.
 */
qat_status qat_fake_quant_int(const void* x, qat_dtype dtype, int64_t rows, int64_t cols, int bits,
                              qat_scheme scheme, qat_granularity granularity, int64_t group,
                              int params_given, float* scale, int32_t* zero_point, void* y,
                              void* codes, uint32_t* mask, int32_t* dev_flags, void* workspace,
                              size_t workspace_bytes, qat_stream_t stream);

/*
 * Calibration options for qat_fake_quant_int_opts.
 *   clip: the calibrated range times clip, in (0, 1] ([EDU] demo 2: the
 *     range c * max|x|, values beyond it clip to the end codes): the absmax
 *     (symmetric), or the min and the max (affine; 0 stays inside), times
 *     clip in one binary32 product, before the usual formulas.  1 is the
 *     plain calibration.
 *   scale_fp16: nonzero rounds every calibrated scale to binary16 (round to
 *     nearest, ties to even) and uses that value ([EDU] demo 3: one FP16
 *     scale per group); the zero point is derived from it; the scale array
 *     still holds fp32 (each value exactly representable in binary16).  A
 *     scale that rounds to 0 or to infinity is QAT_FLAG_DEGENERATE.
 */
typedef struct {
  float clip;
  int scale_fp16;
} qat_calib_options;

/*
 * Calibrated integer fake quantization (as qat_fake_quant_int with
 * params_given = 0) with calibration options (NULL: the plain calibration),
 * nearest (stochastic = 0) or stochastic rounding (the draws of
 * qat_fake_quant_int_sr).  Every granularity.  QAT_ERR_INVALID_ARGUMENT for
 * a clip outside (0, 1].
 */
qat_status qat_fake_quant_int_opts(const void* x, qat_dtype dtype, int64_t rows, int64_t cols,
                                   int bits, qat_scheme scheme, qat_granularity granularity,
                                   int64_t group, const qat_calib_options* options,
                                   int stochastic, uint64_t seed, uint64_t offset, float* scale,
                                   int32_t* zero_point, void* y, void* codes, uint32_t* mask,
                                   int32_t* dev_flags, void* workspace, size_t workspace_bytes,
                                   qat_stream_t stream);

/*
 * Per-tensor integer fake quantization calibrated by percentiles ([QAT]
 * QuantParams::per_tensor_percentile): the n values in the total order (-0
 * before +0), last = n - 1, the nearest-rank quantiles lo = sorted[floor(c *
 * last)] and hi = sorted[min(ceil((1 - c) * last), last)] (the index products
 * in binary64), then from_minmax: symmetric scale = max(|lo|, |hi|) / qmax,
 * affine the min/max calibration of [lo, hi].  Values beyond the quantiles
 * clamp to the end codes.  Outputs as qat_fake_quant_int (scale[0],
 * zero_point[0]), nearest (stochastic = 0) or stochastic rounding (the draws
 * of qat_fake_quant_int_sr).  A NaN or Inf anywhere is the module's
 * calibration error: QAT_FLAG_NONFINITE_CALIB, scale 0, codes 0, y = +0,
 * mask 0.  clip_fraction c outside [0, 0.5): QAT_ERR_INVALID_ARGUMENT; n up
 * to 2^40.  workspace: qat_percentile_workspace_bytes() bytes (the radix
 * select's histograms).  Five kernel launches: a reset, three radix-select
 * passes over x, then the map.
 */
size_t qat_percentile_workspace_bytes(void);
qat_status qat_fake_quant_int_percentile(const void* x, qat_dtype dtype, int64_t n, int bits,
                                         qat_scheme scheme, double clip_fraction, int stochastic,
                                         uint64_t seed, uint64_t offset, float* scale,
                                         int32_t* zero_point, void* y, void* codes,
                                         uint32_t* mask, int32_t* dev_flags, void* workspace,
                                         size_t workspace_bytes, qat_stream_t stream);

/*
 * Block-scaled floating-point fake quantization ([EDU] demo 4, block_scaled;
 * OCP MX formats and NVFP4).  One scale per block of `block` consecutive
 * elements (16 or 32; n a multiple of it), from the block's absmax over
 * finite values:
 *   QAT_BLOCK_SCALE_E8M0  X = 2^(floor(log2 amax) - emax) (amax 0: 2^-emax;
 *     the exponent held to [-127, 127]); block_scales: uint8 E8M0 codes
 *     (exponent + 127)  [MX];
 *   QAT_BLOCK_SCALE_E4M3  g = max|x| / (elem_max * 448) over the tensor
 *     (written to *tensor_scale), X = E4M3(amax / elem_max / g) * g with the
 *     saturating round to nearest even; block_scales: uint8 E4M3 codes
 *     [NVFP4: E2M1 elements, blocks of 16];
 *   QAT_BLOCK_SCALE_FP32  X = amax / elem_max; block_scales: float.
 *   A scale that is 0 or NaN becomes 1.
 * Elements: y = E(x / X) * X with E the saturating round to nearest even on
 * the element grid: E4M3 (max 448), E5M2 (57344), E2M3 (7.5), E3M2 (28),
 * E2M1 (6).  binary32 arithmetic, one rounding per operation in that order.
 * codes (nullable): one byte per element for FP8 / FP6 elements (the FP6 code
 * in the low 6 bits), two per byte for E2M1 (element 2j in the high nibble).
 * NaN elements: y NaN, code 0x7F (FP8) or 0 (FP6 / FP4); Inf saturates.
 * mask (nullable): bit set where |x / X| <= elem_max.  NaN or Inf in x sets
 * QAT_FLAG_NONFINITE_INPUT (informational).  *tensor_scale (nullable) is 1
 * for the E8M0 and FP32 kinds.  workspace: qat_workspace_bytes(1, n,
 * QAT_PER_TENSOR, 0) bytes for the E4M3 kind (its tensor statistics pass),
 * none otherwise.  One launch (two for E4M3).
 */
typedef enum {
  QAT_ELEM_E4M3 = 0,
  QAT_ELEM_E5M2 = 1,
  QAT_ELEM_E2M3 = 2,
  QAT_ELEM_E3M2 = 3,
  QAT_ELEM_E2M1 = 4
} qat_elem_format;
typedef enum {
  QAT_BLOCK_SCALE_E8M0 = 0,
  QAT_BLOCK_SCALE_E4M3 = 1,
  QAT_BLOCK_SCALE_FP32 = 2
} qat_block_scale;

qat_status qat_fake_quant_block(const void* x, qat_dtype dtype, int64_t n, qat_elem_format elem,
                                int64_t block, qat_block_scale scale_kind, float* tensor_scale,
                                void* y, uint8_t* codes, void* block_scales, uint32_t* mask,
                                int32_t* dev_flags, void* workspace, size_t workspace_bytes,
                                qat_stream_t stream);

/*
 * Per-tensor amax-scaled FP8 fake quantization ([QAT] fake_quant_fp8 /
 * fp8_quantize_magnitude; scale as in [MAR]).
 *   scale_given == 0: s = (max |x| over finite x) / fmt_max, written to *scale
 *     (fmt_max = 448 for E4M3, 57344 for E5M2); NaN/Inf in x set
 *     QAT_FLAG_NONFINITE_INPUT but are not an error.
 *   scale_given == 1: s = *scale (s = 1 gives the unscaled cast).
 *   t = x / s;  c = saturating round-to-nearest-even cast of t to the format
 *   (NaN -> NaN, +-Inf -> +-fmt_max, signed zero kept);  y = c * s;
 *   codes[i] = FP8 encoding of c (NaN encoded 0x7F);
 *   mask bit = |x| <= fmt_max * s (NaN -> 0).
 *   s == 0: non-NaN elements get code 0x00 and y = +0 (a zero scale encodes as
 *   byte 0); NaN stays NaN.  A given s that is negative, NaN or inf sets
 *   QAT_FLAG_BAD_PARAMS.
 * y is required; codes and mask are nullable.  scale: one device float.
 * workspace: qat_workspace_bytes(1, n, QAT_PER_TENSOR, 0) bytes when
 * scale_given == 0.
 */
qat_status qat_fake_quant_fp8(const void* x, qat_dtype dtype, int64_t n, qat_fp8_format format,
                              int scale_given, float* scale, void* y, uint8_t* codes,
                              uint32_t* mask, int32_t* dev_flags, void* workspace,
                              size_t workspace_bytes, qat_stream_t stream);

/*
 * Stochastic rounding ([QAT] RoundingMode::Stochastic, round_to_int): the
 * same operations as qat_fake_quant_int and qat_fake_quant_fp8 (same
 * arguments, calibration, window, layouts, flags and errors), with the
 * nearest rounding of r replaced by floor(r) + 1 when the element's draw
 * u < r - floor(r) and floor(r) otherwise (so E[round(r)] = r).
 *   int:  r = x / scale (binary32, IEEE); q = clamp(round(r) + zp, qmin, qmax).
 *   fp8:  r = a / ulp, a = |x / scale|, ulp = 2^(max(floor(log2 a), emin) - mbits)
 *         (an exact power-of-two scaling); magnitude round(r) * ulp, saturated
 *         at the format maximum; the sign of x / scale.
 * Draws: element i (flat index, 0-based) uses word i % 4 of Philox-4x32-10
 * (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC 2011; 10 rounds) with key (low, high 32 bits of seed) and counter
 * (low, high 32 bits of offset + i / 4, 0, 0); u = (word >> 9) * 2^-23, a
 * multiple of 2^-23 in [0, 1).  The draws depend only on (seed, offset, i):
 * results are reproducible and independent of the launch shape.  To draw
 * fresh numbers for a later call on the same seed, advance offset by at
 * least ceil(n / 4).
 */
qat_status qat_fake_quant_int_sr(const void* x, qat_dtype dtype, int64_t rows, int64_t cols,
                                 int bits, qat_scheme scheme, qat_granularity granularity,
                                 int64_t group, int params_given, float* scale, int32_t* zero_point,
                                 uint64_t seed, uint64_t offset, void* y, void* codes,
                                 uint32_t* mask, int32_t* dev_flags, void* workspace,
                                 size_t workspace_bytes, qat_stream_t stream);
qat_status qat_fake_quant_fp8_sr(const void* x, qat_dtype dtype, int64_t n, qat_fp8_format format,
                                 int scale_given, float* scale, uint64_t seed, uint64_t offset,
                                 void* y, uint8_t* codes, uint32_t* mask, int32_t* dev_flags,
                                 void* workspace, size_t workspace_bytes, qat_stream_t stream);

/*
 * One QAT optimizer step ([QAT] QatConfig, QatOptimizer::step + requantize):
 * an Adam / AdamW update of the fp32 master weights in place, then the
 * fake-quant view re-derived from the new master.
 *   master, grad, exp_avg, exp_avg_sq: float32[n] (master, first and second
 *     moments updated in place; grad read).  32-byte aligned.
 *   hp: host pointer; lr, beta1, beta2, eps, weight_decay as in QatConfig and
 *     bias_correction1/2 = 1 - beta1^t, 1 - beta2^t of this step t >= 1 (the
 *     module evaluates them in binary64; the caller passes them rounded to
 *     binary32).  Per element, in binary32 with one rounding per operation:
 *       m = beta1 m + (1 - beta1) g;  v = beta2 v + ((1 - beta2) g) g;
 *       m_hat = m / bc1;  v_hat = v / bc2;
 *       if weight_decay != 0: w = w - (lr weight_decay) w;
 *       w = w - (lr m_hat) / (sqrt(v_hat) + eps).
 *   view target: bits = 8 or 4 -> integer view calibrated per tensor over the
 *     new master (QuantParams::per_tensor_minmax with `scheme`), exactly
 *     qat_fake_quant_int per tensor on the new master (scale, zero_point
 *     written); bits = 0 -> FP8 view, the unscaled saturating cast in
 *     `format` (qat_fake_quant_fp8 with scale 1; *scale set to 1).
 *   stochastic != 0: stochastic rounding of the view with the draws of
 *     (seed, offset), as qat_fake_quant_int_sr / qat_fake_quant_fp8_sr.
 *   view: float32[n]; codes / mask (nullable) as the fake-quant calls;
 *     workspace (integer view only): qat_workspace_bytes(1, n,
 *     QAT_PER_TENSOR, 0) bytes.
 * Errors: hp NULL, a bias correction not finite and > 0, a NULL array ->
 * QAT_ERR_INVALID_ARGUMENT; bits not in {0, 4, 8} or an unknown format ->
 * QAT_ERR_UNSUPPORTED; alignment / workspace as above.  A non-finite new
 * master value flags QAT_FLAG_NONFINITE_CALIB for an integer view (the
 * module's calibration error) and gives codes 0, view +0, mask 0.
 * Two kernel launches: the update (with the view's statistics) and the view.
 */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
  float bias_correction1, bias_correction2;
} qat_adam_hparams;

qat_status qat_optimizer_step(float* master, const float* grad, float* exp_avg, float* exp_avg_sq,
                              int64_t n, const qat_adam_hparams* hp, int bits, qat_scheme scheme,
                              qat_fp8_format format, int stochastic, uint64_t seed,
                              uint64_t offset, float* view, void* codes, uint32_t* mask,
                              float* scale, int32_t* zero_point, int32_t* dev_flags,
                              void* workspace, size_t workspace_bytes, qat_stream_t stream);

/*
 * Straight-through-estimator backward ([QAT] fake_quant_backward) with the
 * window precomputed as the mask of a forward call: grad_in[i] = grad[i]
 * (bit copy) where the mask bit is set, +0 elsewhere.  grad and grad_in have
 * dtype `dtype` and n elements; mask has ceil(n / 32) words.
 */
qat_status qat_ste_backward(const void* grad, qat_dtype dtype, int64_t n, const uint32_t* mask,
                            void* grad_in, qat_stream_t stream);

/*
 * Two-level 4-bit quantization ([DQ] quantize_4bit_double).
 *   Level 1, per 64-element block (the last one may be short):
 *     scale = (max |x| over the block) / 7, code = clamp(round(x / scale), -8, 7)
 *     with round half away from zero; a zero scale gives code 0; NaN -> 0.
 *   Level 2, per 256 block scales (the last group may be short):
 *     super = max(max scale, 1e-8), qscale = clamp(round(scale / super * 255), 0, 255).
 *   data: ceil(n/2) bytes of packed codes; qscales: ceil(n/64) bytes;
 *   super_scales: ceil(ceil(n/64) / 256) floats.
 *   y_roundtrip (nullable): n floats receiving dequantize_4bit_double of the
 *   result, produced in the same pass.
 */
qat_status qat_quant4_double(const float* x, int64_t n, uint8_t* data, uint8_t* qscales,
                             float* super_scales, float* y_roundtrip, qat_stream_t stream);

/*
 * Dequantization of the two-level 4-bit format ([DQ] reconstruct_scales,
 * dequantize_4bit_double): scale = f32(qscale) / 255 * super (two roundings,
 * in that order), y = f32(code) * scale.
 */
qat_status qat_dequant4_double(const uint8_t* data, const uint8_t* qscales,
                               const float* super_scales, int64_t n, float* y, qat_stream_t stream);

/*
 * qat_fake_quant_fp8 without a workspace, for callers that cannot allocate
 * device memory: code embedded in a host framework that owns every device
 * allocation and passes the library only the tensors it works on, or a
 * latency-critical loop that must not call cudaMalloc (which can synchronise
 * the device).  There is no counterpart on the source pages; the arithmetic
 * and the outputs are exactly those of qat_fake_quant_fp8.
 *
 * The amax pass keeps its cross-block partials in a fixed file-scope device
 * array of 1024 slots x 16 bytes (16 KiB), reserved on every GPU that loads the
 * library until the process exits.  The statistics pass uses one slot per
 * block and its grid is capped at 1024 blocks (2 x the SM count on current
 * devices), so every n up to the library's limit of 2^50 elements fits; a
 * larger n is QAT_ERR_INVALID_ARGUMENT.  Nothing is allocated and nothing
 * needs clearing: every slot a call reads is written earlier in the same call.
 * All calls share the array, so calls whose kernels overlap on the GPU (other
 * streams, other host threads on the same device) race and must be ordered by
 * the caller.  Each call looks up the array's device address in the context
 * current at the call (the address belongs to that context); the first call
 * in a context may load the library's device code into it, so make that first
 * call before any stream capture begins.  A failed lookup is QAT_ERR_CUDA.
 * Arguments and errors as qat_fake_quant_fp8, minus the workspace.
 */
qat_status qat_fake_quant_fp8_noalloc(const void* x, qat_dtype dtype, int64_t n,
                                      qat_fp8_format format, int scale_given, float* scale,
                                      void* y, uint8_t* codes, uint32_t* mask, int32_t* dev_flags,
                                      qat_stream_t stream);

/* Number of kernels this library has launched in this process (diagnostic). */
uint64_t qat_kernel_launch_count(void);

/*
 * Testing hook, no counterpart on the source pages: the number of polls a
 * bounded device wait makes before it gives up, for the calls launched after
 * this one in the process (a process-wide setting).  The waits are the grid
 * barrier of the single-launch per-tensor path and the staged-copy waits of the
 * per-column kernels; a wait that runs out sets QAT_FLAG_DEVICE_TIMEOUT in the
 * call's dev_flags and its block returns early, leaving the call's outputs
 * undefined (a block always drains the copies it has issued before it
 * returns, with the default limit).  polls < 0 restores the default (2^24
 * polls, a fraction of a second); 0 makes every such wait give up at once.
 */
void qat_debug_set_wait_limit(int64_t polls);

#ifdef __cplusplus
}
#endif

#endif /* QAT_H */
