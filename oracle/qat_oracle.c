/*
 * qat_oracle.c -- CPU oracle for the fake-quant / STE / 4-bit double-quant path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct CPU
 * statement of what the sources define.  Only the test-suite, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  The CUDA library shares
 * no code, header, table or helper with it.
 *
 * Two evaluation modes:
 *   O32  -- every + - * / is one IEEE binary32 operation, round-to-nearest-even,
 *           no FMA contraction, no flush-to-zero (build with
 *           -O2 -ffp-contract=off -fno-fast-math).  This is the bit-exact
 *           reference for the GPU library.
 *   O64  -- the same formulas evaluated in binary64 on the same inputs, as the
 *           QAT module does; used only as a tolerance reference.
 *
 * Sources (cited by page and item):
 *   [QAT]  optirs-gpu 0.3.2, src/optirs_gpu/quantization.rs  (module docs,
 *          IntDtype::q_range, QuantParams::{from_minmax, from_absmax, quantize,
 *          dequantize, real_min, real_max}, finite_min_max, fake_quant_int,
 *          per_channel_params, fp8_quantize_magnitude, fake_quant_fp8,
 *          fake_quant_backward)
 *   [DQ]   aprender-train 0.32.0, src/entrenar/quant/double_quant.rs
 *          (quantize_4bit_double, reconstruct_scales, dequantize_4bit_double,
 *          DoubleQuantized4Bit::memory_bytes)
 *   [MAR]  ferrum-kernels 0.8.0, src/marlin_repack.rs (per-channel E4M3 scale
 *          absmax/448, zero scale -> code 0)
 *   [EDU]  cs349e 05_quantization_basics.py, demo 3 (groups run along the last
 *          dimension)
 *   [QAT] RoundingMode::{Nearest, Stochastic}::round_to_int (stochastic
 *          rounding), with the uniform draws from a counter-based generator:
 *   [PHX]  Philox-4x32-10, J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel
 *          random numbers: as easy as 1, 2, 3", SC 2011 (the round function
 *          and the Weyl key schedule as published)
 *   [QAT]  QatConfig, QatOptimizer::{step, requantize} (Adam/AdamW update of
 *          the master weights, then the fake-quant view)
 *   [QAT]  QuantParams::per_tensor_percentile (nearest-rank quantiles, then
 *          from_minmax); per_channel_params with axis 1 (per-column units)
 *   [EDU]  demo 2 (the range c * max|x|: clip factor), demo 3 (one FP16
 *          scale per group); IEEE 754 binary16 (round to nearest, ties to even)
 *   [EDU]  demo 4, block_scaled (E8M0 / E4M3 + FP32 / exact block scales)
 *   [MX]   OCP Microscaling Formats (MX) Specification v1.0 (the FP8 / FP6 /
 *          FP4 element encodings, E8M0 scales); NVIDIA NVFP4 (E2M1 elements,
 *          16-element blocks, E4M3 block scales under an FP32 tensor scale)
 *
 * Every place where the sources are silent and a reading was taken is marked
 * "reading:" below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* status codes (the same meaning as the library's, defined independently) */
#define OR_OK 0
#define OR_ERR_INVALID 1
#define OR_ERR_DIM 2
#define OR_ERR_UNSUPPORTED 3

/* data flags OR-ed into *flags */
#define OR_FLAG_NONFINITE 1       /* [QAT] finite_min_max: non-finite value in a calibrated unit */
#define OR_FLAG_DEGENERATE 2      /* [QAT] from_absmax / from_minmax: zero range or scale <= 0 / inf */
#define OR_FLAG_BAD_PARAMS 4      /* caller-given scale / zero point outside the valid domain */
#define OR_FLAG_NONFINITE_INPUT 8 /* FP8 path: NaN/Inf seen while taking amax (not an error) */

#define OR_F32 0
#define OR_BF16 1
#define OR_SYM 0
#define OR_AFFINE 1
#define OR_PER_TENSOR 0
#define OR_PER_ROW 1
#define OR_PER_GROUP 2
#define OR_PER_COLUMN 3
#define OR_E4M3 0
#define OR_E5M2 1

int or_dequant4_double(const uint8_t* data, const uint8_t* qscales, const float* supers, int64_t n,
                       float* y);

/* ------------------------------------------------------------------------- */
/* bit-level helpers                                                          */
/* ------------------------------------------------------------------------- */

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 is the upper half of a binary32 pattern: widening is exact. */
static float bf16_to_f32(uint16_t h) { return u2f((uint32_t)h << 16); }

/* binary32 -> bf16, round to nearest even on the bit pattern; NaN becomes the
 * canonical quiet NaN 0x7FC0.  reading: outputs are computed in fp32 and
 * rounded once to the output dtype. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = f2u(f);
  if (isnan(f)) return 0x7FC0;
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static float load_elem(const void* x, int dtype, int64_t i) {
  if (dtype == OR_BF16) return bf16_to_f32(((const uint16_t*)x)[i]);
  return ((const float*)x)[i];
}

/* reading: a NaN output is the canonical positive quiet NaN (the QAT module
 * returns f64::NAN). */
static void store_elem(void* y, int dtype, int64_t i, float v) {
  if (dtype == OR_BF16) {
    ((uint16_t*)y)[i] = f32_to_bf16_rne(v);
  } else {
    ((float*)y)[i] = isnan(v) ? u2f(0x7FC00000u) : v;
  }
}

/* Total order on finite values with -0 < +0.  reading: min/max of a unit must
 * not depend on visiting order, so the two zeros are ordered. */
static int less_total(float a, float b) {
  if (a < b) return 1;
  if (a == b && signbit(a) && !signbit(b)) return 1;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* [QAT] IntDtype::from_bits + IntDtype::q_range                              */
/* symmetric uses the restricted range, affine the full two's-complement one. */
/* ------------------------------------------------------------------------- */
int or_q_range(int bits, int scheme, int32_t* qmin, int32_t* qmax) {
  if (bits != 8 && bits != 4) return OR_ERR_UNSUPPORTED;
  if (scheme != OR_SYM && scheme != OR_AFFINE) return OR_ERR_INVALID;
  if (bits == 8) {
    *qmin = (scheme == OR_SYM) ? -127 : -128;
    *qmax = 127;
  } else {
    *qmin = (scheme == OR_SYM) ? -7 : -8;
    *qmax = 7;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* [QAT] finite_min_max / symmetric_from_absmax: statistics of one unit.      */
/* The module stops at the first non-finite value; the oracle folds over the  */
/* finite ones and counts the rest, so the caller can decide (int path:       */
/* error flag; FP8 path: informational).                                      */
/* An empty fold leaves min=+inf, max=-inf, absmax=0.                         */
/* ------------------------------------------------------------------------- */
/* elements off, off + stride, ..., off + (len - 1) stride */
void or_unit_stats_strided(const void* x, int dtype, int64_t off, int64_t len, int64_t stride,
                           float* mn, float* mx, float* amax, int64_t* nonfinite) {
  float m = INFINITY, M = -INFINITY, A = 0.0f;
  int64_t bad = 0;
  for (int64_t i = 0; i < len; ++i) {
    float v = load_elem(x, dtype, off + i * stride);
    if (!isfinite(v)) { bad++; continue; }
    if (less_total(v, m)) m = v;
    if (less_total(M, v)) M = v;
    float a = fabsf(v);
    if (a > A) A = a;
  }
  *mn = m; *mx = M; *amax = A; *nonfinite = bad;
}

void or_unit_stats(const void* x, int dtype, int64_t off, int64_t len, float* mn, float* mx,
                   float* amax, int64_t* nonfinite) {
  or_unit_stats_strided(x, dtype, off, len, 1, mn, mx, amax, nonfinite);
}

/* ------------------------------------------------------------------------- */
/* [QAT] QuantParams::from_absmax: scale = absmax / qmax, zero point 0.       */
/* Returns 0 on success, OR_FLAG_DEGENERATE when absmax <= 0 or the scale is  */
/* not a positive finite number.                                              */
/* ------------------------------------------------------------------------- */
/* ------------------------------------------------------------------------- */
/* IEEE binary16 rounding of a binary32 value (round to nearest, ties to     */
/* even): the grid step is 2^(e-10) for a normal binary16 exponent e in      */
/* [-14, 15] and 2^-24 below 2^-14 (subnormals); a magnitude that rounds past */
/* the largest finite value 65504 (i.e. >= 65520) becomes infinity.  x / step */
/* and k * step are exact power-of-two scalings in binary32.  Used for fp16   */
/* group scales ([EDU] demo 3: one FP16 scale per group).                     */
/* ------------------------------------------------------------------------- */
float or_round_fp16(float x) {
  if (isnan(x) || isinf(x) || x == 0.0f) return x;
  float a = fabsf(x);
  if (a >= 65520.0f) return copysignf(INFINITY, x);
  int e;
  frexpf(a, &e); /* a = f * 2^e, f in [0.5, 1): the binary exponent is e - 1 */
  int ex = e - 1;
  if (ex < -14) ex = -14; /* subnormal binary16: step 2^-24 */
  float step = ldexpf(1.0f, ex - 10);
  float k = rintf(a / step);
  return copysignf(k * step, x);
}

int or_params_from_absmax(float absmax, int32_t qmax, float* scale) {
  if (!(absmax > 0.0f) || isinf(absmax)) { *scale = absmax / (float)qmax; return OR_FLAG_DEGENERATE; }
  float s = absmax / (float)qmax;
  *scale = s;
  if (!(s > 0.0f) || isinf(s)) return OR_FLAG_DEGENERATE;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* [QAT] QuantParams::from_minmax, affine branch: nudge [min,max] to include  */
/* 0, scale = (rmax - rmin) / (qmax - qmin),                                  */
/* zero_point = clamp(rne(qmin - rmin / scale), qmin, qmax).                  */
/* ------------------------------------------------------------------------- */
int or_params_affine(float mn, float mx, int32_t qmin, int32_t qmax, float* scale, int32_t* zp) {
  float rmin = (mn < 0.0f) ? mn : 0.0f;
  float rmax = (mx > 0.0f) ? mx : 0.0f;
  float range = rmax - rmin;
  float s = range / (float)(qmax - qmin);
  *scale = s;
  *zp = 0;
  if (!(range > 0.0f)) return OR_FLAG_DEGENERATE;
  if (!(s > 0.0f) || isinf(s)) return OR_FLAG_DEGENERATE;
  float t = (float)qmin - rmin / s;
  float z = rintf(t);
  if (z < (float)qmin) z = (float)qmin;
  if (z > (float)qmax) z = (float)qmax;
  *zp = (int32_t)z;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* [QAT] QuantParams::quantize.                                               */
/* The module docs write quant(x) = clamp(round(x/scale) + zp, qmin, qmax);   */
/* the code adds zp before rounding.  reading: the documented form, the only  */
/* one for which the zero point cancels exactly in the round trip, as the     */
/* docs state.  doc_form = 0 selects the code's form for comparison.          */
/* A NaN quotient gives code 0 (a NaN clamped and cast to i32 is 0).          */
/* ------------------------------------------------------------------------- */
int32_t or_quantize(float x, float scale, int32_t zp, int32_t qmin, int32_t qmax, int doc_form) {
  float r = x / scale;
  if (doc_form) {
    if (isnan(r)) return 0;
    float k = rintf(r);
    float lo = (float)(qmin - zp), hi = (float)(qmax - zp);
    if (k < lo) k = lo;
    if (k > hi) k = hi;
    return (int32_t)k + zp;
  } else {
    float t = r + (float)zp;
    if (isnan(t)) return 0;
    float k = rintf(t);
    if (k < (float)qmin) k = (float)qmin;
    if (k > (float)qmax) k = (float)qmax;
    return (int32_t)k;
  }
}

/* [QAT] QuantParams::dequantize: (q - zp) * scale. */
float or_dequantize(int32_t q, float scale, int32_t zp) { return (float)(q - zp) * scale; }

/* [QAT] real_min / real_max + fake_quant_backward: inclusive window. */
static int in_window(float x, float scale, int32_t zp, int32_t qmin, int32_t qmax) {
  float lo = or_dequantize(qmin, scale, zp);
  float hi = or_dequantize(qmax, scale, zp);
  if (lo > hi) { float t = lo; lo = hi; hi = t; }
  return (x >= lo && x <= hi) ? 1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Stochastic rounding.                                                       */
/* [QAT] RoundingMode::Stochastic: lower = floor(r), frac = r - lower, the    */
/* result is lower + 1 when the draw u < frac and lower otherwise, so that    */
/* E[round(r)] = r.  reading: the module draws u in [0, 1) from a caller's    */
/* Rng in element order; here the draw of element i of a call is a function   */
/* of (seed, offset, i) alone, so that any evaluation order gives the same    */
/* result:                                                                    */
/*   w = word (i mod 4) of Philox-4x32-10 [PHX] with key (lo32 seed,          */
/*       hi32 seed) and counter (lo32 j, hi32 j, 0, 0), j = offset + i / 4;   */
/*   u = (w >> 9) * 2^-23, a multiple of 2^-23 in [0, 1).                     */
/* A caller advances offset by ceil(n / 4) per call for fresh draws.  In      */
/* binary32, frac = r - floor(r) is exact (Sterbenz) and so is u, so the      */
/* decision u < frac is exact.                                                */
/* ------------------------------------------------------------------------- */
void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    /* [PHX] Philox S-box: two 32x32 -> 64-bit products with the round
     * multipliers, high halves mixed with the other words and the key. */
    uint64_t p0 = (uint64_t)0xD2511F53u * x0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * x2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ x1 ^ k0;
    uint32_t n2 = hi0 ^ x3 ^ k1;
    x0 = n0;
    x1 = lo1;
    x2 = n2;
    x3 = lo0;
    /* [PHX] Weyl sequence key schedule */
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

float or_sr_uniform(uint64_t seed, uint64_t offset, int64_t i) {
  uint64_t j = offset + (uint64_t)i / 4u;
  uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), 0u, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  or_philox4x32_10(ctr, key, out);
  return (float)(out[i & 3] >> 9) * 0x1p-23f;
}

/* [QAT] round_to_int, Stochastic arm, in binary32.  NaN stays NaN; for an
 * infinite r, frac is NaN and the comparison is false, so r itself is
 * returned (as floor(+-inf) is +-inf). */
float or_sr_round(float r, float u) {
  float lower = floorf(r);
  float frac = r - lower;
  return (u < frac) ? lower + 1.0f : lower;
}

/* QuantParams::quantize with stochastic rounding, in the documented form
 * (the zero point is added after rounding, as for or_quantize). */
int32_t or_quantize_sr(float x, float scale, int32_t zp, int32_t qmin, int32_t qmax, float u) {
  float r = x / scale;
  if (isnan(r)) return 0;
  float k = or_sr_round(r, u);
  float lo = (float)(qmin - zp), hi = (float)(qmax - zp);
  if (k < lo) k = lo;
  if (k > hi) k = hi;
  return (int32_t)k + zp;
}

static void set_code(void* codes, int bits, int64_t i, int32_t q) {
  if (!codes) return;
  if (bits == 8) {
    ((int8_t*)codes)[i] = (int8_t)q;
  } else {
    /* reading: two 4-bit codes per byte, element 2j in the high nibble and
     * 2j+1 in the low nibble, two's complement ([DQ] dequantize_4bit_double). */
    uint8_t* b = (uint8_t*)codes + (i >> 1);
    uint8_t nib = (uint8_t)(q & 0xF);
    if ((i & 1) == 0) *b = (uint8_t)((*b & 0x0F) | (nib << 4));
    else *b = (uint8_t)((*b & 0xF0) | nib);
  }
}

static void set_mask(uint32_t* mask, int64_t i, int bit) {
  if (!mask) return;
  uint32_t w = mask[i >> 5];
  uint32_t b = 1u << (i & 31);
  mask[i >> 5] = bit ? (w | b) : (w & ~b);
}

/* ------------------------------------------------------------------------- */
/* [QAT] fake_quant_int / per_channel_params / fake_quant_int_per_channel,    */
/* restated for a row-major [rows, cols] tensor whose units are the whole     */
/* tensor, each row (axis 0), or each run of `group` elements along the last  */
/* dimension ([EDU] demo 3).                                                  */
/*                                                                            */
/* params_given = 0: calibrate every unit (scale, zp written);                */
/*              = 1: read scale[u], zp[u].                                    */
/* Outputs (each nullable): y (dtype of x), codes (int8[n] for 8 bits, packed */
/* uint8[ceil(n/2)] for 4 bits), mask words (bit i%32 of word i/32).          */
/* A unit that fails calibration (flag set) or has invalid given params gets  */
/* codes 0, y = +0, mask 0.  reading: the module returns an error there.      */
/* ------------------------------------------------------------------------- */
/* Calibration with the range options: the observed absmax (symmetric) or
 * min and max (affine) times the clip factor c, one binary32 product each
 * ([EDU] demo 2: the range c * max|x|, values beyond it clip; reading: for
 * the affine scheme the same factor scales both ends, so 0 stays inside);
 * with fp16 set the scale is rounded to binary16 and that value is the
 * unit's scale (reading of the FP16 group scales of [EDU] demo 3), the zero
 * point derived from it.  c = 1 and fp16 = 0 are the module's calibration. */
static int calib_opts(int scheme, float mn, float mx, float A, int32_t qmin, int32_t qmax, float c,
                      int fp16, float* s, int32_t* z) {
  int flag;
  if (scheme == OR_SYM) {
    *z = 0;
    float Ac = (c == 1.0f) ? A : c * A;
    if (!fp16) return or_params_from_absmax(Ac, qmax, s);
    flag = or_params_from_absmax(Ac, qmax, s);
    *s = or_round_fp16(*s);
    if (!flag && (!(*s > 0.0f) || isinf(*s))) flag = OR_FLAG_DEGENERATE;
    return flag;
  }
  if (c != 1.0f) {
    mn = c * mn;
    mx = c * mx;
  }
  if (!fp16) return or_params_affine(mn, mx, qmin, qmax, s, z);
  /* from_minmax with the binary16 scale */
  float rmin = (mn < 0.0f) ? mn : 0.0f;
  float rmax = (mx > 0.0f) ? mx : 0.0f;
  float range = rmax - rmin;
  *s = or_round_fp16(range / (float)(qmax - qmin));
  *z = 0;
  if (!(range > 0.0f)) return OR_FLAG_DEGENERATE;
  if (!(*s > 0.0f) || isinf(*s)) return OR_FLAG_DEGENERATE;
  float t = (float)qmin - rmin / *s;
  float zz = rintf(t);
  if (zz < (float)qmin) zz = (float)qmin;
  if (zz > (float)qmax) zz = (float)qmax;
  *z = (int32_t)zz;
  return 0;
}

static int fq_int(const void* x, int dtype, int64_t rows, int64_t cols, int bits, int scheme,
                  int gran, int64_t group, int params_given, float* scale, int32_t* zp, void* y,
                  void* codes, uint32_t* mask, int32_t* flags, int doc_form, int stochastic,
                  uint64_t seed, uint64_t offset, float clip, int fp16) {
  int32_t qmin, qmax;
  int st = or_q_range(bits, scheme, &qmin, &qmax);
  if (st) return st;
  if (rows < 0 || cols < 0) return OR_ERR_INVALID;
  int64_t n = rows * cols;
  /* unit u holds L elements: start(u) + k * stride, k < L */
  int64_t L, stride = 1, units;
  if (gran == OR_PER_TENSOR) L = n;
  else if (gran == OR_PER_ROW) L = cols;
  else if (gran == OR_PER_GROUP) {
    if (group <= 0 || cols % group != 0) return OR_ERR_INVALID;
    L = group;
  } else if (gran == OR_PER_COLUMN) {
    /* [QAT] per_channel_params / fake_quant_int_per_channel with axis 1:
     * each column is a channel, calibrated from that column only */
    L = rows;
    stride = cols;
  } else return OR_ERR_INVALID;
  if (n == 0) return OR_OK;
  if (codes && bits == 4) memset(codes, 0, (size_t)((n + 1) / 2));
  if (mask) memset(mask, 0, (size_t)((n + 31) / 32) * 4);
  units = gran == OR_PER_COLUMN ? cols : n / L;
  for (int64_t u = 0; u < units; ++u) {
    int64_t off = gran == OR_PER_COLUMN ? u : u * L;
    float s;
    int32_t z;
    int flag = 0;
    if (params_given) {
      s = scale[u];
      z = (scheme == OR_SYM) ? 0 : zp[u];
      if (!(s > 0.0f) || isinf(s) || z < qmin || z > qmax) flag = OR_FLAG_BAD_PARAMS;
    } else {
      float mn, mx, A;
      int64_t bad;
      or_unit_stats_strided(x, dtype, off, L, stride, &mn, &mx, &A, &bad);
      flag = calib_opts(scheme, mn, mx, A, qmin, qmax, clip, fp16, &s, &z);
      if (bad) flag = OR_FLAG_NONFINITE;
      scale[u] = s;
      if (zp) zp[u] = z;
    }
    if (flag && flags) *flags |= flag;
    for (int64_t k = 0; k < L; ++k) {
      int64_t i = off + k * stride;
      float v = load_elem(x, dtype, i);
      if (flag) {
        set_code(codes, bits, i, 0);
        if (y) store_elem(y, dtype, i, 0.0f);
        set_mask(mask, i, 0);
        continue;
      }
      int32_t q = stochastic
                      ? or_quantize_sr(v, s, z, qmin, qmax, or_sr_uniform(seed, offset, i))
                      : or_quantize(v, s, z, qmin, qmax, doc_form);
      set_code(codes, bits, i, q);
      if (y) store_elem(y, dtype, i, or_dequantize(q, s, z));
      set_mask(mask, i, in_window(v, s, z, qmin, qmax));
    }
  }
  return OR_OK;
}

int or_fake_quant_int(const void* x, int dtype, int64_t rows, int64_t cols, int bits, int scheme,
                      int gran, int64_t group, int params_given, float* scale, int32_t* zp,
                      void* y, void* codes, uint32_t* mask, int32_t* flags, int doc_form) {
  return fq_int(x, dtype, rows, cols, bits, scheme, gran, group, params_given, scale, zp, y, codes,
                mask, flags, doc_form, 0, 0, 0, 1.0f, 0);
}

/* The same with stochastic rounding: element i rounds with the draw
 * or_sr_uniform(seed, offset, i); calibration and the STE window are those of
 * the nearest-rounding path. */
int or_fake_quant_int_sr(const void* x, int dtype, int64_t rows, int64_t cols, int bits,
                         int scheme, int gran, int64_t group, int params_given, float* scale,
                         int32_t* zp, uint64_t seed, uint64_t offset, void* y, void* codes,
                         uint32_t* mask, int32_t* flags) {
  return fq_int(x, dtype, rows, cols, bits, scheme, gran, group, params_given, scale, zp, y, codes,
                mask, flags, 1, 1, seed, offset, 1.0f, 0);
}

/* Calibrated integer fake quant with the range options (clip factor c in
 * (0, 1], binary16 scales), nearest or stochastic rounding. */
int or_fake_quant_int_opts(const void* x, int dtype, int64_t rows, int64_t cols, int bits,
                           int scheme, int gran, int64_t group, float clip, int fp16,
                           int stochastic, uint64_t seed, uint64_t offset, float* scale,
                           int32_t* zp, void* y, void* codes, uint32_t* mask, int32_t* flags) {
  if (!(clip > 0.0f) || !(clip <= 1.0f)) return OR_ERR_INVALID;
  return fq_int(x, dtype, rows, cols, bits, scheme, gran, group, 0, scale, zp, y, codes, mask,
                flags, 1, stochastic, seed, offset, clip, fp16);
}

/* ------------------------------------------------------------------------- */
/* [QAT] QuantParams::per_tensor_percentile: the values sorted in the total   */
/* order (-0 before +0), last = n - 1, the nearest-rank quantiles             */
/* lo = sorted[floor(c * last)] and hi = sorted[min(ceil((1 - c) * last),     */
/* last)] with the index products in binary64 as printed, then from_minmax:   */
/* symmetric from_absmax(max(|lo|, |hi|)), affine the min/max calibration.    */
/* c outside [0, 0.5) is an error; a non-finite value anywhere is the         */
/* module's calibration error, reported as OR_FLAG_NONFINITE (the tensor is   */
/* then a failed unit: codes 0, y = +0, mask 0).                              */
/* ------------------------------------------------------------------------- */
static int cmp_total(const void* a, const void* b) {
  float x = *(const float*)a, y = *(const float*)b;
  if (x < y) return -1;
  if (x > y) return 1;
  /* equal values: only the zeros differ, -0 first */
  return (int)(signbit(y) != 0) - (int)(signbit(x) != 0);
}

int or_percentile_minmax(const void* x, int dtype, int64_t n, double clip_fraction, float* lo,
                         float* hi, int32_t* flags) {
  if (!(clip_fraction >= 0.0 && clip_fraction < 0.5)) return OR_ERR_INVALID;
  if (n <= 0) return OR_ERR_INVALID;
  float* v = (float*)malloc((size_t)n * sizeof(float));
  if (!v) return OR_ERR_INVALID;
  int bad = 0;
  for (int64_t i = 0; i < n; ++i) {
    v[i] = load_elem(x, dtype, i);
    if (!isfinite(v[i])) bad = 1;
  }
  if (bad) {
    free(v);
    *lo = *hi = 0.0f;
    if (flags) *flags |= OR_FLAG_NONFINITE;
    return OR_OK;
  }
  qsort(v, (size_t)n, sizeof(float), cmp_total);
  int64_t last = n - 1;
  int64_t lo_idx = (int64_t)floor(clip_fraction * (double)last);
  int64_t hi_idx = (int64_t)ceil((1.0 - clip_fraction) * (double)last);
  if (lo_idx > last) lo_idx = last;
  if (hi_idx > last) hi_idx = last;
  *lo = v[lo_idx];
  *hi = v[hi_idx];
  free(v);
  return OR_OK;
}

/* Per-tensor fake quant of x[n] calibrated by per_tensor_percentile, nearest
 * or stochastic rounding (elements beyond the quantiles clamp to the code
 * range). */
int or_fake_quant_int_percentile(const void* x, int dtype, int64_t n, int bits, int scheme,
                                 double clip_fraction, int stochastic, uint64_t seed,
                                 uint64_t offset, float* scale, int32_t* zp, void* y, void* codes,
                                 uint32_t* mask, int32_t* flags) {
  int32_t qmin, qmax;
  int st = or_q_range(bits, scheme, &qmin, &qmax);
  if (st) return st;
  if (!(clip_fraction >= 0.0 && clip_fraction < 0.5) || n < 0) return OR_ERR_INVALID;
  if (n == 0) return OR_OK;
  float lo, hi;
  int32_t f = 0;
  st = or_percentile_minmax(x, dtype, n, clip_fraction, &lo, &hi, &f);
  if (st) return st;
  float s;
  int32_t z = 0;
  int flag;
  if (f) {
    flag = OR_FLAG_NONFINITE;
    s = 0.0f;
  } else if (scheme == OR_SYM) {
    flag = or_params_from_absmax(fmaxf(fabsf(lo), fabsf(hi)), qmax, &s);
  } else {
    flag = or_params_affine(lo, hi, qmin, qmax, &s, &z);
  }
  *scale = s;
  if (zp) *zp = z;
  if (flags) *flags |= flag;
  if (codes && bits == 4) memset(codes, 0, (size_t)((n + 1) / 2));
  if (mask) memset(mask, 0, (size_t)((n + 31) / 32) * 4);
  for (int64_t i = 0; i < n; ++i) {
    float v = load_elem(x, dtype, i);
    if (flag) {
      set_code(codes, bits, i, 0);
      if (y) store_elem(y, dtype, i, 0.0f);
      continue;
    }
    int32_t q = stochastic ? or_quantize_sr(v, s, z, qmin, qmax, or_sr_uniform(seed, offset, i))
                           : or_quantize(v, s, z, qmin, qmax, 1);
    set_code(codes, bits, i, q);
    if (y) store_elem(y, dtype, i, or_dequantize(q, s, z));
    set_mask(mask, i, in_window(v, s, z, qmin, qmax));
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Block-scaled floating-point formats ([EDU] demo 4, block_scaled).          */
/*                                                                            */
/* Element formats (the module's numfmt definitions are not on the pages;    */
/* written from the OCP Microscaling (MX) v1.0 and NVIDIA NVFP4 public        */
/* definitions): sign, `ebits` exponent bits with bias, `mbits` mantissa      */
/* bits, subnormals, largest finite value maxv; FP6 / FP4 have no Inf or NaN. */
/*   E4M3 (bias 7, max 448), E5M2 (15, 57344), E2M3 (1, 7.5), E3M2 (3, 28),   */
/*   E2M1 (1, 6); emax = floor(log2 maxv).                                    */
/* The page's steps, per block of `block` consecutive elements:               */
/*   amax = max |x| over the block;                                           */
/*   scale X:  E8M0 -- 2^(floor(log2 amax) - emax) (amax = 0: 2^-emax, the    */
/*               page's frexp(1.0) branch);                                   */
/*             E4M3 -- g = max|x| over the tensor / (maxv * 448),             */
/*               X = E4M3_round_sat(amax / maxv / g) * g (NVFP4);             */
/*             FP32 -- X = amax / maxv;                                       */
/*             X <= 0 or NaN -> 1;                                            */
/*   y = x / X; out = round_sat(y) * X (round to nearest even on the element  */
/*   grid, magnitudes past maxv saturate).                                    */
/* reading: binary32 throughout with one rounding per printed operation (the  */
/* page computes in binary64); amax and the tensor max over finite values; a  */
/* NaN element stays NaN (code 0x7F for FP8 elements, 0 for FP6 / FP4), an   */
/* Inf saturates; the E8M0 exponent is held to [-127, 127]; the STE mask bit  */
/* is |y| <= maxv.                                                            */
/* ------------------------------------------------------------------------- */
typedef struct {
  int ebits, mbits, bias, emax;
  float maxv;
} or_elemfmt;

static const or_elemfmt OR_ELEM[5] = {
    {4, 3, 7, 8, 448.0f},     /* E4M3 */
    {5, 2, 15, 15, 57344.0f}, /* E5M2 */
    {2, 3, 1, 2, 7.5f},       /* E2M3 */
    {3, 2, 3, 4, 28.0f},      /* E3M2 */
    {2, 1, 1, 2, 6.0f},       /* E2M1 */
};

/* round to nearest even on the element grid, saturating; sign kept */
float or_elem_round(float y, int fmt) {
  const or_elemfmt f = OR_ELEM[fmt];
  if (isnan(y)) return y;
  float a = fabsf(y);
  if (isinf(a)) return copysignf(f.maxv, y);
  if (a == 0.0f) return y;
  int emin = 1 - f.bias;
  int e = (int)((f2u(a) >> 23) & 0xFF) - 127; /* floor(log2 a); -127 for binary32 subnormals */
  int se = (e > emin ? e : emin) - f.mbits;
  float step = ldexpf(1.0f, se);
  float mag = rintf(a / step) * step;
  if (mag > f.maxv) mag = f.maxv;
  return copysignf(mag, y);
}

/* the element code of a grid value: sign, biased exponent, mantissa */
uint8_t or_elem_encode(float c, int fmt) {
  const or_elemfmt f = OR_ELEM[fmt];
  if (isnan(c)) return fmt <= 1 ? 0x7F : 0x00;
  uint8_t sign = signbit(c) ? (uint8_t)(1u << (f.ebits + f.mbits)) : 0;
  float a = fabsf(c);
  if (a == 0.0f) return sign;
  int emin = 1 - f.bias;
  int ex;
  (void)frexpf(a, &ex);
  int e = ex - 1;
  if (e < emin) return (uint8_t)(sign | (int)(a / ldexpf(1.0f, emin - f.mbits)));
  int man = (int)((a / ldexpf(1.0f, e) - 1.0f) * ldexpf(1.0f, f.mbits));
  return (uint8_t)(sign | ((e + f.bias) << f.mbits) | man);
}

/* The value of an element code (inverse of or_elem_encode on the grid). */
float or_elem_decode(uint8_t code, int fmt) {
  const or_elemfmt f = OR_ELEM[fmt];
  int nb = f.ebits + f.mbits;
  int sign = (code >> nb) & 1;
  int E = (code >> f.mbits) & ((1 << f.ebits) - 1);
  int M = code & ((1 << f.mbits) - 1);
  float mag = E == 0 ? ldexpf((float)M, 1 - f.bias - f.mbits)
                     : ldexpf(1.0f + ldexpf((float)M, -f.mbits), E - f.bias);
  return sign ? -mag : mag;
}

int or_fake_quant_block(const void* x, int dtype, int64_t n, int fmt, int64_t block, int kind,
                        float* tensor_scale, void* y, uint8_t* codes, void* bscales,
                        uint32_t* mask, int32_t* flags) {
  if (fmt < 0 || fmt > 4 || kind < 0 || kind > 2) return OR_ERR_UNSUPPORTED;
  if (block <= 0 || n < 0 || n % block != 0) return OR_ERR_INVALID;
  const or_elemfmt f = OR_ELEM[fmt];
  int nonfinite = 0;
  float A = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float v = load_elem(x, dtype, i);
    if (!isfinite(v)) nonfinite = 1;
    else if (fabsf(v) > A) A = fabsf(v);
  }
  float g = 1.0f;
  if (kind == 1) g = A / (f.maxv * 448.0f);
  if (tensor_scale) *tensor_scale = g;
  if (mask) memset(mask, 0, (size_t)((n + 31) / 32) * 4);
  for (int64_t b = 0; b < n / block; ++b) {
    float amax = 0.0f;
    for (int64_t k = 0; k < block; ++k) {
      float v = load_elem(x, dtype, b * block + k);
      if (isfinite(v) && fabsf(v) > amax) amax = fabsf(v);
    }
    float X;
    if (kind == 0) {
      int e = amax > 0.0f ? (int)((f2u(amax) >> 23) & 0xFF) - 127 : 0;
      if (amax > 0.0f && e == -127) { /* binary32 subnormal: its own exponent */
        int ex;
        (void)frexpf(amax, &ex);
        e = ex - 1;
      }
      int es = e - f.emax;
      if (es < -127) es = -127;
      if (es > 127) es = 127;
      X = ldexpf(1.0f, es);
      if (bscales) ((uint8_t*)bscales)[b] = (uint8_t)(es + 127);
    } else if (kind == 1) {
      float c = or_elem_round((amax / f.maxv) / g, 0);
      X = c * g;
      if (bscales) ((uint8_t*)bscales)[b] = or_elem_encode(c, 0);
    } else {
      X = amax / f.maxv;
    }
    if (!(X > 0.0f)) X = 1.0f;
    if (kind == 2 && bscales) ((float*)bscales)[b] = X;
    for (int64_t k = 0; k < block; ++k) {
      int64_t i = b * block + k;
      float v = load_elem(x, dtype, i);
      float t = v / X;
      float q = or_elem_round(t, fmt);
      if (y) store_elem(y, dtype, i, q * X);
      if (codes) codes[i] = or_elem_encode(q, fmt);
      set_mask(mask, i, fabsf(t) <= f.maxv);
    }
  }
  if (flags && nonfinite) *flags |= OR_FLAG_NONFINITE_INPUT;
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* FP8 formats, [QAT] module docs table + Fp8Format.                          */
/* ------------------------------------------------------------------------- */
static int fp8_mbits(int fmt) { return fmt == OR_E4M3 ? 3 : 2; }
static int fp8_bias(int fmt) { return fmt == OR_E4M3 ? 7 : 15; }
static float fp8_max(int fmt) { return fmt == OR_E4M3 ? 448.0f : 57344.0f; }

/* [QAT] fp8_quantize_magnitude: e = floor(log2 a) read from the exponent
 * field, ulp = 2^(max(e, emin) - mbits), round a/ulp to nearest even,
 * saturate at max-normal.  For a binary32 subnormal the field is 0, so
 * e = -127 and max(e, emin) = emin, the subnormal granularity. */
float or_fp8_magnitude(float a, int fmt) {
  if (a == 0.0f) return 0.0f;
  int emin = 1 - fp8_bias(fmt);
  int e = (int)((f2u(a) >> 23) & 0xFF) - 127;
  int se = (e > emin ? e : emin) - fp8_mbits(fmt);
  float step = ldexpf(1.0f, se);
  float ratio = a / step;
  float k = rintf(ratio);
  float mag = k * step;
  if (mag > fp8_max(fmt)) return fp8_max(fmt);
  return mag;
}

/* [QAT] fp8_quantize_magnitude with RoundingMode::Stochastic: the ratio a/ulp
 * (an exact power-of-two scaling) is rounded by or_sr_round with draw u, then
 * saturated as in the nearest-rounding rule. */
float or_fp8_magnitude_sr(float a, int fmt, float u) {
  if (a == 0.0f) return 0.0f;
  int emin = 1 - fp8_bias(fmt);
  int e = (int)((f2u(a) >> 23) & 0xFF) - 127;
  int se = (e > emin ? e : emin) - fp8_mbits(fmt);
  float step = ldexpf(1.0f, se);
  float ratio = a / step;
  float k = or_sr_round(ratio, u);
  float mag = k * step;
  if (mag > fp8_max(fmt)) return fp8_max(fmt);
  return mag;
}

float or_fp8_cast_sr(float t, int fmt, float u) {
  if (isnan(t)) return u2f(0x7FC00000u);
  if (isinf(t)) return copysignf(fp8_max(fmt), t);
  return copysignf(or_fp8_magnitude_sr(fabsf(t), fmt, u), t);
}

/* [QAT] fake_quant_fp8, one element: NaN -> NaN, +-Inf -> +-max, otherwise the
 * magnitude rule with the input's sign (signed zero kept). */
float or_fp8_cast(float t, int fmt) {
  if (isnan(t)) return u2f(0x7FC00000u);
  if (isinf(t)) return copysignf(fp8_max(fmt), t);
  return copysignf(or_fp8_magnitude(fabsf(t), fmt), t);
}

/* Encoding of an FP8 grid value (sign | exponent field | mantissa field).
 * reading: NaN is encoded 0x7F in both formats (E4M3 has the single NaN
 * pattern S.1111.111; positive sign chosen). */
uint8_t or_fp8_encode(float c, int fmt) {
  if (isnan(c)) return 0x7F;
  int mb = fp8_mbits(fmt), bias = fp8_bias(fmt);
  int emin = 1 - bias;
  uint8_t sign = signbit(c) ? 0x80 : 0x00;
  float a = fabsf(c);
  if (a == 0.0f) return sign;
  int ex;
  (void)frexpf(a, &ex);
  int e = ex - 1; /* a in [2^e, 2^(e+1)) */
  if (e < emin) {
    int man = (int)(a / ldexpf(1.0f, emin - mb));
    return (uint8_t)(sign | man);
  }
  int E = e + bias;
  int man = (int)((a / ldexpf(1.0f, e) - 1.0f) * ldexpf(1.0f, mb));
  return (uint8_t)(sign | (E << mb) | man);
}

/* ------------------------------------------------------------------------- */
/* Per-tensor amax-scaled FP8 fake quant.                                     */
/*   scale_given = 0: A = max |x| over finite x, s = A / fmt_max ([MAR]       */
/*                    per-channel E4M3 scale absmax/448), written to *scale;  */
/*   scale_given = 1: s = *scale (s = 1 is the unscaled cast of [QAT]).       */
/*   t = x / s, c = cast(t), y = c * s, code = encode(c),                     */
/*   mask = |x| <= fmt_max * s  (reading: the real interval the saturating    */
/*   cast maps without clamping; NaN -> 0).                                   */
/* reading: s == 0 -> every non-NaN element gets code 0 and y = +0 ([MAR]     */
/* zero scale gives byte 0); NaN stays NaN.  reading: NaN/Inf are excluded    */
/* from the amax and reported with OR_FLAG_NONFINITE_INPUT, not an error.     */
/* A given s that is negative, NaN or infinite: OR_FLAG_BAD_PARAMS and every  */
/* element gets code 0, y = +0, mask 0.                                       */
/* ------------------------------------------------------------------------- */
static int fq_fp8(const void* x, int dtype, int64_t n, int fmt, int scale_given, float* scale,
                  void* y, uint8_t* codes, uint32_t* mask, int32_t* flags, int stochastic,
                  uint64_t seed, uint64_t offset) {
  if (fmt != OR_E4M3 && fmt != OR_E5M2) return OR_ERR_UNSUPPORTED;
  if (n < 0) return OR_ERR_INVALID;
  if (n == 0) return OR_OK;
  if (mask) memset(mask, 0, (size_t)((n + 31) / 32) * 4);
  float fmax = fp8_max(fmt);
  float s;
  if (!scale_given) {
    float mn, mx, A;
    int64_t bad;
    or_unit_stats(x, dtype, 0, n, &mn, &mx, &A, &bad);
    if (bad && flags) *flags |= OR_FLAG_NONFINITE_INPUT;
    s = A / fmax;
    *scale = s;
  } else {
    s = *scale;
  }
  int badp = isnan(s) || isinf(s) || s < 0.0f;
  if (badp && flags) *flags |= OR_FLAG_BAD_PARAMS;
  float lim = fmax * s;
  for (int64_t i = 0; i < n; ++i) {
    float v = load_elem(x, dtype, i);
    float c, yv;
    int m;
    if (badp) {
      c = 0.0f; yv = 0.0f; m = 0;
    } else if (s == 0.0f) {
      c = isnan(v) ? v : 0.0f;
      yv = c;
      m = (fabsf(v) <= lim) ? 1 : 0;
    } else {
      float t = v / s;
      c = stochastic ? or_fp8_cast_sr(t, fmt, or_sr_uniform(seed, offset, i)) : or_fp8_cast(t, fmt);
      yv = c * s;
      m = (fabsf(v) <= lim) ? 1 : 0;
    }
    if (codes) codes[i] = badp ? 0 : or_fp8_encode(c, fmt);
    if (y) store_elem(y, dtype, i, yv);
    set_mask(mask, i, m);
  }
  return OR_OK;
}

int or_fake_quant_fp8(const void* x, int dtype, int64_t n, int fmt, int scale_given, float* scale,
                      void* y, uint8_t* codes, uint32_t* mask, int32_t* flags) {
  return fq_fp8(x, dtype, n, fmt, scale_given, scale, y, codes, mask, flags, 0, 0, 0);
}

/* The same with stochastic rounding of the FP8 magnitude (draw of element i:
 * or_sr_uniform(seed, offset, i)); the scale and the STE window are those of
 * the nearest-rounding path. */
int or_fake_quant_fp8_sr(const void* x, int dtype, int64_t n, int fmt, int scale_given,
                         float* scale, uint64_t seed, uint64_t offset, void* y, uint8_t* codes,
                         uint32_t* mask, int32_t* flags) {
  return fq_fp8(x, dtype, n, fmt, scale_given, scale, y, codes, mask, flags, 1, seed, offset);
}

/* ------------------------------------------------------------------------- */
/* [QAT] QatOptimizer::step, the element loop, in binary32:                   */
/*   m = beta1 m + (1 - beta1) g;  v = beta2 v + (1 - beta2) g g;             */
/*   m_hat = m / bc1;  v_hat = v / bc2;                                       */
/*   if wd != 0: w = w - lr wd w   (decoupled, AdamW);                        */
/*   w = w - lr m_hat / (sqrt(v_hat) + eps).                                  */
/* reading: every quantity is binary32 (master, moments, hyper-parameters),   */
/* each product / quotient / sum / square root rounded once, in the printed   */
/* order (left to right: (1 - beta2) g is rounded before the second g, lr wd  */
/* before w, lr m_hat before the division); 1 - beta is a binary32            */
/* subtraction; the bias corrections bc = 1 - beta^t of step t are given by   */
/* the caller (the module evaluates them in binary64).                        */
/* ------------------------------------------------------------------------- */
void or_adam_update(float* w, const float* g, float* m, float* v, int64_t n, float lr,
                    float beta1, float beta2, float eps, float wd, float bc1, float bc2) {
  const float omb1 = 1.0f - beta1, omb2 = 1.0f - beta2;
  const float lrwd = lr * wd;
  for (int64_t i = 0; i < n; ++i) {
    float gi = g[i];
    float mi = beta1 * m[i] + omb1 * gi;
    float vi = beta2 * v[i] + (omb2 * gi) * gi;
    m[i] = mi;
    v[i] = vi;
    float mh = mi / bc1;
    float vh = vi / bc2;
    float wi = w[i];
    if (wd != 0.0f) wi = wi - lrwd * wi;
    wi = wi - (lr * mh) / (sqrtf(vh) + eps);
    w[i] = wi;
  }
}

/* [QAT] QatOptimizer::step + requantize: the update above, then the view
 * re-derived from the new master: an integer target (bits 8 or 4) is
 * calibrated per tensor over the finite values (per_tensor_minmax: absmax
 * for symmetric, min/max for affine) and fake-quantized; an FP8 target is
 * the unscaled saturating cast (scale 1).  Rounding nearest or stochastic
 * (draws or_sr_uniform(seed, offset, i)).  *scale (and *zp) receive the view's
 * parameters; mask and codes as for the fake-quant calls. */
int or_qat_optimizer_step(float* w, const float* g, float* m, float* v, int64_t n, float lr,
                          float beta1, float beta2, float eps, float wd, float bc1, float bc2,
                          int bits, int scheme, int fmt, int stochastic, uint64_t seed,
                          uint64_t offset, float* view, void* codes, uint32_t* mask, float* scale,
                          int32_t* zp, int32_t* flags) {
  if (n < 0) return OR_ERR_INVALID;
  or_adam_update(w, g, m, v, n, lr, beta1, beta2, eps, wd, bc1, bc2);
  if (n == 0) return OR_OK;
  if (bits == 8 || bits == 4)
    return fq_int(w, OR_F32, 1, n, bits, scheme, OR_PER_TENSOR, 0, 0, scale, zp, view, codes, mask,
                  flags, 1, stochastic, seed, offset, 1.0f, 0);
  if (bits != 0) return OR_ERR_UNSUPPORTED;
  *scale = 1.0f;
  return fq_fp8(w, OR_F32, n, fmt, 1, scale, view, (uint8_t*)codes, mask, flags, stochastic, seed,
                offset);
}

/* ------------------------------------------------------------------------- */
/* [QAT] fake_quant_backward with the window precomputed as a bit mask:       */
/* dx = g where the bit is set, +0 elsewhere (a bit copy of g).               */
/* ------------------------------------------------------------------------- */
int or_ste_backward(const void* g, int dtype, int64_t n, const uint32_t* mask, void* dx) {
  if (n < 0) return OR_ERR_INVALID;
  for (int64_t i = 0; i < n; ++i) {
    int m = (mask[i >> 5] >> (i & 31)) & 1u;
    if (dtype == OR_BF16) ((uint16_t*)dx)[i] = m ? ((const uint16_t*)g)[i] : 0;
    else ((uint32_t*)dx)[i] = m ? ((const uint32_t*)g)[i] : 0u;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* 4-bit absmax blocks (level 1).  quantize_4bit itself is imported from a    */
/* sibling module that the sources do not show; what [DQ] fixes: 64-element  */
/* blocks, fp32 scales that are absmax / 7, 4-bit two's-complement codes two  */
/* per byte (even element high nibble).                                       */
/* reading: code = clamp(round_half_away(x / scale), -8, 7), the rounding the */
/* same file uses for level 2 (f32::round); an all-zero block has scale 0 and */
/* codes 0; a short tail block covers the remaining elements; NaN elements    */
/* are skipped by the absmax and get code 0.                                  */
/* ------------------------------------------------------------------------- */
#define OR_Q4_BLOCK 64
#define OR_Q4_SUPER 256

static int32_t q4_code(float v, float s) {
  if (s == 0.0f) return 0;
  float r = roundf(v / s);
  if (isnan(r)) return 0;
  if (r < -8.0f) r = -8.0f;
  if (r > 7.0f) r = 7.0f;
  return (int32_t)r;
}

int or_quant4_single(const float* x, int64_t n, uint8_t* data, float* scales) {
  if (n < 0) return OR_ERR_INVALID;
  int64_t nb = (n + OR_Q4_BLOCK - 1) / OR_Q4_BLOCK;
  memset(data, 0, (size_t)((n + 1) / 2));
  for (int64_t b = 0; b < nb; ++b) {
    int64_t s0 = b * OR_Q4_BLOCK, e0 = s0 + OR_Q4_BLOCK < n ? s0 + OR_Q4_BLOCK : n;
    float A = 0.0f;
    for (int64_t i = s0; i < e0; ++i) A = fmaxf(A, fabsf(x[i]));
    float s = A / 7.0f;
    scales[b] = s;
    for (int64_t i = s0; i < e0; ++i) set_code(data, 4, i, q4_code(x[i], s));
  }
  return OR_OK;
}

static int32_t nibble_value(const uint8_t* data, int64_t i) {
  uint8_t byte = data[i >> 1];
  uint8_t nib = (i & 1) == 0 ? (uint8_t)((byte >> 4) & 0x0F) : (uint8_t)(byte & 0x0F);
  return (nib & 0x08) ? (int32_t)nib - 16 : (int32_t)nib;
}

/* reading: a NaN result (0 * inf or a NaN scale) is written as the canonical
 * quiet NaN, as for every other floating-point output of this file. */
static float canon_nan(float v) { return isnan(v) ? u2f(0x7FC00000u) : v; }

int or_dequant4_single(const uint8_t* data, const float* scales, int64_t n, float* y) {
  for (int64_t i = 0; i < n; ++i)
    y[i] = canon_nan((float)nibble_value(data, i) * scales[i / OR_Q4_BLOCK]);
  return OR_OK;
}

/* [DQ] quantize_4bit_double: per run of 256 block scales, super = max scale
 * (at least 1e-8), q = clamp(round_half_away(scale / super * 255), 0, 255).
 * NaN (0/0 cannot occur; inf/inf can) converts to 0 like a float-to-u8 cast.
 * y_roundtrip (nullable) receives dequantize_4bit_double of the result. */
int or_quant4_double(const float* x, int64_t n, uint8_t* data, uint8_t* qscales, float* supers,
                     float* y_roundtrip) {
  if (n < 0) return OR_ERR_INVALID;
  if (n == 0) return OR_OK;
  int64_t nb = (n + OR_Q4_BLOCK - 1) / OR_Q4_BLOCK;
  int64_t ns = (nb + OR_Q4_SUPER - 1) / OR_Q4_SUPER;
  float* scales = (float*)malloc((size_t)nb * sizeof(float));
  if (!scales) return OR_ERR_INVALID;
  or_quant4_single(x, n, data, scales);
  for (int64_t sb = 0; sb < ns; ++sb) {
    int64_t s0 = sb * OR_Q4_SUPER, e0 = s0 + OR_Q4_SUPER < nb ? s0 + OR_Q4_SUPER : nb;
    float mx = scales[s0];
    for (int64_t b = s0 + 1; b < e0; ++b)
      if (scales[b] > mx) mx = scales[b];
    if (!(mx >= 1e-8f)) mx = 1e-8f;
    supers[sb] = mx;
    for (int64_t b = s0; b < e0; ++b) {
      float normalized = scales[b] / mx;
      float q = roundf(normalized * 255.0f);
      if (isnan(q)) q = 0.0f;
      if (q < 0.0f) q = 0.0f;
      if (q > 255.0f) q = 255.0f;
      qscales[b] = (uint8_t)q;
    }
  }
  free(scales);
  if (y_roundtrip) or_dequant4_double(data, qscales, supers, n, y_roundtrip);
  return OR_OK;
}

/* [DQ] reconstruct_scales: scale = f32(q) / 255 * super (two roundings). */
float or_reconstruct_scale(uint8_t q, float super) { return (float)q / 255.0f * super; }

/* [DQ] dequantize_4bit_double: y = f32(sign-extended nibble) * scale. */
int or_dequant4_double(const uint8_t* data, const uint8_t* qscales, const float* supers, int64_t n,
                       float* y) {
  if (n < 0) return OR_ERR_INVALID;
  int64_t nb = (n + OR_Q4_BLOCK - 1) / OR_Q4_BLOCK;
  for (int64_t b = 0; b < nb; ++b) {
    float s = or_reconstruct_scale(qscales[b], supers[b / OR_Q4_SUPER]);
    int64_t s0 = b * OR_Q4_BLOCK, e0 = s0 + OR_Q4_BLOCK < n ? s0 + OR_Q4_BLOCK : n;
    for (int64_t i = s0; i < e0; ++i) y[i] = canon_nan((float)nibble_value(data, i) * s);
  }
  return OR_OK;
}

/* [DQ] DoubleQuantized4Bit::memory_bytes for n values: packed data
 * ceil(n/2) + one byte per block + four bytes per super-block. */
int64_t or_q4d_memory_bytes(int64_t n) {
  int64_t nb = (n + OR_Q4_BLOCK - 1) / OR_Q4_BLOCK;
  int64_t ns = (nb + OR_Q4_SUPER - 1) / OR_Q4_SUPER;
  return (n + 1) / 2 + nb + 4 * ns;
}

/* ========================================================================= */
/* O64: the [QAT] formulas in binary64 on the same inputs (tolerance only).   */
/* ========================================================================= */

static double rne64(double v) { return nearbyint(v); }

/* int fake quant in f64, documented form.  Writes y64 (double per element),
 * scale64 / zp64 per unit; dead units (as in O32) get y = 0. */
int or64_fake_quant_int(const void* x, int dtype, int64_t rows, int64_t cols, int bits, int scheme,
                        int gran, int64_t group, double* y64, double* scale64, int32_t* zp64) {
  int32_t qmin, qmax;
  int st = or_q_range(bits, scheme, &qmin, &qmax);
  if (st) return st;
  int64_t n = rows * cols, L, stride = 1;
  if (gran == OR_PER_TENSOR) L = n;
  else if (gran == OR_PER_ROW) L = cols;
  else if (gran == OR_PER_COLUMN) {
    L = rows;
    stride = cols;
  } else {
    if (group <= 0 || cols % group) return OR_ERR_INVALID;
    L = group;
  }
  if (n == 0) return OR_OK;
  const int64_t units = gran == OR_PER_COLUMN ? cols : n / L;
  for (int64_t u = 0; u < units; ++u) {
    int64_t off = gran == OR_PER_COLUMN ? u : u * L;
    double mn = INFINITY, mx = -INFINITY, A = 0.0;
    int bad = 0;
    for (int64_t k = 0; k < L; ++k) {
      double v = load_elem(x, dtype, off + k * stride);
      if (!isfinite(v)) { bad = 1; continue; }
      if (v < mn) mn = v;
      if (v > mx) mx = v;
      if (fabs(v) > A) A = fabs(v);
    }
    double s = 0.0;
    int32_t z = 0;
    int dead = bad;
    if (scheme == OR_SYM) {
      s = A / (double)qmax;
      if (!(s > 0.0)) dead = 1;
    } else {
      double rmin = mn < 0.0 ? mn : 0.0, rmax = mx > 0.0 ? mx : 0.0;
      s = (rmax - rmin) / (double)(qmax - qmin);
      if (!(s > 0.0) || isinf(s)) dead = 1;
      else {
        double zz = rne64((double)qmin - rmin / s);
        if (zz < qmin) zz = qmin;
        if (zz > qmax) zz = qmax;
        z = (int32_t)zz;
      }
    }
    scale64[u] = s;
    zp64[u] = z;
    for (int64_t k0 = 0; k0 < L; ++k0) {
      const int64_t i = off + k0 * stride;
      if (dead) { y64[i] = 0.0; continue; }
      double v = load_elem(x, dtype, i);
      double k = rne64(v / s);
      if (k < (double)(qmin - z)) k = qmin - z;
      if (k > (double)(qmax - z)) k = qmax - z;
      y64[i] = k * s;
    }
  }
  return OR_OK;
}

/* FP8 fake quant in f64 ([QAT] fp8_quantize_magnitude on f64 bits). */
static double fp8_mag64(double a, int fmt) {
  if (a == 0.0) return 0.0;
  int emin = 1 - fp8_bias(fmt);
  uint64_t u;
  memcpy(&u, &a, 8);
  int e = (int)((u >> 52) & 0x7FF) - 1023;
  int se = (e > emin ? e : emin) - fp8_mbits(fmt);
  double step = ldexp(1.0, se);
  double mag = rne64(a / step) * step;
  return mag > fp8_max(fmt) ? (double)fp8_max(fmt) : mag;
}

int or64_fake_quant_fp8(const void* x, int dtype, int64_t n, int fmt, double* y64, double* scale64) {
  double A = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double v = load_elem(x, dtype, i);
    if (isfinite(v) && fabs(v) > A) A = fabs(v);
  }
  double s = A / (double)fp8_max(fmt);
  *scale64 = s;
  for (int64_t i = 0; i < n; ++i) {
    double v = load_elem(x, dtype, i);
    double c;
    if (isnan(v)) c = NAN;
    else if (s == 0.0) c = 0.0;
    else {
      double t = v / s;
      if (isinf(t)) c = copysign((double)fp8_max(fmt), t);
      else c = copysign(fp8_mag64(fabs(t), fmt), t);
    }
    y64[i] = (s == 0.0 || isnan(c)) ? c : c * s;
  }
  return OR_OK;
}
