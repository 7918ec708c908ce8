// qat_sr.h -- the stochastic-rounding call context shared by the host
// launchers and the kernels (internal; not part of the C ABI).
#pragma once

#include <cstdint>

namespace qat {

// Philox-4x32-10 key and counter base of one call: element i draws word
// i % 4 of the block with counter offset + i / 4.  rk holds the key of every
// round (the Weyl schedule k + r * (0x9E3779B9, 0xBB67AE85), r = 0..9), set
// once per call on the host by sr_set_round_keys, so the kernels read them
// from their parameters instead of stepping the schedule per thread.
constexpr int kPhiloxRounds = 10;
struct SrCtx {
  uint32_t k0, k1;  // key: low and high word of the seed
  uint64_t offset;  // counter base
  uint32_t rk[2 * kPhiloxRounds];
};
inline void sr_set_round_keys(SrCtx& c) {
  uint32_t a = c.k0, b = c.k1;
  for (int r = 0; r < kPhiloxRounds; ++r) {
    c.rk[2 * r] = a;
    c.rk[2 * r + 1] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
}

// Calibration options of a call (the module's calibration is {1, 0, 0}):
// the observed absmax (symmetric) or min and max (affine) times `clip` (one
// binary32 product, clip in (0, 1]); with `fp16` the scale is rounded to
// binary16 and that value is the unit's scale; `clamp` makes the symmetric
// fast path clamp its codes, which every option that can leave values beyond
// the calibrated range needs (a clip below 1, a rounded scale, percentile
// bounds).
struct CalOpts {
  float clip;
  int fp16;
  int clamp;
};
constexpr CalOpts kCalPlain{1.0f, 0, 0};

}  // namespace qat

// Each kernel source is compiled twice: with QAT_SR 0 (nearest rounding, the
// statistics kernels and every launcher) and with QAT_SR 1 (only the kernels
// whose rounding is stochastic, behind launchers named *_sr).
#ifndef QAT_SR
#define QAT_SR 0
#endif
#if QAT_SR
#define QAT_SR_NAME(f) f##_sr
#else
#define QAT_SR_NAME(f) f
#endif
