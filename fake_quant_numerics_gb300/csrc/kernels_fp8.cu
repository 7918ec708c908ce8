// kernels_fp8.cu -- per-tensor amax-scaled FP8 fake quant.
//
// optirs-gpu quantization.rs, module docs "fp8 quantization (E4M3 / E5M2)",
// fp8_quantize_magnitude and fake_quant_fp8: the value is rounded to the
// nearest FP8 grid point (ties to even), magnitudes above the format maximum
// and infinities saturate to +-max, NaN stays NaN, signed zero is kept.  The
// per-tensor scale follows ferrum-kernels marlin_repack.rs
// (prepare_f16_weight_for_fp8_marlin: scale = absmax / 448; a zero scale
// encodes as byte 0).
//
// The cast itself is the hardware saturating conversion
// cvt.rn.satfinite.{e4m3x2,e5m2x2}.f32 (round to nearest even, +-inf and
// overflow -> +-max, NaN -> NaN), decoded back with cvt.rn.f16x2.{e4m3x2,
// e5m2x2} (every FP8 value is exact in fp16).  The library's tests compare
// this against the rule above over every fp16, every bf16 and sampled fp32
// bit patterns, ties included.  NaN handling is made explicit (code 0x7F,
// canonical quiet NaN output) instead of relying on the conversion's NaN
// payload.
#include <cuda_fp16.h>

#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

template <int FMT>
__device__ __forceinline__ uint32_t fp8x2_encode(float lo, float hi) {
  uint16_t r;
  if (FMT == QAT_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int FMT>
__device__ __forceinline__ void fp8x2_decode(uint32_t c2, float& lo, float& hi) {
  uint32_t h2;
  uint16_t c = (uint16_t)c2;
  if (FMT == QAT_E4M3)
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  else
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(c));
  lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
  hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

// Exact cast without a per-element division.  With rcp = RN(1/s),
// rlo = RN(rcp (1 - 2^-21)) and rhi = RN(rcp (1 + 2^-21)), the products
// lo = RN(x rlo) and hi = RN(x rhi) satisfy |lo| < |RN(x/s)| < |hi| (each of
// rcp, rlo / rhi and the product carries at most 2^-24 relative error, the
// margin is 8 * 2^-24) with the sign of x, whenever s is in [2^-80, 2^100]
// (below the normal range all three are far under half the smallest FP8
// subnormal and cast to the same signed zero; above FP8's range all saturate).
// The saturating FP8 rounding is monotone in magnitude, so when lo and hi
// cast to the same code, that is the code of RN(x/s); otherwise the pair is
// recomputed from the correctly rounded quotient.
struct Fp8Params {
  float s;          // scale
  float lim;        // fmt_max * s: the STE window |x| <= lim
  float rlo, rhi;   // bracketing reciprocals (fast == 1)
  float rcp, ns;    // RN(1/s) and -s for the exact quotient (stochastic rounding, fast == 1)
  uint32_t limh2;   // (bf16 magnitude bits of the largest bf16 <= lim) | 0x8000, in both halves
  int mode;         // 0 normal, 1 zero scale, 2 invalid given scale
  int fast;
};

__device__ __forceinline__ void fp8_params_finish(Fp8Params& p) {
  p.fast = p.mode == 0 && quot_scale_ok(p.s);
  const float rcp = p.fast ? __frcp_rn(p.s) : 1.0f;
  p.rlo = __fmul_rn(rcp, 1.0f - 0x1p-21f);
  p.rhi = __fmul_rn(rcp, 1.0f + 0x1p-21f);
  p.rcp = rcp;
  p.ns = -p.s;
  // lim >= 0 is finite when fast; truncating its bits to 16 rounds toward 0
  p.limh2 = ((__float_as_uint(p.lim) >> 16) | 0x8000u) * 0x00010001u;
}

constexpr uint32_t kNaN32 = 0x7fc00000u;
constexpr uint32_t kNaN16 = 0x7fc0u;

// One bf16 vector (16 elements, 8 bf16x2 words) on the bracketing path,
// with the element tests done on the packed words: a = w & 0x7fff7fff holds
// both magnitudes; a half above 0x7f80 is a NaN (adding 0x7f carries into
// its top bit), and |x| <= lim is (0x8000 | L) - a >= 0x8000 per half, L the
// magnitude bits of the largest bf16 not above lim (no borrow crosses the
// halves since every a <= 0x7fff).  Returns false, leaving the vector to the
// element-wise path, when a NaN is present or a bracket splits.
template <int FMT, bool CODES>
__device__ __forceinline__ bool fp8_vec_bf16_fast(const V32& v, const Fp8Params& p, V32& out,
                                                  CodeVec<8, 16>& cv, uint32_t& mb) {
  uint32_t bad = 0u, macc = 0u, pend = 0u;
#pragma unroll
  for (int e = 14; e >= 0; e -= 2) {
    const uint32_t w = v.w[e >> 1];
    const uint32_t a = w & 0x7fff7fffu;
    bad |= (a + 0x007f007fu) & 0x80008000u;
    // window bits of elements e and e + 1 land on bits e and 16 + e
    macc |= ((p.limh2 - a) & 0x80008000u) >> (15 - e);
    const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xffff0000u);
    float l0, l1, h0, h1;
    mul2(x0, x1, p.rlo, p.rlo, l0, l1);
    mul2(x0, x1, p.rhi, p.rhi, h0, h1);
    const uint32_t c2 = fp8x2_encode<FMT>(l0, l1);
    bad |= c2 ^ fp8x2_encode<FMT>(h0, h1);
    float d0, d1, y0, y1;
    fp8x2_decode<FMT>(c2, d0, d1);
    mul2(d0, d1, p.s, p.s, y0, y1);
    out.w[e >> 1] = pack_bf16x2(y0, y1);
    if (CODES) {
      if (e & 2)
        pend = c2;
      else
        cv.w[e >> 2] = __byte_perm(c2, pend, 0x5410);  // codes e .. e + 3
    }
  }
  mb = (macc & 0x5555u) | ((macc >> 15) & 0xaaaau);
  return bad == 0u;
}

// fp8_quantize_magnitude with stochastic rounding (RoundingMode::Stochastic)
// for the quotient t = RN(x/s) of an element x (s > 0): with e = floor(log2
// |t|), ulp = 2^(max(e, emin) - mbits); |t| / ulp (an exact power-of-two
// scaling) is rounded by the draw u (up when u < its fraction), times ulp,
// saturated at the format maximum, with the sign of t.  Here 2^max(e, emin)
// is the larger of the exponent fields of |t| and of 2^emin (a zero or
// binary32 subnormal t has field 0), ulp and 1 / ulp (exponent field 254 +
// mbits - that field) are exact, and the sign is taken from x, which t
// shares, so a quotient whose sign or value the residual steps lost needs no
// repair: t = +0 for x = -0 gives -0 again, and a NaN quotient of x = +-inf
// (or of an x whose quotient overflows) gives fminf(NaN, max) = max, the
// rule's value for an infinite t (an element with x NaN is replaced by the
// caller).  u = (w >> 9) 2^-23 as (1 + u) - 1, 1 + u having the bits
// hi(w 2^23) + 0x3f800000 (one multiply-add).
template <int FMT>
__device__ __forceinline__ float fp8_sr_value_x(float t, float x, uint32_t w) {
  constexpr uint32_t MB = FMT == QAT_E4M3 ? 3u : 2u;
  constexpr uint32_t kEminField = (uint32_t)((FMT == QAT_E4M3 ? -6 : -14) + 127) << 23;
  constexpr float kMaxF = FMT == QAT_E4M3 ? 448.0f : 57344.0f;
  constexpr float kStepOfExp = FMT == QAT_E4M3 ? 0x1p-3f : 0x1p-2f;  // 2^-mbits
  uint32_t ub;
  asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(ub) : "r"(w), "r"(0x00800000u), "r"(0x3f800000u));
  const float u = __fsub_rn(__uint_as_float(ub), 1.0f);
  const float a = fabsf(t);
  const uint32_t eb = max(__float_as_uint(a) & 0x7f800000u, kEminField);
  const float inv = __uint_as_float(((254u + MB) << 23) - eb);
  const float step = __fmul_rn(__uint_as_float(eb), kStepOfExp);
  // sr_round(r, u) as floor(r) + ceil(frac - u): frac - u is exact in sign
  // (u a multiple of 2^-23 in [0, 1), frac in [0, 1)) and in (-1, 1), so its
  // ceiling is 1 when u < frac and +-0 otherwise.  An infinite or NaN r gives
  // a NaN k here (r itself in sr_round), and fminf turns either into max.
  const float r = __fmul_rn(a, inv);
  const float lower = floorf(r);
  const float k = __fadd_rn(lower, ceilf(__fsub_rn(__fsub_rn(r, lower), u)));
  return copysignf(fminf(__fmul_rn(k, step), kMaxF), x);
}

// One vector with stochastic rounding for a usable scale (mode 0): the
// quotient t = RN(x/s) (exact residual-step quotient for a safe scale, the
// division otherwise), fp8_sr_value_x, y = g s and the code of the grid value
// g; NaN elements get the canonical NaN and code 0x7F.  For bf16 the window
// and the NaN test run on the packed magnitudes a = w & 0x7fff7fff as in
// fp8_vec_bf16_fast (a half above 0x7f80 is a NaN: adding 0x7f carries into
// its top bit).
template <typename T, int FMT, bool CODES, bool FULL>
__device__ __forceinline__ void fp8_vec_sr_mode0(const V32& v, const Fp8Params& p, const SrCtx& sr,
                                                 int64_t base, int cnt, V32& out,
                                                 CodeVec<8, T::VEC>& cv, uint32_t& mb) {
  constexpr int VEC = T::VEC;
  cv.clear();
  uint32_t macc = 0u, amax2 = 0u;
  mb = 0u;
#pragma unroll
  for (int g = VEC / 4 - 1; g >= 0; --g) {
    const uint4 wd = philox4x32_10(sr.offset + (uint64_t)(base / 4 + g), sr.rk);
    const uint32_t w4[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
    for (int h = 1; h >= 0; --h) {
      const int e = 4 * g + 2 * h;
      const float x0 = elem<T>(v, e), x1 = elem<T>(v, e + 1);
      float t0, t1;
      if (p.fast) {
        quotient_rn2(x0, x1, p.rcp, p.ns, t0, t1);
      } else {
        t0 = __fdiv_rn(x0, p.s);
        t1 = __fdiv_rn(x1, p.s);
      }
      const float g0 = fp8_sr_value_x<FMT>(t0, x0, w4[2 * h]);
      const float g1 = fp8_sr_value_x<FMT>(t1, x1, w4[2 * h + 1]);
      float y0, y1;
      mul2(g0, g1, p.s, p.s, y0, y1);
      bool n0 = false, n1 = false;
      if constexpr (T::BYTES == 4) {
        n0 = isnan(x0);
        n1 = isnan(x1);
        mb |= (uint32_t)(fabsf(x0) <= p.lim) << e;
        mb |= (uint32_t)(fabsf(x1) <= p.lim) << (e + 1);
        out.w[e] = n0 ? kNaN32 : __float_as_uint(y0);
        out.w[e + 1] = n1 ? kNaN32 : __float_as_uint(y1);
      } else {
        const uint32_t am = v.w[e >> 1] & 0x7fff7fffu;
        // window bits of elements e and e + 1 land on bits e and 16 + e
        macc |= ((p.limh2 - am) & 0x80008000u) >> (15 - e);
        out.w[e >> 1] = pack_bf16x2(y0, y1);
        if (CODES) {
          const uint32_t nan = (am + 0x007f007fu) & 0x80008000u;
          const uint32_t keep = (nan >> 15) * 0xffffu;  // 0xffff in each NaN half
          out.w[e >> 1] = (out.w[e >> 1] & ~keep) | (((kNaN16 << 16) | kNaN16) & keep);
          n0 = (nan & 0x8000u) != 0u;
          n1 = (nan >> 31) != 0u;
        } else {
          amax2 = __vmaxu2(amax2, am);
        }
      }
      if (CODES) {
        const uint32_t c2 = fp8x2_encode<FMT>(g0, g1);
        const uint32_t c0 = n0 ? 0x7fu : (c2 & 0xffu), c1 = n1 ? 0x7fu : ((c2 >> 8) & 0xffu);
        cv.set2(e, (FULL || e < cnt) ? (int)(int8_t)c0 : 0,
                (FULL || e + 1 < cnt) ? (int)(int8_t)c1 : 0);
      }
    }
  }
  if constexpr (T::BYTES == 2) {
    mb = (macc & 0x5555u) | ((macc >> 15) & 0xaaaau);
    // without codes, the NaN elements (magnitude bits above 0x7f80) are
    // patched only in a vector that holds one
    if (!CODES && max(amax2 & 0xffffu, amax2 >> 16) > 0x7f80u) {
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) {
        const uint32_t nan = ((v.w[i] & 0x7fff7fffu) + 0x007f007fu) & 0x80008000u;
        const uint32_t keep = (nan >> 15) * 0xffffu;
        out.w[i] = (out.w[i] & ~keep) | (((kNaN16 << 16) | kNaN16) & keep);
      }
    }
  }
}

// One vector with stochastic rounding: fp8_vec_sr_mode0 for a usable scale;
// for a zero or invalid scale the outputs of the nearest-rounding path (no
// draw changes them).
template <typename T, int FMT, bool CODES, bool FULL>
__device__ __forceinline__ void fp8_vec_sr(const V32& v, const Fp8Params& p, const SrCtx& sr,
                                           int64_t base, int cnt, V32& out,
                                           CodeVec<8, T::VEC>& cv, uint32_t& mb) {
  constexpr int VEC = T::VEC;
  if (p.mode == 0) {
    fp8_vec_sr_mode0<T, FMT, CODES, FULL>(v, p, sr, base, cnt, out, cv, mb);
    return;
  }
  // a zero scale (mode 1: codes 0, y +0, NaN kept with code 0x7F, the
  // window |x| <= 0) or an invalid given scale (mode 2: codes 0, y +0,
  // mask 0): no quotients and no draws
  cv.clear();
  mb = 0u;
#pragma unroll
  for (int e = VEC - 2; e >= 0; e -= 2) {
    const float x0 = elem<T>(v, e), x1 = elem<T>(v, e + 1);
    const bool n0 = p.mode != 2 && isnan(x0), n1 = p.mode != 2 && isnan(x1);
    if (p.mode != 2) {
      mb |= (uint32_t)(fabsf(x0) <= p.lim) << e;
      mb |= (uint32_t)(fabsf(x1) <= p.lim) << (e + 1);
    }
    if (CODES) {
      cv.set2(e, (FULL || e < cnt) && n0 ? 0x7f : 0, (FULL || e + 1 < cnt) && n1 ? 0x7f : 0);
    }
    if (T::BYTES == 4) {
      out.w[e] = n0 ? kNaN32 : 0u;
      out.w[e + 1] = n1 ? kNaN32 : 0u;
    } else {
      out.w[e >> 1] = (n0 ? kNaN16 : 0u) | (n1 ? (kNaN16 << 16) : 0u);
    }
  }
}

template <typename T, int FMT, bool CODES, bool FULL, bool SR>
__device__ __forceinline__ void fp8_tile(const void* __restrict__ x, int64_t n, int64_t tile,
                                         V32 (&v)[kTile / (32 * T::VEC)], bool have, int64_t next,
                                         const Fp8Params& p, const SrCtx& sr,
                                         void* __restrict__ y, uint8_t* __restrict__ codes,
                                         uint32_t* __restrict__ mask, int lane) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC);
  const int64_t tb = tile * kTile;
  int cnt[SLOTS];
  tile_load<T, FULL>(x, n, tile, v, cnt, have, lane);
  uint32_t mw[SLOTS];
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) {
    const int64_t base = tb + (int64_t)(j * 32 + lane) * VEC;
    V32 out;
    CodeVec<8, VEC> cv;
    uint32_t mb = 0u;
    bool done = false;
    if constexpr (SR) {
      fp8_vec_sr<T, FMT, CODES, FULL>(v[j], p, sr, base, cnt[j], out, cv, mb);
      done = true;
    } else if constexpr (T::BYTES == 2) {
      if (p.fast) done = fp8_vec_bf16_fast<FMT, CODES>(v[j], p, out, cv, mb);
    }
    if (!done) {
      cv.clear();
      mb = 0u;
  #pragma unroll
      for (int e = VEC - 2; e >= 0; e -= 2) {
        const float x0 = elem<T>(v[j], e), x1 = elem<T>(v[j], e + 1);
        const bool n0 = isnan(x0), n1 = isnan(x1);
        uint32_t c0, c1;
        float y0, y1;
        if (p.mode == 0) {
          uint32_t c2;
          if (p.fast) {
            float l0, l1, h0, h1;
            mul2(x0, x1, p.rlo, p.rlo, l0, l1);
            mul2(x0, x1, p.rhi, p.rhi, h0, h1);
            c2 = fp8x2_encode<FMT>(l0, l1);
            const uint32_t h2 = fp8x2_encode<FMT>(h0, h1);
            if (c2 != h2) c2 = fp8x2_encode<FMT>(__fdiv_rn(x0, p.s), __fdiv_rn(x1, p.s));
          } else {
            c2 = fp8x2_encode<FMT>(__fdiv_rn(x0, p.s), __fdiv_rn(x1, p.s));
          }
          float d0, d1;
          fp8x2_decode<FMT>(c2, d0, d1);
          c0 = c2 & 0xffu;
          c1 = (c2 >> 8) & 0xffu;
          mul2(d0, d1, p.s, p.s, y0, y1);
        } else {
          c0 = c1 = 0u;
          y0 = y1 = 0.0f;
        }
        if (p.mode != 2) {
          if (n0) c0 = 0x7fu;
          if (n1) c1 = 0x7fu;
          mb |= (uint32_t)(fabsf(x0) <= p.lim) << e;
          mb |= (uint32_t)(fabsf(x1) <= p.lim) << (e + 1);
        }
        if (CODES) {
          cv.set2(e, (FULL || e < cnt[j]) ? (int)(int8_t)c0 : 0,
                  (FULL || e + 1 < cnt[j]) ? (int)(int8_t)c1 : 0);
        }
        if (T::BYTES == 4) {
          out.w[e] = (p.mode != 2 && n0) ? kNaN32 : __float_as_uint(y0);
          out.w[e + 1] = (p.mode != 2 && n1) ? kNaN32 : __float_as_uint(y1);
        } else {
          uint32_t w = pack_bf16x2(y0, y1);
          if (p.mode != 2) {
            if (n0) w = (w & 0xffff0000u) | kNaN16;
            if (n1) w = (w & 0x0000ffffu) | (kNaN16 << 16);
          }
          out.w[e >> 1] = w;
        }
      }
    }
    slot_prefetch<T>(x, next, j, v[j], lane);
    if (!FULL) mb &= (cnt[j] >= 32) ? 0xffffffffu : ((1u << cnt[j]) - 1u);
    if (cnt[j] > 0) {
      store_vec<T>(y, base, out, cnt[j]);
      if (CODES) cv.store(codes, base, cnt[j]);
    }
    mw[j] = mask_word_of_slot<VEC>(mb, lane);
  }
  if (mask) {
    uint32_t w = gather_tile_word<VEC, SLOTS>(mw, lane);
    int64_t wi = tile * 32 + lane;
    if (FULL || wi < (n + 31) / 32) mask[wi] = w;
  }
}

template <typename T, int FMT, bool GIVEN, bool CODES, bool SR>
__global__ void __launch_bounds__(256) k_fp8_tensor(const void* __restrict__ x, int64_t n,
                                                    const uint4* __restrict__ part, int nparts,
                                                    float* scale, SrCtx sr, void* y,
                                                    uint8_t* codes, uint32_t* mask,
                                                    int32_t* flags) {
  constexpr float kMax = FMT == QAT_E4M3 ? 448.0f : 57344.0f;
  __shared__ __align__(16) uint32_t red[4 * 8];
  __shared__ Fp8Params sp;
  if (GIVEN) {
    pdl_wait();  // after the optimizer's update, x and the scale are its outputs
    if (threadIdx.x == 0) {
      float s = scale[0];
      sp.s = s;
      sp.mode = (isnan(s) || isinf(s) || s < 0.0f) ? 2 : (s == 0.0f ? 1 : 0);
      sp.lim = __fmul_rn(kMax, s);
      fp8_params_finish(sp);
      if (blockIdx.x == 0) flag_or(flags, sp.mode == 2 ? QAT_FLAG_BAD_PARAMS : 0);
    }
  } else {
    // launched early (after the statistics pass): request the warp's first
    // tile into L2, then wait for the partials
    {
      const int64_t ntiles = (n + kTile - 1) / kTile;
      const int64_t t0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
      if (t0 < ntiles) prefetch_tile_l2<T>(x, n, ntiles - 1 - t0, threadIdx.x & 31);
    }
    pdl_wait();
    Stats st = reduce_partials<kMMNone>(part, nparts, red);
    if (threadIdx.x == 0) {
      float s = __fdiv_rn(st.absmax_f(), kMax);
      sp.s = s;
      sp.mode = s == 0.0f ? 1 : 0;
      sp.lim = __fmul_rn(kMax, s);
      fp8_params_finish(sp);
      if (blockIdx.x == 0) {
        scale[0] = s;
        flag_or(flags, st.has_nonfinite() ? QAT_FLAG_NONFINITE_INPUT : 0);
      }
    }
  }
  __syncthreads();
  const Fp8Params p = sp;
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t nfull = n / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  V32 v[kTile / (32 * T::VEC)];
  bool have = false;
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < ntiles;
       t += wstride) {
    const int64_t tile = GIVEN ? t : ntiles - 1 - t;
    const int64_t nt = t + wstride;
    const int64_t ntile = GIVEN ? nt : ntiles - 1 - nt;
    // no rolling prefetch here: the extra live vectors cost more occupancy
    // than the overlap gains for this arithmetic-heavy map
    const int64_t next = -1;
    (void)ntile;
    if (tile < nfull)
      fp8_tile<T, FMT, CODES, true, SR>(x, n, tile, v, have, next, p, sr, y, codes, mask, lane);
    else
      fp8_tile<T, FMT, CODES, false, SR>(x, n, tile, v, have, next, p, sr, y, codes, mask, lane);
    have = next >= 0;
  }
}

template <typename T, int FMT>
static void fp8_t(bool given, const void* x, int64_t n, const void* ws, int nparts, float* scale,
                  const SrCtx& sr, void* y, uint8_t* codes, uint32_t* mask, int32_t* flags,
                  cudaStream_t s, bool pdl) {
  const int64_t ntiles = (n + kTile - 1) / kTile;
  int64_t g = (ntiles + 7) / 8;
  int64_t cap = (int64_t)device_info().sms * 8;
  int grid = (int)(g > cap ? cap : (g < 1 ? 1 : g));
  const uint4* part = static_cast<const uint4*>(ws);
#define QAT_K(G, C)                                                                             \
  launch_kernel(k_fp8_tensor<T, FMT, G, C, QAT_SR>, dim3(grid), dim3(256), 0, s, pdl, x, n, part, \
                nparts, scale, sr, y, codes, mask, flags)
  if (given) {
    if (codes) QAT_K(true, true); else QAT_K(true, false);
  } else {
    if (codes) QAT_K(false, true); else QAT_K(false, false);
  }
#undef QAT_K
}

QAT_DECL_FP8_TENSOR(QAT_SR_NAME(launch_fp8_tensor)) {
#define QAT_F8(T, F) fp8_t<T, F>(given, x, n, ws, nparts, scale, sr, y, codes, mask, flags, s, pdl)
  if (dt == QAT_F32) {
    if (fmt == QAT_E4M3) QAT_F8(F32, QAT_E4M3);
    else QAT_F8(F32, QAT_E5M2);
  } else {
    if (fmt == QAT_E4M3) QAT_F8(BF16, QAT_E4M3);
    else QAT_F8(BF16, QAT_E5M2);
  }
#undef QAT_F8
  count_launch(1);
  return launch_status();
}

}  // namespace qat
