// kernels_block.cu -- block-scaled floating-point fake quant (MX and NVFP4).
//
// cs349e 05_quantization_basics.py, demo 4, block_scaled: one scale per block
// of `block` consecutive elements (32 for the OCP MX formats, 16 for NVFP4),
// from the block's absmax:
//   E8M0 -- X = 2^(floor(log2 amax) - emax_elem) (amax = 0: 2^-emax_elem);
//   E4M3 -- g = max|x| / (max_elem * 448) over the tensor,
//           X = E4M3_round_sat(amax / max_elem / g) * g;
//   FP32 -- X = amax / max_elem;
//   X <= 0 or NaN -> 1;
// then y = x / X rounded to nearest even on the element grid with saturation,
// times X.  Elements: E4M3, E5M2 (FP8), E2M3, E3M2 (FP6), E2M1 (FP4), whose
// saturating round-to-nearest-even casts are single conversions
// (cvt.rn.satfinite.{e4m3x2,e5m2x2,e2m3x2,e3m2x2,e2m1x2}.f32), decoded back
// with cvt.rn.f16x2.* (every element value is exact in fp16).  binary32
// arithmetic, one rounding per operation in the printed order; amax over
// finite values; a NaN element gives y NaN (code 0x7F for FP8 elements, 0 for
// FP6 / FP4); the E8M0 exponent is held to [-127, 127]; the STE mask bit is
// |x / X| <= max_elem.
//
// A lane owns one 32-byte vector (8 fp32 or 16 bf16 elements), so a block is
// 1 to 4 lanes and its absmax a shuffle reduction over them; a warp takes a
// 1024-element tile and writes its 32 mask words at once.
#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

template <int FMT>
struct ElemFmt;
template <>
struct ElemFmt<QAT_ELEM_E4M3> {
  static constexpr float kMax = 448.0f;
  static constexpr int kEmax = 8, kBits = 8;
};
template <>
struct ElemFmt<QAT_ELEM_E5M2> {
  static constexpr float kMax = 57344.0f;
  static constexpr int kEmax = 15, kBits = 8;
};
template <>
struct ElemFmt<QAT_ELEM_E2M3> {
  static constexpr float kMax = 7.5f;
  static constexpr int kEmax = 2, kBits = 6;
};
template <>
struct ElemFmt<QAT_ELEM_E3M2> {
  static constexpr float kMax = 28.0f;
  static constexpr int kEmax = 4, kBits = 6;
};
template <>
struct ElemFmt<QAT_ELEM_E2M1> {
  static constexpr float kMax = 6.0f;
  static constexpr int kEmax = 2, kBits = 4;
};

// Codes of elements (a, b) = (e, e + 1): FP8 / FP6 as a 16-bit word with a's
// code in the low byte; FP4 as a byte with a's code in the high nibble.
// NaN must not reach the FP6 / FP4 conversions (the caller replaces it).
template <int FMT>
__device__ __forceinline__ uint32_t elem_enc2(float a, float b) {
  uint32_t r;
  if (FMT == QAT_ELEM_E2M1) {
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
        : "=r"(r) : "f"(a), "f"(b));
    return r;
  }
  uint16_t h;
  if (FMT == QAT_ELEM_E4M3) asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(b), "f"(a));
  if (FMT == QAT_ELEM_E5M2) asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(h) : "f"(b), "f"(a));
  if (FMT == QAT_ELEM_E2M3) asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(b), "f"(a));
  if (FMT == QAT_ELEM_E3M2) asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(h) : "f"(b), "f"(a));
  return h;
}

// the values of a code pair as elem_enc2 packs it
template <int FMT>
__device__ __forceinline__ void elem_dec2(uint32_t c, float& a, float& b) {
  uint32_t h2;
  if (FMT == QAT_ELEM_E2M1) {
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(c));
    a = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
    b = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
    return;
  }
  const uint16_t c16 = (uint16_t)c;
  if (FMT == QAT_ELEM_E4M3) asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  if (FMT == QAT_ELEM_E5M2) asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(c16));
  if (FMT == QAT_ELEM_E2M3) asm("cvt.rn.f16x2.e2m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  if (FMT == QAT_ELEM_E3M2) asm("cvt.rn.f16x2.e3m2x2 %0, %1;" : "=r"(h2) : "h"(c16));
  a = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
  b = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

// E4M3 saturating round to nearest even of one value, and its code
__device__ __forceinline__ float e4m3_round(float s, uint32_t& code) {
  float r, unused;
  const uint32_t c2 = elem_enc2<QAT_ELEM_E4M3>(s, 0.0f);
  code = c2 & 0xffu;
  elem_dec2<QAT_ELEM_E4M3>(c2, r, unused);
  return r;
}

// floor(log2 a) of a positive finite binary32 value (subnormals included)
__device__ __forceinline__ int ilog2f(uint32_t bits) {
  const int E = (int)(bits >> 23);
  return E ? E - 127 : (31 - __clz((int)(bits & 0x7fffffu))) - 149;
}

// The block scale from the block's finite absmax (bits), the tensor scale g
// (KIND E4M3); the scale code (E8M0 byte, E4M3 byte) in `code`.
template <int FMT, int KIND>
__device__ __forceinline__ float block_scale(uint32_t amax_bits, float g, uint32_t& code) {
  constexpr float kMax = ElemFmt<FMT>::kMax;
  float X;
  code = 0u;
  if (KIND == QAT_BLOCK_SCALE_E8M0) {
    int es = (amax_bits ? ilog2f(amax_bits) : 0) - ElemFmt<FMT>::kEmax;
    es = es < -127 ? -127 : (es > 127 ? 127 : es);
    code = (uint32_t)(es + 127);
    X = es >= -126 ? __uint_as_float((uint32_t)(es + 127) << 23) : __uint_as_float(0x00400000u);
  } else if (KIND == QAT_BLOCK_SCALE_E4M3) {
    const float c = e4m3_round(__fdiv_rn(__fdiv_rn(__uint_as_float(amax_bits), kMax), g), code);
    X = __fmul_rn(c, g);
  } else {
    X = __fdiv_rn(__uint_as_float(amax_bits), kMax);
  }
  return X > 0.0f ? X : 1.0f;
}

template <typename T, int FMT, int KIND, int BLOCK>
__global__ void __launch_bounds__(256) k_block_fq(const void* __restrict__ x, int64_t n,
                                                  const uint4* __restrict__ part, int nparts,
                                                  float* tensor_scale, void* y, uint8_t* codes,
                                                  void* bscales, uint32_t* mask,
                                                  int32_t* flags) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC), LPB = BLOCK / VEC;
  constexpr float kMax = ElemFmt<FMT>::kMax;
  static_assert(LPB >= 1 && LPB <= 4, "a block is 1 to 4 lanes");
  __shared__ __align__(16) uint32_t red[4 * 8];
  __shared__ float g_sh;
  // E4M3 scales: the tensor's finite absmax from the statistics pass (g and
  // the non-finite flag); the other kinds see their non-finite values here
  if (KIND == QAT_BLOCK_SCALE_E4M3) {
    // launched early (after the statistics pass): request the warp's first
    // tile into L2, then wait for the partials
    {
      const int64_t t0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
      if (t0 * kTile < n) prefetch_tile_l2<T>(x, n, t0, threadIdx.x & 31);
    }
    pdl_wait();
    const Stats st = reduce_partials<kMMNone>(part, nparts, red);
    if (threadIdx.x == 0) {
      const float g = __fdiv_rn(st.absmax_f(), kMax * 448.0f);
      g_sh = g;
      if (blockIdx.x == 0) {
        if (tensor_scale) *tensor_scale = g;
        flag_or(flags, st.has_nonfinite() ? QAT_FLAG_NONFINITE_INPUT : 0);
      }
    }
    __syncthreads();
  } else if (blockIdx.x == 0 && threadIdx.x == 0 && tensor_scale) {
    *tensor_scale = 1.0f;
  }
  const float g = KIND == QAT_BLOCK_SCALE_E4M3 ? g_sh : 1.0f;
  int nonfinite = 0;
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t tile = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tile < ntiles;
       tile += wstride) {
    uint32_t mw[SLOTS];
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      const int64_t base = tile * kTile + (int64_t)(j * 32 + lane) * VEC;
      // n is a multiple of BLOCK, so a lane's vector is all present or absent
      const bool present = base < n;
      V32 v;
      if (present) v = ld_v32(static_cast<const char*>(x) + base * T::BYTES);
      else
#pragma unroll
        for (int k = 0; k < 8; ++k) v.w[k] = 0u;
      // the block's finite absmax over its LPB lanes
      Stats st;
      st.init<kMMNone>();
      st.add_absmax<T>(v);
      nonfinite |= (int)st.nonfinite;
      uint32_t am = st.amax;
#pragma unroll
      for (int o = 1; o < LPB; o <<= 1) am = max(am, __shfl_xor_sync(kFull, am, o));
      uint32_t scode;
      const float X = block_scale<FMT, KIND>(am, g, scode);
      if (present && bscales && (lane % LPB) == 0) {
        const int64_t b = base / BLOCK;
        if (KIND == QAT_BLOCK_SCALE_FP32)
          static_cast<float*>(bscales)[b] = X;
        else
          static_cast<uint8_t*>(bscales)[b] = (uint8_t)scode;
      }
      OutVec<T> ov;
      uint32_t mb = 0u;
      uint32_t cw[VEC / 4] = {};  // the vector's codes: a byte per element (FP4: a nibble)
      // The quotient t = RN(x / X) without a division: for a power-of-two
      // scale the product with its exact reciprocal; otherwise, for a finite
      // vector and a scale in the reciprocal's safe range, the exact quotient
      // of the residual steps (a quotient small enough to underflow rounds to
      // 0 in every element format either way); else the IEEE division.
      const bool fin = st.nonfinite == 0u;
      const bool quot = KIND != QAT_BLOCK_SCALE_E8M0 && fin && quot_scale_ok(X);
      float inv = 0.0f;
      if (KIND == QAT_BLOCK_SCALE_E8M0) {
        const int ei = 127 - (int)(__float_as_uint(X) >> 23);  // -es (X normal)
        inv = __float_as_uint(X) >= 0x00800000u
                  ? __uint_as_float((uint32_t)(ei + 127) << 23)
                  : __uint_as_float(0x7f000000u);  // X = 2^-127: 1 / X = 2^127
      } else if (quot) {
        inv = __frcp_rn(X);
      }
#pragma unroll
      for (int e = 0; e < VEC; e += 2) {
        const float xa = elem<T>(v, e), xb = elem<T>(v, e + 1);
        float ta, tb;
        if (KIND == QAT_BLOCK_SCALE_E8M0) {
          mul2(xa, xb, inv, inv, ta, tb);
        } else if (quot) {
          quotient_rn2(xa, xb, inv, -X, ta, tb);
          // the residual steps turn -0 into +0; X > 0, so t has the sign of x
          ta = copysignf(ta, xa);
          tb = copysignf(tb, xb);
        } else {
          ta = __fdiv_rn(xa, X);
          tb = __fdiv_rn(xb, X);
        }
        const bool na = isnan(ta), nb = isnan(tb);
        const bool nan_code = FMT == QAT_ELEM_E4M3 || FMT == QAT_ELEM_E5M2;
        const uint32_t c2 =
            elem_enc2<FMT>(na && !nan_code ? 0.0f : ta, nb && !nan_code ? 0.0f : tb);
        float qa, qb;
        elem_dec2<FMT>(c2, qa, qb);
        float ya = __fmul_rn(qa, X), yb = __fmul_rn(qb, X);
        if (na) ya = __uint_as_float(0x7fc00000u);
        if (nb) yb = __uint_as_float(0x7fc00000u);
        ov.set2(e, ya, yb);
        if (T::BYTES == 2 && (na || nb)) {
          // the canonical bf16 NaN (the packing conversion writes its own)
          uint32_t& w = ov.v.w[e >> 1];
          if (na) w = (w & 0xffff0000u) | 0x7fc0u;
          if (nb) w = (w & 0x0000ffffu) | 0x7fc00000u;
        }
        mb |= (uint32_t)(fabsf(ta) <= kMax) << e;
        mb |= (uint32_t)(fabsf(tb) <= kMax) << (e + 1);
        if (ElemFmt<FMT>::kBits == 4) {
          cw[e >> 3] |= (c2 & 0xffu) << (8 * ((e >> 1) & 3));
        } else {
          cw[e >> 2] |= (c2 & 0xffffu) << (8 * (e & 3));
        }
      }
      if (present) {
        if (y) st_v32(static_cast<char*>(y) + base * T::BYTES, ov.v);
        if (codes) {
          if (ElemFmt<FMT>::kBits == 4) {
            uint8_t* p = codes + base / 2;
            if (VEC == 16) *reinterpret_cast<uint2*>(p) = make_uint2(cw[0], cw[1]);
            else *reinterpret_cast<uint32_t*>(p) = cw[0];
          } else {
            uint8_t* p = codes + base;
            if (VEC == 16) *reinterpret_cast<uint4*>(p) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            else *reinterpret_cast<uint2*>(p) = make_uint2(cw[0], cw[1]);
          }
        }
      }
      mw[j] = mask_word_of_slot<VEC>(present ? mb : 0u, lane);
    }
    if (mask) {
      const uint32_t w = gather_tile_word<VEC, SLOTS>(mw, lane);
      const int64_t wi = tile * 32 + lane;
      if (wi < (n + 31) / 32) mask[wi] = w;
    }
  }
  if (KIND != QAT_BLOCK_SCALE_E4M3) warp_flag_or(flags, nonfinite ? QAT_FLAG_NONFINITE_INPUT : 0);
}

template <typename T, int FMT, int KIND>
static void block_t(int64_t block, const void* x, int64_t n, const void* ws, int nparts,
                    float* tensor_scale, void* y, uint8_t* codes, void* bscales, uint32_t* mask,
                    int32_t* flags, cudaStream_t s) {
  const int64_t ntiles = (n + kTile - 1) / kTile;
  int64_t g = (ntiles + 7) / 8;
  const int64_t cap = (int64_t)device_info().sms * 8;
  const int grid = (int)(g > cap ? cap : (g < 1 ? 1 : g));
  const uint4* part = static_cast<const uint4*>(ws);
  // E4M3 scales follow the call's statistics pass: launched early
  const bool pdl = KIND == QAT_BLOCK_SCALE_E4M3;
  if (block == 16)
    launch_kernel(k_block_fq<T, FMT, KIND, 16>, dim3(grid), dim3(256), 0, s, pdl, x, n, part,
                  nparts, tensor_scale, y, codes, bscales, mask, flags);
  else
    launch_kernel(k_block_fq<T, FMT, KIND, 32>, dim3(grid), dim3(256), 0, s, pdl, x, n, part,
                  nparts, tensor_scale, y, codes, bscales, mask, flags);
}

template <typename T, int FMT>
static void block_fmt_t(int kind, int64_t block, const void* x, int64_t n, const void* ws,
                        int nparts, float* tensor_scale, void* y, uint8_t* codes, void* bscales,
                        uint32_t* mask, int32_t* flags, cudaStream_t s) {
  if (kind == QAT_BLOCK_SCALE_E8M0)
    block_t<T, FMT, QAT_BLOCK_SCALE_E8M0>(block, x, n, ws, nparts, tensor_scale, y, codes,
                                          bscales, mask, flags, s);
  else if (kind == QAT_BLOCK_SCALE_E4M3)
    block_t<T, FMT, QAT_BLOCK_SCALE_E4M3>(block, x, n, ws, nparts, tensor_scale, y, codes,
                                          bscales, mask, flags, s);
  else
    block_t<T, FMT, QAT_BLOCK_SCALE_FP32>(block, x, n, ws, nparts, tensor_scale, y, codes,
                                          bscales, mask, flags, s);
}

qat_status launch_block_fq(qat_dtype dt, int fmt, int kind, int64_t block, const void* x,
                           int64_t n, const void* ws, int nparts, float* tensor_scale, void* y,
                           uint8_t* codes, void* bscales, uint32_t* mask, int32_t* flags,
                           cudaStream_t s) {
#define QAT_BF(T, F) \
  block_fmt_t<T, F>(kind, block, x, n, ws, nparts, tensor_scale, y, codes, bscales, mask, flags, s)
#define QAT_BT(T)                                                  \
  switch (fmt) {                                                   \
    case QAT_ELEM_E4M3: QAT_BF(T, QAT_ELEM_E4M3); break;           \
    case QAT_ELEM_E5M2: QAT_BF(T, QAT_ELEM_E5M2); break;           \
    case QAT_ELEM_E2M3: QAT_BF(T, QAT_ELEM_E2M3); break;           \
    case QAT_ELEM_E3M2: QAT_BF(T, QAT_ELEM_E3M2); break;           \
    default: QAT_BF(T, QAT_ELEM_E2M1); break;                      \
  }
  if (dt == QAT_F32) {
    QAT_BT(F32)
  } else {
    QAT_BT(BF16)
  }
#undef QAT_BT
#undef QAT_BF
  count_launch(1);
  return launch_status();
}

}  // namespace qat
