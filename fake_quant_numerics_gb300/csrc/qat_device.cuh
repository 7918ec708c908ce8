// qat_device.cuh -- device-side building blocks shared by the library's kernels.
//
// Data movement: every lane moves 32-byte vectors (ld/st .v8.b32, the 256-bit
// global accesses of sm_100-class GPUs), so a warp instruction covers 1 KiB of
// contiguous memory.  A "tile" is 1024 consecutive elements handled by one
// warp: it owns exactly 32 mask words, which a warp writes with one coalesced
// 128-byte store.
//
// Arithmetic: every floating-point operation that decides an output bit uses
// an explicitly rounded intrinsic (__fdiv_rn, __fmul_rn, __fsub_rn), so the
// results do not depend on FMA contraction; no flush-to-zero anywhere.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qat.h"
#include "qat_sr.h"

namespace qat {

constexpr int kTile = 1024;  // elements per warp tile
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kMaxPartials = 1024;  // cross-CTA partial statistics slots

// ---------------------------------------------------------------------------
// element types: 32-byte vectors of VEC elements
// ---------------------------------------------------------------------------
struct F32 {
  static constexpr int VEC = 8;
  static constexpr int BYTES = 4;
  static constexpr qat_dtype kDtype = QAT_F32;
};
struct BF16 {
  static constexpr int VEC = 16;
  static constexpr int BYTES = 2;
  static constexpr qat_dtype kDtype = QAT_BF16;
};

struct V32 {
  uint32_t w[8];
};

__device__ __forceinline__ V32 ld_v32(const void* p) {
  V32 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
        "=r"(v.w[6]), "=r"(v.w[7])
      : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v32(void* p, const V32& v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7])
               : "memory");
}

// element e of a vector, widened to fp32 bits
template <typename T>
__device__ __forceinline__ uint32_t elem_bits(const V32& v, int e);
template <>
__device__ __forceinline__ uint32_t elem_bits<F32>(const V32& v, int e) {
  return v.w[e];
}
template <>
__device__ __forceinline__ uint32_t elem_bits<BF16>(const V32& v, int e) {
  uint32_t w = v.w[e >> 1];
  return (e & 1) ? (w & 0xffff0000u) : (w << 16);
}

template <typename T>
__device__ __forceinline__ float elem(const V32& v, int e) {
  return __uint_as_float(elem_bits<T>(v, e));
}

// scalar element i of a tensor (tails only)
template <typename T>
__device__ __forceinline__ uint32_t load_elem_bits(const void* x, int64_t i);
template <>
__device__ __forceinline__ uint32_t load_elem_bits<F32>(const void* x, int64_t i) {
  return static_cast<const uint32_t*>(x)[i];
}
template <>
__device__ __forceinline__ uint32_t load_elem_bits<BF16>(const void* x, int64_t i) {
  return static_cast<uint32_t>(static_cast<const uint16_t*>(x)[i]) << 16;
}

// Load the VEC elements starting at element `base`; `cnt` of them exist
// (cnt == VEC is the fast path; missing elements read as +0).  The tail loop
// is fully unrolled with predicates so the vector stays in registers.  UA: x
// holds whole elements but may be off the 32-byte grid, so every element is
// loaded on its own.
template <typename T, bool UA = false>
__device__ __forceinline__ V32 load_vec(const void* x, int64_t base, int cnt) {
  if (!UA && cnt >= T::VEC) return ld_v32(static_cast<const char*>(x) + base * T::BYTES);
  V32 v;
#pragma unroll
  for (int j = 0; j < 8; ++j) v.w[j] = 0u;
#pragma unroll
  for (int e = 0; e < T::VEC; ++e) {
    if (e < cnt) {
      uint32_t b = load_elem_bits<T>(x, base + e);
      if (T::BYTES == 4) {
        v.w[e] = b;
      } else {
        v.w[e >> 1] |= (e & 1) ? (b & 0xffff0000u) : (b >> 16);
      }
    }
  }
  return v;
}

// ---------------------------------------------------------------------------
// tile loads with a rolling prefetch
// ---------------------------------------------------------------------------
// `v` may already hold this tile (have, full tiles only); after a slot is
// consumed, the same slot of the warp's next full tile (next >= 0) is
// requested into it, so loads stay in flight while the warp computes.
template <typename T, bool FULL>
__device__ __forceinline__ void tile_load(const void* __restrict__ x, int64_t n, int64_t tile,
                                          V32 (&v)[kTile / (32 * T::VEC)],
                                          int (&cnt)[kTile / (32 * T::VEC)], bool have, int lane) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC);
  const int64_t tb = tile * kTile;
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) {
    const int64_t base = tb + (int64_t)(j * 32 + lane) * VEC;
    if (FULL) {
      cnt[j] = VEC;
      if (!have) v[j] = ld_v32(static_cast<const char*>(x) + base * T::BYTES);
    } else {
      const int64_t c = n - base;
      cnt[j] = c >= VEC ? VEC : (c > 0 ? (int)c : 0);
      v[j] = load_vec<T>(x, cnt[j] > 0 ? base : 0, cnt[j]);
    }
  }
}

template <typename T>
__device__ __forceinline__ void slot_prefetch(const void* __restrict__ x, int64_t next, int j,
                                              V32& vj, int lane) {
  if (next >= 0)
    vj = ld_v32(static_cast<const char*>(x) +
                (next * kTile + (int64_t)(j * 32 + lane) * T::VEC) * T::BYTES);
}

// fp32 -> bf16 bits, round to nearest even (cvt.rn.bf16x2.f32 packs hi, lo)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Output vector builder: y values (fp32) -> the output dtype's 32 bytes.
template <typename T>
struct OutVec;
template <>
struct OutVec<F32> {
  V32 v;
  __device__ __forceinline__ void set(int e, float y) { v.w[e] = __float_as_uint(y); }
  __device__ __forceinline__ void set2(int e, float ya, float yb) {
    v.w[e] = __float_as_uint(ya);
    v.w[e + 1] = __float_as_uint(yb);
  }
};
template <>
struct OutVec<BF16> {
  V32 v;
  float pend;
  __device__ __forceinline__ void set(int e, float y) {
    if ((e & 1) == 0) {
      pend = y;
    } else {
      v.w[e >> 1] = pack_bf16x2(pend, y);
    }
  }
  __device__ __forceinline__ void set2(int e, float ya, float yb) { v.w[e >> 1] = pack_bf16x2(ya, yb); }
};

// Store the first `cnt` elements of an output vector at element `base` (UA:
// element by element, y being possibly off the 32-byte grid).
template <typename T, bool UA = false>
__device__ __forceinline__ void store_vec(void* y, int64_t base, const V32& v, int cnt) {
  if (!UA && cnt >= T::VEC) {
    st_v32(static_cast<char*>(y) + base * T::BYTES, v);
    return;
  }
#pragma unroll
  for (int e = 0; e < T::VEC; ++e) {
    if (e < cnt) {
      if (T::BYTES == 4) {
        static_cast<uint32_t*>(y)[base + e] = v.w[e];
      } else {
        uint32_t w = v.w[e >> 1];
        static_cast<uint16_t*>(y)[base + e] = (uint16_t)((e & 1) ? (w >> 16) : (w & 0xffffu));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// codes: int8 (VEC bytes per lane) or packed int4 (VEC/2 bytes per lane,
// element 2j in the high nibble of byte j).  Packing uses
// cvt.pack.sat.{s8,s4}.s32.b32 d, a, b, c  ->  d = c << 2w | sat(a) << w | sat(b)
// (w = 8 or 4); the codes are already in range, so the saturation never acts.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_s8x2(int a, int b, uint32_t c) {
  uint32_t d;
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t pack_s4x2(int a, int b, uint32_t c) {
  uint32_t d;
  asm("cvt.pack.sat.s4.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <int BITS, int VEC>
struct CodeVec {
  static constexpr int NBYTES = BITS == 8 ? VEC : VEC / 2;
  static constexpr int NW = (NBYTES + 3) / 4;
  uint32_t w[NW];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int j = 0; j < NW; ++j) w[j] = 0u;
  }
  // codes of elements e and e + 1 (e even), packed into their word with the
  // cvt.pack chain; within a word, pairs must come in descending order
  // (the earlier bytes are shifted up by the later calls)
  __device__ __forceinline__ void set2(int e, int qa, int qb) {
    if (BITS == 8) {
      w[e >> 2] = pack_s8x2(qb, qa, w[e >> 2]);
    } else {
      w[e >> 3] = pack_s4x2(qa, qb, w[e >> 3]);
    }
  }
  // one code, any order (OR-ed into a cleared word)
  __device__ __forceinline__ void set(int e, int q) {
    if (BITS == 8) {
      w[e >> 2] |= (static_cast<uint32_t>(q) & 0xffu) << ((e & 3) * 8);
    } else {
      const int byte = e >> 1;
      w[byte >> 2] |= (static_cast<uint32_t>(q) & 0xfu) << ((byte & 3) * 8 + ((e & 1) ? 0 : 4));
    }
  }
  // store at element offset `base` (codes buffer byte offset base*BITS/8);
  // `cnt` elements present (absent ones must hold code 0)
  __device__ __forceinline__ void store(void* codes, int64_t base, int cnt) const {
    uint8_t* p = static_cast<uint8_t*>(codes) + (BITS == 8 ? base : base / 2);
    if (cnt >= VEC) {
      if (NBYTES == 16) {
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
      } else if (NBYTES == 8) {
        *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
      } else {
        *reinterpret_cast<uint32_t*>(p) = w[0];
      }
      return;
    }
    const int nb = BITS == 8 ? cnt : (cnt + 1) / 2;
#pragma unroll
    for (int b = 0; b < NBYTES; ++b)
      if (b < nb) p[b] = (uint8_t)(w[b >> 2] >> ((b & 3) * 8));
  }
};

// ---------------------------------------------------------------------------
// mask assembly: per slot a lane holds VEC mask bits; the 32/VEC lanes that
// share a mask word OR their shifted bits together.  After all slots of a
// tile, lane L holds tile word L.
// ---------------------------------------------------------------------------
template <int VEC>
__device__ __forceinline__ uint32_t mask_word_of_slot(uint32_t bits, int lane) {
  constexpr int LPW = 32 / VEC;  // lanes per mask word
  uint32_t w = bits << ((lane % LPW) * VEC);
#pragma unroll
  for (int o = 1; o < LPW; o <<= 1) w |= __shfl_xor_sync(kFull, w, o);
  return w;
}

template <int VEC, int SLOTS>
__device__ __forceinline__ uint32_t gather_tile_word(const uint32_t (&mw)[SLOTS], int lane) {
  constexpr int LPW = 32 / VEC;
  uint32_t out = 0u;
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) {
    uint32_t v = __shfl_sync(kFull, mw[j], (lane % VEC) * LPW);
    if (lane / VEC == j) out = v;
  }
  return out;
}

// ---------------------------------------------------------------------------
// packed fp32 pairs: Blackwell f32x2 arithmetic, one IEEE round-to-nearest
// operation per lane of the pair (the same results as two scalar ops)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mul2(float a0, float a1, float b0, float b1, float& r0, float& r1) {
  asm("{ .reg .b64 x, y, r;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
      " mul.rn.f32x2 r, x, y;\n mov.b64 {%0, %1}, r; }"
      : "=f"(r0), "=f"(r1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add2(float a0, float a1, float b0, float b1, float& r0, float& r1) {
  asm("{ .reg .b64 x, y, r;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
      " add.rn.f32x2 r, x, y;\n mov.b64 {%0, %1}, r; }"
      : "=f"(r0), "=f"(r1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float a0, float a1, float b0, float b1, float& r0, float& r1) {
  asm("{ .reg .b64 x, y, r;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
      " sub.rn.f32x2 r, x, y;\n mov.b64 {%0, %1}, r; }"
      : "=f"(r0), "=f"(r1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// r = a * b + c, one rounding per lane
__device__ __forceinline__ void fma2(float a0, float a1, float b0, float b1, float c0, float c1,
                                     float& r0, float& r1) {
  asm("{ .reg .b64 x, y, z, r;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
      " mov.b64 z, {%6, %7};\n fma.rn.f32x2 r, x, y, z;\n mov.b64 {%0, %1}, r; }"
      : "=f"(r0), "=f"(r1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// max with NaN propagation (max.NaN): NaN if either input is NaN
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
// three-input forms (sm_100 and later): one instruction for two steps of a fold
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmin3_nan(float a, float b, float c) {
  float r;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// ---------------------------------------------------------------------------
// statistics on fp32 bit patterns: finite absmax (as bits of |x|), min / max
// as order-preserving keys (-0 below +0), non-finite detection
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(uint32_t u) {
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint32_t key_to_bits(uint32_t k) {
  return (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
}
constexpr uint32_t kKeyPosInf = 0xff800000u;  // order_key(+inf)
constexpr uint32_t kKeyNegInf = 0x007fffffu;  // order_key(-inf)

// What a Stats fold tracks besides the finite absmax:
//   kMMNone  -- nothing (symmetric grids, FP8);
//   kMMFloat -- finite min / max as floats (calibration of affine grids, where
//               the sign of a zero extreme cannot matter: only min(m, 0) and
//               max(M, 0) are used);
//   kMMKeys  -- finite min / max as order keys with -0 below +0 (the
//               statistics entry point, whose outputs expose the zero sign).
constexpr int kMMNone = 0, kMMFloat = 1, kMMKeys = 2;

struct Stats {
  uint32_t amax;       // bits of the finite absmax
  uint32_t nonfinite;  // 1 if a NaN/Inf was seen
  uint32_t kmin;       // finite min: key (kMMKeys) or float bits (kMMFloat)
  uint32_t kmax;       // finite max: key (kMMKeys) or float bits (kMMFloat)
  template <int MM>
  __device__ __forceinline__ void init() {
    amax = 0u;
    nonfinite = 0u;
    kmin = MM == kMMFloat ? 0x7f800000u : kKeyPosInf;  // +inf
    kmax = MM == kMMFloat ? 0xff800000u : kKeyNegInf;  // -inf
  }
  // one element, NaN/Inf filtered out (the general path)
  template <int MM>
  __device__ __forceinline__ void add(uint32_t u) {
    const uint32_t a = u & 0x7fffffffu;
    const bool fin = a < 0x7f800000u;
    amax = max(amax, fin ? a : 0u);
    nonfinite |= fin ? 0u : 1u;
    if (MM == kMMKeys) {
      const uint32_t k = order_key(u);
      kmin = min(kmin, fin ? k : kKeyPosInf);
      kmax = max(kmax, fin ? k : kKeyNegInf);
    } else if (MM == kMMFloat && fin) {
      kmin = __float_as_uint(fminf(__uint_as_float(kmin), __uint_as_float(u)));
      kmax = __float_as_uint(fmaxf(__uint_as_float(kmax), __uint_as_float(u)));
    }
  }
  // max.NaN of |x| over a 32-byte vector: the finite absmax bits, or a value
  // >= 0x7f800000 when the vector holds NaN or Inf
  template <typename T>
  __device__ __forceinline__ uint32_t vec_absmax_nan(const V32& v) const {
    if (T::BYTES == 2) {
      uint32_t m2 = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) m2 = bf16x2_max_nan(m2, v.w[k] & 0x7fff7fffu);
      return __float_as_uint(fmax_nan(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u)));
    }
    auto a = [&](int k) { return fabsf(__uint_as_float(v.w[k])); };
    float m = fmax3_nan(a(0), a(1), a(2));
    m = fmax3_nan(m, a(3), a(4));
    m = fmax3_nan(m, a(5), a(6));
    return __float_as_uint(fmax_nan(m, a(7)));
  }
  // absmax of one 32-byte vector (absent tail elements read +0): one max.NaN
  // per element (per two for bf16); only a vector holding NaN or Inf takes
  // the filtered per-element fold.
  template <typename T>
  __device__ __forceinline__ void add_absmax(const V32& v) {
    const uint32_t r = vec_absmax_nan<T>(v);
    if (r < 0x7f800000u) {
      amax = max(amax, r);
    } else {
#pragma unroll
      for (int e = 0; e < T::VEC; ++e) add<kMMNone>(elem_bits<T>(v, e));
    }
  }
  // finite min / max as floats of one full 32-byte vector (kMMFloat): the
  // running min and max folded with the elements by three-input min.NaN /
  // max.NaN, kept when both results are finite (then every element was: a
  // NaN makes both NaN, an Inf shows as the min or the max); a vector with a
  // NaN or Inf takes the filtered per-element fold instead
  template <typename T>
  __device__ __forceinline__ void add_minmax_float(const V32& v) {
    auto x = [&](int e) { return __uint_as_float(elem_bits<T>(v, e)); };
    float mn = __uint_as_float(kmin), mx = __uint_as_float(kmax);
#pragma unroll
    for (int e = 0; e < T::VEC; e += 2) {
      mn = fmin3_nan(mn, x(e), x(e + 1));
      mx = fmax3_nan(mx, x(e), x(e + 1));
    }
    if (fabsf(mn) < __int_as_float(0x7f800000) && fabsf(mx) < __int_as_float(0x7f800000)) {
      kmin = __float_as_uint(mn);
      kmax = __float_as_uint(mx);
    } else {
#pragma unroll
      for (int e = 0; e < T::VEC; ++e) add<kMMFloat>(elem_bits<T>(v, e));
    }
  }
  template <int MM>
  __device__ __forceinline__ void merge(const Stats& o) {
    amax = max(amax, o.amax);
    nonfinite |= o.nonfinite;
    if (MM == kMMKeys) {
      kmin = min(kmin, o.kmin);
      kmax = max(kmax, o.kmax);
    } else if (MM == kMMFloat) {
      kmin = __float_as_uint(fminf(__uint_as_float(kmin), __uint_as_float(o.kmin)));
      kmax = __float_as_uint(fmaxf(__uint_as_float(kmax), __uint_as_float(o.kmax)));
    }
  }
  // reduce over `width` consecutive lanes (a power of two <= 32); the whole
  // warp takes one redux.sync per field (amax bits of a non-negative float
  // and order keys are monotone as unsigned integers)
  template <int MM>
  __device__ __forceinline__ void reduce_lanes(int width) {
    if (width == 32) {
      amax = __reduce_max_sync(kFull, amax);
      nonfinite = __reduce_or_sync(kFull, nonfinite);
      if (MM == kMMKeys) {
        kmin = __reduce_min_sync(kFull, kmin);
        kmax = __reduce_max_sync(kFull, kmax);
      } else if (MM == kMMFloat) {
        kmin = key_to_bits(__reduce_min_sync(kFull, order_key(kmin)));
        kmax = key_to_bits(__reduce_max_sync(kFull, order_key(kmax)));
      }
      return;
    }
    for (int o = 1; o < width; o <<= 1) {
      Stats t;
      t.amax = __shfl_xor_sync(kFull, amax, o);
      t.nonfinite = __shfl_xor_sync(kFull, nonfinite, o);
      if (MM != kMMNone) {
        t.kmin = __shfl_xor_sync(kFull, kmin, o);
        t.kmax = __shfl_xor_sync(kFull, kmax, o);
      }
      merge<MM>(t);
    }
  }
  __device__ __forceinline__ bool has_nonfinite() const { return nonfinite != 0u; }
  __device__ __forceinline__ float absmax_f() const { return __uint_as_float(amax); }
  template <int MM>
  __device__ __forceinline__ float min_f() const {
    return __uint_as_float(MM == kMMKeys ? key_to_bits(kmin) : kmin);
  }
  template <int MM>
  __device__ __forceinline__ float max_f() const {
    return __uint_as_float(MM == kMMKeys ? key_to_bits(kmax) : kmax);
  }
  __device__ __forceinline__ uint4 pack() const { return make_uint4(amax, nonfinite, kmin, kmax); }
  __device__ __forceinline__ void unpack(const uint4& p) {
    amax = p.x;
    nonfinite = p.y;
    kmin = p.z;
    kmax = p.w;
  }
};

// statistics of one full vector
template <typename T, int MM>
__device__ __forceinline__ void stats_add_vec(Stats& st, const V32& v) {
  if (MM == kMMKeys) {
#pragma unroll
    for (int e = 0; e < T::VEC; ++e) st.add<kMMKeys>(elem_bits<T>(v, e));
  } else if (MM == kMMFloat) {
    st.add_minmax_float<T>(v);
  } else {
    st.add_absmax<T>(v);
  }
}

// Block-wide reduction of Stats (all threads get the result).  `red` needs
// 4 * (blockDim.x / 32) words of shared memory.
template <int MM>
__device__ __forceinline__ Stats block_reduce_stats(Stats s, uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  s.reduce_lanes<MM>(32);
  __syncthreads();  // red may still be read from a previous use
  if (lane == 0) reinterpret_cast<uint4*>(red)[warp] = s.pack();
  __syncthreads();
  Stats t;
  t.init<MM>();
  for (int w = 0; w < nw; ++w) {
    Stats o;
    o.unpack(reinterpret_cast<const uint4*>(red)[w]);
    t.merge<MM>(o);
  }
  return t;
}

// ---------------------------------------------------------------------------
// the correctly rounded quotient without a per-element division
//
// With y = RN(1/s) (within half an ulp of 1/s) and Q = x/s:
//   q0 = RN(x y) is within 2^-24 |Q| + ulp/2 < 2 ulp(Q) of Q;
//   r0 = RN(x - q0 s) (one fma) is s (Q - q0)(1 + eta), |eta| <= 2^-24;
//   q1 = RN(q0 + r0 y) (one fma) rounds Q + (Q - q0)(eta + delta + eta delta),
//   |delta| = |s y - 1| <= 2^-24, i.e. Q moved by less than 2^-22 ulp(Q), so
//   q1 is within one ulp of Q (faithful);
//   r1 = x - q1 s is then exactly representable and one fma gives it, and
//   q2 = RN(q1 + r1 y) = RN(Q) by Markstein's theorem (y correctly rounded,
//   q1 within one ulp; P. Markstein, IBM J. Res. Dev. 34(1), 1990).
// q2 is the IEEE quotient RN(x/s) itself, so rint(q2) and an FP8 cast of q2
// equal those of the divided value.  Preconditions: no overflow and no
// underflow of the products and remainders, which the scale range below
// guarantees for |Q| >= 2^-20 (smaller quotients round to 0 under rint
// whatever the last bits are).
// Safe scales: s and 1/s normal and far from overflow, s in [2^-80, 2^100].
// ---------------------------------------------------------------------------
__device__ __forceinline__ float quotient_rn(float x, float rcp, float ns) {
  const float q0 = __fmul_rn(x, rcp);
  const float q1 = __fmaf_rn(__fmaf_rn(q0, ns, x), rcp, q0);
  return __fmaf_rn(__fmaf_rn(q1, ns, x), rcp, q1);
}

// the same for a pair (f32x2 arithmetic); ns = -s
__device__ __forceinline__ void quotient_rn2(float xa, float xb, float rcp, float ns, float& qa,
                                             float& qb) {
  float ra, rb;
  mul2(xa, xb, rcp, rcp, qa, qb);
  fma2(qa, qb, ns, ns, xa, xb, ra, rb);
  fma2(ra, rb, rcp, rcp, qa, qb, qa, qb);
  fma2(qa, qb, ns, ns, xa, xb, ra, rb);
  fma2(ra, rb, rcp, rcp, qa, qb, qa, qb);
}

__device__ __forceinline__ bool quot_scale_ok(float s) { return s >= 0x1p-80f && s <= 0x1p100f; }

// ---------------------------------------------------------------------------
// integer grid parameters of one unit
// ---------------------------------------------------------------------------
struct IntParams {
  float s;         // scale
  float rcp;       // RN(1/s), used when `fast`
  float wlo, whi;  // STE window [(qmin-zp)*s, (qmax-zp)*s]
  float klof, khif;  // the clamp range as floats
  int klo, khi;    // clamp range of k = q - zp
  int zp;
  int dead;        // unit outputs are codes 0, y +0, mask 0
  int fast;        // calibrated unit with a scale in the safe range (quot_scale_ok):
                   // 1, or 2 when a symmetric unit's codes need the clamp too
                   // (calibration options can leave values beyond the range),
                   // or 3 when, besides, a quotient x * RN(1/s) may overflow
                   // binary32 (kQuotGuard): the per-tensor map then clamps x
                   // to +-2^24 s before the quotient, the other maps take the
                   // division path for the unit
};

// A calibrated unit whose largest magnitude times RN(1/s) stays at or below
// this bound keeps every product and remainder of quotient_rn finite.
constexpr float kQuotGuard = 0x1p64f;

template <int BITS, bool AFFINE>
struct QRange {
  static constexpr int qmin = AFFINE ? (BITS == 8 ? -128 : -8) : (BITS == 8 ? -127 : -7);
  static constexpr int qmax = BITS == 8 ? 127 : 7;
};

__device__ __forceinline__ void finish_params(IntParams& p, int qmin, int qmax) {
  p.klo = qmin - p.zp;
  p.khi = qmax - p.zp;
  p.klof = (float)p.klo;
  p.khif = (float)p.khi;
  p.wlo = __fmul_rn(__int2float_rn(qmin - p.zp), p.s);
  p.whi = __fmul_rn(__int2float_rn(qmax - p.zp), p.s);
}

// Calibration (QuantParams::from_absmax / from_minmax).  Returns the flag bit
// (0, QAT_FLAG_NONFINITE_CALIB or QAT_FLAG_DEGENERATE).
// With options (CalOpts): the range times co.clip before the formulas, the
// scale rounded to binary16 after them (the zero point follows the rounded
// scale).
template <int BITS, bool AFFINE, int MM>
__device__ __forceinline__ int calibrate(const Stats& st, IntParams& p,
                                         const CalOpts& co = CalOpts{1.0f, 0, 0}) {
  constexpr int qmin = QRange<BITS, AFFINE>::qmin, qmax = QRange<BITS, AFFINE>::qmax;
  int degenerate = 0;
  p.zp = 0;
  if (!AFFINE) {
    float A = st.absmax_f();
    if (co.clip != 1.0f) A = __fmul_rn(co.clip, A);
    p.s = __fdiv_rn(A, (float)qmax);
    if (co.fp16) p.s = __half2float(__float2half_rn(p.s));
    degenerate = !(A > 0.0f) || !(p.s > 0.0f) || isinf(p.s);
  } else {
    float mn = st.min_f<MM>(), mx = st.max_f<MM>();
    if (co.clip != 1.0f) {
      mn = __fmul_rn(co.clip, mn);
      mx = __fmul_rn(co.clip, mx);
    }
    float rmin = (mn < 0.0f) ? mn : 0.0f;
    float rmax = (mx > 0.0f) ? mx : 0.0f;
    float range = __fsub_rn(rmax, rmin);
    p.s = __fdiv_rn(range, (float)(qmax - qmin));
    if (co.fp16) p.s = __half2float(__float2half_rn(p.s));
    degenerate = !(range > 0.0f) || !(p.s > 0.0f) || isinf(p.s);
    if (!degenerate) {
      float t = __fsub_rn((float)qmin, __fdiv_rn(rmin, p.s));
      float z = rintf(t);
      z = fminf(fmaxf(z, (float)qmin), (float)qmax);
      p.zp = (int)z;
    }
  }
  int flag = st.has_nonfinite() ? QAT_FLAG_NONFINITE_CALIB : (degenerate ? QAT_FLAG_DEGENERATE : 0);
  p.dead = flag != 0;
  p.fast = 0;
  p.rcp = 0.0f;
  if (!p.dead && quot_scale_ok(p.s)) {
    p.rcp = __frcp_rn(p.s);
    const bool opts = co.clamp || co.clip != 1.0f || co.fp16;
    p.fast = (!AFFINE && opts) ? 2 : 1;
    // With options a value can lie far beyond the range; its quotient by s
    // must stay finite on the reciprocal path (QuantParams::quantize clamps
    // the real quotient, so such a value takes an end code).  The statistics
    // of a percentile calibration (clamp) are the quantiles, not the unit's
    // extremes, so it always takes the guard.
    if (opts) {
      const float ext =
          AFFINE ? fmaxf(fabsf(st.min_f<MM>()), fabsf(st.max_f<MM>())) : st.absmax_f();
      if (co.clamp || !(__fmul_rn(ext, p.rcp) <= kQuotGuard)) p.fast = 3;
    }
  }
  finish_params(p, qmin, qmax);
  return flag;
}

// The parameters of lane `src` (calibrated there), as the map needs them:
// s, rcp, the window, zp and the dead / fast bits travel; the clamp range is
// rebuilt from zp.  For the symmetric grid wlo = RN(qmin s) = -RN(qmax s).
template <int BITS, bool AFFINE>
__device__ __forceinline__ IntParams shfl_params(const IntParams& q, int src) {
  constexpr int qmin = QRange<BITS, AFFINE>::qmin, qmax = QRange<BITS, AFFINE>::qmax;
  IntParams p;
  p.s = __shfl_sync(kFull, q.s, src);
  p.rcp = __shfl_sync(kFull, q.rcp, src);
  p.whi = __shfl_sync(kFull, q.whi, src);
  const int bitsw =
      __shfl_sync(kFull, q.dead | (q.fast << 1) | (AFFINE ? ((q.zp & 0xff) << 3) : 0), src);
  p.dead = bitsw & 1;
  p.fast = (bitsw >> 1) & 3;
  if (AFFINE) {
    p.zp = (int)(int8_t)(uint8_t)((bitsw >> 3) & 0xff);
    p.wlo = __shfl_sync(kFull, q.wlo, src);
  } else {
    p.zp = 0;
    p.wlo = -p.whi;
  }
  p.klo = qmin - p.zp;
  p.khi = qmax - p.zp;
  p.klof = (float)p.klo;
  p.khif = (float)p.khi;
  return p;
}

// Given parameters: validity check.
template <int BITS, bool AFFINE>
__device__ __forceinline__ int given_params(float s, int zp, IntParams& p) {
  constexpr int qmin = QRange<BITS, AFFINE>::qmin, qmax = QRange<BITS, AFFINE>::qmax;
  p.s = s;
  p.zp = AFFINE ? zp : 0;
  int bad = !(s > 0.0f) || isinf(s) || p.zp < qmin || p.zp > qmax;
  p.dead = bad;
  p.fast = 0;
  p.rcp = 0.0f;
  finish_params(p, qmin, qmax);
  return bad ? QAT_FLAG_BAD_PARAMS : 0;
}

// One element: q = clamp(rne(x/s) + zp), y = (q - zp) * s, mask bit.
// NAN_TO_ZERO: a NaN quotient gives code 0 (given parameters only; a
// calibrated unit containing NaN is dead).
template <bool NAN_TO_ZERO>
__device__ __forceinline__ void int_elem(float x, const IntParams& p, int& q, float& y,
                                         uint32_t& m) {
  float r = __fdiv_rn(x, p.s);
  int k = __float2int_rn(r);  // saturating; NaN -> 0
  k = min(max(k, p.klo), p.khi);
  if (NAN_TO_ZERO && isnan(r)) k = -p.zp;
  q = k + p.zp;
  y = __fmul_rn(__int2float_rn(k), p.s);
  m = (x >= p.wlo) && (x <= p.whi);
}

// rint without the conversion unit: for |q| < 2^22, RN(q + M) with M = 1.5*2^23
// lies in [2^23, 2^24) where the spacing is 1, so it is M + rint(q) (ties to
// even, M being even); subtracting M back is exact and gives +0 for zero.  The
// bit pattern of M + k is 0x4b400000 + k, so the integer comes for free.
constexpr float kRintMagic = 12582912.0f;
constexpr uint32_t kRintMagicBits = 0x4b400000u;

// One vector of a calibrated unit with p.fast set.  A calibrated unit with
// p.fast holds only finite values (a NaN or Inf makes it dead), which the
// window test below relies on.
//   quotient: q = RN(x/s) by quotient_rn2, f = rint(q) by the magic constant;
//   k = clamp(f) (affine, or CL >= 1: p.fast == 2), y = k * s, code k + zp from
//   the bits of k + M;
//   CL == 2 (p.fast == 3): the quotient is taken of x clamped to
//     [-2^24 s, 2^24 s] (2^24 s is exact: s <= 2^100), so it stays finite; an
//     element beyond that bound has |x / s| > 2^24, far past every code, and
//     both forms give it the end code of its sign (the window test keeps x);
//   STE window: whi - |x| >= 0 (symmetric), whi - x >= 0 and x - wlo >= 0
//     (affine); RN never changes the sign of a difference and an exact zero
//     difference is +0, except (-0) - (+0) = -0: a lower bound of +0 is used
//     as -0 (x - (-0) is +0 for both zeros), and the whi side never meets
//     that case (whi >= +0, and whi - |x| has |x| >= +0).  So the sign bits
//     are the window test (affine: the sign of the product of the two
//     differences); they are shifted into the mask with funnel shifts,
//     highest element first.
// FULL == false: elements e >= cnt are absent (read as +0) and get code 0.
template <typename T, int BITS, bool AFFINE, bool FULL, int CL = 0>
__device__ __forceinline__ void int_vec_cal(const V32& v, const IntParams& p, int cnt,
                                            OutVec<T>& ov, CodeVec<BITS, T::VEC>& cv,
                                            uint32_t& mb) {
  constexpr int VEC = T::VEC;
  const float ns = -p.s;
  const float wlo = p.wlo == 0.0f ? -0.0f : p.wlo;
  const float kloM = __fadd_rn(p.klof, kRintMagic), khiM = __fadd_rn(p.khif, kRintMagic);
  const float xlim = CL == 2 ? __fmul_rn(p.s, 0x1p24f) : 0.0f;
  cv.clear();
  uint32_t out = 0u;  // out-of-window bits
#pragma unroll
  for (int e = VEC - 2; e >= 0; e -= 2) {
    const float xa = elem<T>(v, e), xb = elem<T>(v, e + 1);
    float fa, fb, ta, tb, ya, yb;
    if (CL == 2)
      quotient_rn2(fminf(fmaxf(xa, -xlim), xlim), fminf(fmaxf(xb, -xlim), xlim), p.rcp, ns, fa,
                   fb);
    else
      quotient_rn2(xa, xb, p.rcp, ns, fa, fb);
    add2(fa, fb, kRintMagic, kRintMagic, ta, tb);
    if (AFFINE || CL >= 1) {
      // M + clamp(f) = clamp(M + f) to [M + klo, M + khi], all exact integers
      ta = fminf(fmaxf(ta, kloM), khiM);
      tb = fminf(fmaxf(tb, kloM), khiM);
    }
    sub2(ta, tb, kRintMagic, kRintMagic, fa, fb);
    mul2(fa, fb, p.s, p.s, ya, yb);
    ov.set2(e, ya, yb);
    int qa = (int)(__float_as_uint(ta) - kRintMagicBits) + (AFFINE ? p.zp : 0);
    int qb = (int)(__float_as_uint(tb) - kRintMagicBits) + (AFFINE ? p.zp : 0);
    if (!FULL) {
      if (e >= cnt) qa = 0;
      if (e + 1 >= cnt) qb = 0;
    }
    cv.set2(e, qa, qb);
    uint32_t oa, ob;
    if (AFFINE) {
      // out of the window when one difference is negative (both cannot be:
      // wlo <= whi); a product keeps the sign of the pair even when it rounds
      // to zero or overflows, so its sign bit is the test
      float ha, hb, la, lb, pa, pb;
      sub2(p.whi, p.whi, xa, xb, ha, hb);
      sub2(xa, xb, wlo, wlo, la, lb);
      mul2(ha, hb, la, lb, pa, pb);
      oa = __float_as_uint(pa);
      ob = __float_as_uint(pb);
    } else {
      oa = __float_as_uint(__fsub_rn(p.whi, fabsf(xa)));
      ob = __float_as_uint(__fsub_rn(p.whi, fabsf(xb)));
    }
    out = __funnelshift_l(ob, out, 1);
    out = __funnelshift_l(oa, out, 1);
  }
  mb = ~out & (VEC == 32 ? 0xffffffffu : ((1u << VEC) - 1u));
}

// ---------------------------------------------------------------------------
// stochastic rounding (optirs-gpu quantization.rs, RoundingMode::Stochastic:
// floor(r) + 1 when the draw u < r - floor(r), floor(r) otherwise)
//
// The draw of element i of a call: word i % 4 of Philox-4x32-10 (J. Salmon,
// M. Moraes, R. Dror, D. Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC 2011) with key (low, high word of the seed) and counter (low, high word
// of offset + i / 4, 0, 0); u = (w >> 9) * 2^-23.  r - floor(r) and u are
// exact in binary32, so the decision is exact.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint64_t ctr, const uint32_t (&rk)[2 * kPhiloxRounds]) {
  uint32_t x0 = (uint32_t)ctr, x1 = (uint32_t)(ctr >> 32), x2 = 0u, x3 = 0u;
#pragma unroll
  for (int round = 0; round < kPhiloxRounds; ++round) {
    const uint32_t k0 = rk[2 * round], k1 = rk[2 * round + 1];  // the round's key (Weyl schedule)
    // the Philox S-box: 32 x 32 -> 64-bit products by the two round
    // multipliers, high halves mixed with the other words and the round key
    const uint64_t p0 = (uint64_t)0xD2511F53u * x0;  // one 32 x 32 -> 64-bit multiply each
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * x2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ x1 ^ k0, n2 = hi0 ^ x3 ^ k1;
    x0 = n0;
    x1 = lo1;
    x2 = n2;
    x3 = lo0;
  }
  return make_uint4(x0, x1, x2, x3);
}

// draws of the four elements 4 g .. 4 g + 3 (g = element index / 4)
__device__ __forceinline__ void sr_draws4(const SrCtx& sr, int64_t g, float (&u)[4]) {
  const uint4 w = philox4x32_10(sr.offset + (uint64_t)g, sr.rk);
  // (w >> 9) * 2^-23 exactly: 1 + (w >> 9) 2^-23 has those bits, minus 1
  u[0] = __uint_as_float(0x3f800000u | (w.x >> 9)) - 1.0f;
  u[1] = __uint_as_float(0x3f800000u | (w.y >> 9)) - 1.0f;
  u[2] = __uint_as_float(0x3f800000u | (w.z >> 9)) - 1.0f;
  u[3] = __uint_as_float(0x3f800000u | (w.w >> 9)) - 1.0f;
}

// the stochastic rounding of r with draw u (NaN stays NaN; for +-inf the
// fraction is NaN, no increment, and r is returned)
__device__ __forceinline__ float sr_round(float r, float u) {
  const float lower = floorf(r);
  const float frac = __fsub_rn(r, lower);  // exact
  return (u < frac) ? __fadd_rn(lower, 1.0f) : lower;
}

// One vector of a calibrated unit with p.fast set, stochastic rounding: the
// quotient is the exact RN(x/s) (quotient_rn2), k = sr_round(q, u) clamped to
// the code range (a value just above qmax - zp can round up past it), y = k s,
// the window as in int_vec_cal.  base: element index of element 0 (a
// multiple of 4).  GUARD (p.fast == 3): the quotient of x clamped to
// [-2^24 s, 2^24 s], as int_vec_cal with CL == 2.
template <typename T, int BITS, bool AFFINE, bool FULL, bool GUARD = false>
__device__ __forceinline__ void int_vec_cal_sr(const V32& v, const IntParams& p, int cnt,
                                               const SrCtx& sr, int64_t base, OutVec<T>& ov,
                                               CodeVec<BITS, T::VEC>& cv, uint32_t& mb) {
  constexpr int VEC = T::VEC;
  const float ns = -p.s;
  const float wlo = p.wlo == 0.0f ? -0.0f : p.wlo;
  const float xlim = GUARD ? __fmul_rn(p.s, 0x1p24f) : 0.0f;
  cv.clear();
  uint32_t out = 0u;
#pragma unroll
  for (int g = VEC / 4 - 1; g >= 0; --g) {
    float u[4];
    sr_draws4(sr, base / 4 + g, u);
#pragma unroll
    for (int h = 1; h >= 0; --h) {
      const int e = 4 * g + 2 * h;
      const float xa = elem<T>(v, e), xb = elem<T>(v, e + 1);
      float qa, qb, ta, tb, ya, yb;
      if (GUARD)
        quotient_rn2(fminf(fmaxf(xa, -xlim), xlim), fminf(fmaxf(xb, -xlim), xlim), p.rcp, ns, qa,
                     qb);
      else
        quotient_rn2(xa, xb, p.rcp, ns, qa, qb);
      float fa = fminf(fmaxf(sr_round(qa, u[2 * h]), p.klof), p.khif);
      float fb = fminf(fmaxf(sr_round(qb, u[2 * h + 1]), p.klof), p.khif);
      add2(fa, fb, kRintMagic, kRintMagic, ta, tb);
      mul2(fa, fb, p.s, p.s, ya, yb);
      ov.set2(e, ya, yb);
      int qa_ = (int)(__float_as_uint(ta) - kRintMagicBits) + (AFFINE ? p.zp : 0);
      int qb_ = (int)(__float_as_uint(tb) - kRintMagicBits) + (AFFINE ? p.zp : 0);
      if (!FULL) {
        if (e >= cnt) qa_ = 0;
        if (e + 1 >= cnt) qb_ = 0;
      }
      cv.set2(e, qa_, qb_);
      uint32_t oa, ob;
      if (AFFINE) {
        // out of the window when one difference is negative (both cannot be:
        // wlo <= whi); a product keeps the sign of the pair even when it rounds
        // to zero or overflows, so its sign bit is the test
        float ha, hb, la, lb, pa, pb;
        sub2(p.whi, p.whi, xa, xb, ha, hb);
        sub2(xa, xb, wlo, wlo, la, lb);
        mul2(ha, hb, la, lb, pa, pb);
        oa = __float_as_uint(pa);
        ob = __float_as_uint(pb);
      } else {
        oa = __float_as_uint(__fsub_rn(p.whi, fabsf(xa)));
        ob = __float_as_uint(__fsub_rn(p.whi, fabsf(xb)));
      }
      out = __funnelshift_l(ob, out, 1);
      out = __funnelshift_l(oa, out, 1);
    }
  }
  mb = ~out & (VEC == 32 ? 0xffffffffu : ((1u << VEC) - 1u));
}

// One element with the IEEE quotient and stochastic rounding (given
// parameters, or a calibrated scale outside the reciprocal's safe range):
// k = clamp(sr_round(x / s, u)), a NaN quotient gives code 0 (NAN_TO_ZERO,
// given parameters; a calibrated unit with a NaN is dead).
template <bool NAN_TO_ZERO>
__device__ __forceinline__ void int_elem_sr(float x, float u, const IntParams& p, int& q, float& y,
                                            uint32_t& m) {
  const float r = __fdiv_rn(x, p.s);
  float kf = fminf(fmaxf(sr_round(r, u), p.klof), p.khif);  // fminf/fmaxf drop a NaN r
  int k = (int)kf;
  if (NAN_TO_ZERO && isnan(r)) k = -p.zp;
  q = k + p.zp;
  y = __fmul_rn(__int2float_rn(k), p.s);
  m = (x >= p.wlo) && (x <= p.whi);
}

// Element map of one full vector with calibrated or given parameters: the
// reciprocal path when p.fast is 1 or 2, the IEEE path otherwise (a unit whose
// quotients may overflow, p.fast == 3, is rare: an extreme outlier against a
// clipped range), zeros for a dead unit.
// SR: stochastic rounding with the draws of elements base .. base + VEC - 1.
// OPT = false: the unit comes from the plain calibration (p.fast is 0 or 1).
template <typename T, int BITS, bool AFFINE, bool SR = false, bool OPT = true>
__device__ __forceinline__ void int_map_vec(const V32& v, const IntParams& p, OutVec<T>& ov,
                                            CodeVec<BITS, T::VEC>& cv, uint32_t& mb,
                                            const SrCtx& sr = SrCtx{}, int64_t base = 0) {
  constexpr int VEC = T::VEC;
  cv.clear();
  mb = 0u;
  if (p.fast && (!OPT || p.fast != 3)) {
    if (SR)
      int_vec_cal_sr<T, BITS, AFFINE, true>(v, p, VEC, sr, base, ov, cv, mb);
    else if (OPT && !AFFINE && p.fast == 2)
      int_vec_cal<T, BITS, AFFINE, true, 1>(v, p, VEC, ov, cv, mb);
    else
      int_vec_cal<T, BITS, AFFINE, true>(v, p, VEC, ov, cv, mb);
  } else if (!p.dead) {
#pragma unroll
    for (int g = 0; g < VEC / 4; ++g) {
      float u[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (SR) sr_draws4(sr, base / 4 + g, u);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = 4 * g + c;
        int q;
        float yv;
        uint32_t m;
        if (SR)
          int_elem_sr<false>(elem<T>(v, e), u[c], p, q, yv, m);
        else
          int_elem<false>(elem<T>(v, e), p, q, yv, m);
        ov.set(e, yv);
        cv.set(e, q);
        mb |= m << e;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) ov.set(e, 0.0f);
  }
}

// Programmatic dependent launch: pdl_wait() returns once the previous kernel
// of the stream has completed and its writes are visible (at once for an
// ordinary launch); pdl_trigger() lets the next kernel, if it was launched with
// the attribute, be scheduled while this one finishes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// the 128-byte line at p into L2 (no registers held)
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// each lane of the warp prefetches one 128-byte line of a 1024-element tile
template <typename T>
__device__ __forceinline__ void prefetch_tile_l2(const void* x, int64_t n, int64_t tile, int lane) {
  const int64_t e = tile * kTile + (int64_t)lane * (128 / T::BYTES);
  if (e < n) prefetch_l2(static_cast<const char*>(x) + e * T::BYTES);
}

__device__ __forceinline__ void flag_or(int32_t* flags, int bits) {
  if (flags && bits) atomicOr(flags, bits);
}

// Warp-aggregated flag update: one atomic per warp.
__device__ __forceinline__ void warp_flag_or(int32_t* flags, int bits) {
  int all = __reduce_or_sync(kFull, bits);
  if (flags && all && (threadIdx.x & 31) == 0) atomicOr(flags, all);
}

// Read the cross-CTA partials written by the per-tensor statistics kernel
// and reduce them (every thread of the block gets the result).
template <int MM>
__device__ __forceinline__ Stats reduce_partials(const uint4* part, int nparts, uint32_t* red) {
  Stats s;
  s.init<MM>();
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
    Stats o;
    o.unpack(part[i]);
    s.merge<MM>(o);
  }
  return block_reduce_stats<MM>(s, red);
}

}  // namespace qat
