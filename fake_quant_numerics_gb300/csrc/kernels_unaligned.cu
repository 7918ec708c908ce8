// kernels_unaligned.cu -- the hot-path calls on tensors whose x, y, grad or
// grad_in are aligned to their element but not to the 32-byte vectors the
// main kernels move (a view such as x[1:] of a contiguous tensor).
//
// Same arithmetic as the main kernels, one element per lane: lane l of a warp
// takes element 32 w + l of the warp's 32-element run, so every load and store
// is still one coalesced warp access, a run is exactly one mask word (a warp
// ballot), int8 codes are byte stores and int4 codes pair a lane with its odd
// neighbour (element 2j in the high nibble).  Scales come from the same
// calibrate() / given_params() and the elements take the division path
// (int_elem, the IEEE quotient), so the results equal the aligned kernels'.
//   k_ua_stats:    per-tensor statistics, one partial per block;
//   k_ua_int_map:  integer fake quant with one parameter set (calibrated from
//                  the partials in every block, or given) or per-unit arrays
//                  (rows, groups: calibrated by k_unit_generic);
//   k_ua_fp8_map:  per-tensor FP8 fake quant (IEEE quotient, saturating cast);
//   k_ua_ste:      the STE backward.
// Stochastic rounding: element i draws word i % 4 of the Philox block of
// counter offset + i / 4, computed by each lane for its own element.
#include <cuda_fp16.h>

#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

constexpr int kUaThreads = 256;

// element i of a tensor, widened to fp32 bits (scalar; any element alignment)
template <typename T>
__device__ __forceinline__ float ua_load(const void* x, int64_t i) {
  return __uint_as_float(load_elem_bits<T>(x, i));
}
template <typename T>
__device__ __forceinline__ void ua_store(void* y, int64_t i, float v) {
  if (T::BYTES == 4) {
    static_cast<float*>(y)[i] = v;
  } else {
    static_cast<uint16_t*>(y)[i] = (uint16_t)(pack_bf16x2(v, 0.0f) & 0xffffu);  // RNE, as the vector kernels
  }
}
// canonical quiet NaN of the output type
template <typename T>
__device__ __forceinline__ void ua_store_nan(void* y, int64_t i) {
  if (T::BYTES == 4)
    static_cast<uint32_t*>(y)[i] = 0x7fc00000u;
  else
    static_cast<uint16_t*>(y)[i] = 0x7fc0u;
}

__device__ __forceinline__ float ua_draw(const SrCtx& sr, int64_t i) {
  float u[4];
  sr_draws4(sr, i / 4, u);
  const int k = (int)(i & 3);
  return k == 0 ? u[0] : (k == 1 ? u[1] : (k == 2 ? u[2] : u[3]));
}

// codes of one warp run: int8 one byte per lane; int4 lanes 2j and 2j + 1
// share byte j (even element high); absent lanes hold code 0
template <int BITS>
__device__ __forceinline__ void ua_store_code(void* codes, int64_t i, int q, bool present,
                                              int lane) {
  if (BITS == 8) {
    if (present) static_cast<int8_t*>(codes)[i] = (int8_t)q;
  } else {
    const int lo = __shfl_down_sync(kFull, q, 1);
    if (present && (lane & 1) == 0)
      static_cast<uint8_t*>(codes)[i >> 1] = (uint8_t)(((q & 0xf) << 4) | (lo & 0xf));
  }
}

// ---------------------------------------------------------------------------
template <typename T, int MM>
__global__ void __launch_bounds__(kUaThreads) k_ua_stats(const void* __restrict__ x, int64_t n,
                                                         uint4* __restrict__ part) {
  __shared__ __align__(16) uint32_t red[4 * (kUaThreads / 32)];
  Stats st;
  st.init<MM>();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    st.add<MM>(load_elem_bits<T>(x, i));
  const Stats b = block_reduce_stats<MM>(st, red);
  if (threadIdx.x == 0) part[blockIdx.x] = b.pack();
}

// MODE 0: one parameter set calibrated from the nparts partials; MODE 1: one
// given parameter set (scale[0], zp[0]); MODE 2: per-unit arrays (unit = i / L)
// calibrated earlier (dead[u] marks a failed unit); MODE 3: per-unit given.
template <typename T, int BITS, bool AFFINE, int MODE, bool SR>
__global__ void __launch_bounds__(kUaThreads)
    k_ua_int_map(const void* __restrict__ x, int64_t n, int64_t L, const uint4* __restrict__ part,
                 int nparts, float* scale, int32_t* zp, const uint8_t* __restrict__ dead, SrCtx sr,
                 CalOpts co, void* y, void* codes, uint32_t* mask, int32_t* flags) {
  constexpr int qmin = QRange<BITS, AFFINE>::qmin, qmax = QRange<BITS, AFFINE>::qmax;
  constexpr int MM = AFFINE ? kMMFloat : kMMNone;
  __shared__ __align__(16) uint32_t red[4 * (kUaThreads / 32)];
  __shared__ IntParams sp;
  if (MODE == 0) {
    const Stats s = reduce_partials<MM>(part, nparts, red);
    if (threadIdx.x == 0) {
      IntParams q;
      const int f = calibrate<BITS, AFFINE, MM>(s, q, co);
      q.fast = 0;  // the division path, as for given parameters
      sp = q;
      if (blockIdx.x == 0) {
        scale[0] = q.s;
        if (zp) zp[0] = q.zp;
        flag_or(flags, f);
      }
    }
  } else if (MODE == 1) {
    if (threadIdx.x == 0) {
      const int f = given_params<BITS, AFFINE>(scale[0], zp ? zp[0] : 0, sp);
      if (blockIdx.x == 0) flag_or(flags, f);
    }
  }
  if (MODE <= 1) __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t runs = (n + 31) / 32;
  int fl = 0;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < runs;
       r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t i = r * 32 + lane;
    const bool present = i < n;
    IntParams p;
    if (MODE <= 1) {
      p = sp;
    } else {
      const int64_t u = present ? i / L : 0;
      if (MODE == 3) {
        fl |= present ? given_params<BITS, AFFINE>(scale[u], zp ? zp[u] : 0, p) : 0;
      } else {
        p.s = scale[u];
        p.zp = AFFINE ? zp[u] : 0;
        p.dead = dead[u];
        p.fast = 0;
        finish_params(p, qmin, qmax);
      }
    }
    int q = 0;
    float yv = 0.0f;
    uint32_t m = 0u;
    if (present && !p.dead) {
      const float xv = ua_load<T>(x, i);
      if (SR)
        int_elem_sr<(MODE & 1) != 0>(xv, ua_draw(sr, i), p, q, yv, m);
      else
        int_elem<(MODE & 1) != 0>(xv, p, q, yv, m);
    }
    if (present && y) ua_store<T>(y, i, yv);
    if (codes) ua_store_code<BITS>(codes, i, q, present, lane);
    const uint32_t w = __ballot_sync(kFull, m != 0u);
    if (mask && lane == 0) mask[r] = w;
  }
  if (MODE == 3) warp_flag_or(flags, fl);
}

// FP8: t = x / s (IEEE), the saturating cast, y = c s; NaN stays NaN (code
// 0x7F); s == 0 gives code 0 and y = +0; an invalid given s gives zeros and
// mask 0; mask = |x| <= fmt_max s.
template <int FMT>
__device__ __forceinline__ uint32_t ua_fp8_encode(float t) {
  uint16_t r;
  if (FMT == QAT_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  return r & 0xffu;
}
template <int FMT>
__device__ __forceinline__ float ua_fp8_decode(uint32_t c) {
  uint32_t h2;
  const uint16_t c16 = (uint16_t)c;
  if (FMT == QAT_E4M3)
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  else
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(c16));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}
// the stochastic magnitude rule on the grid of the format (as the aligned
// kernels: floor(log2 a) from the exponent field, ulp 2^(max(e, emin) - mbits),
// a / ulp rounded by the draw, saturated)
template <int FMT>
__device__ __forceinline__ float ua_fp8_sr_value(float t, float u) {
  constexpr int MB = FMT == QAT_E4M3 ? 3 : 2, EMIN = FMT == QAT_E4M3 ? -6 : -14;
  constexpr float kMaxF = FMT == QAT_E4M3 ? 448.0f : 57344.0f;
  const float a = fabsf(t);
  const int e = (int)(__float_as_uint(a) >> 23) - 127;
  const int se = (e > EMIN ? e : EMIN) - MB;
  const float inv = __uint_as_float((uint32_t)(127 - se) << 23);
  const float step = __uint_as_float((uint32_t)(127 + se) << 23);
  const float k = sr_round(__fmul_rn(a, inv), u);
  return copysignf(fminf(__fmul_rn(k, step), kMaxF), t);
}

template <typename T, int FMT, bool GIVEN, bool SR>
__global__ void __launch_bounds__(kUaThreads)
    k_ua_fp8_map(const void* __restrict__ x, int64_t n, const uint4* __restrict__ part, int nparts,
                 float* scale, SrCtx sr, void* y, uint8_t* codes, uint32_t* mask, int32_t* flags) {
  constexpr float kMaxF = FMT == QAT_E4M3 ? 448.0f : 57344.0f;
  __shared__ __align__(16) uint32_t red[4 * (kUaThreads / 32)];
  __shared__ float s_sh;
  __shared__ int mode_sh;
  if (!GIVEN) {
    const Stats s = reduce_partials<kMMNone>(part, nparts, red);
    if (threadIdx.x == 0) {
      const float sc = __fdiv_rn(s.absmax_f(), kMaxF);
      s_sh = sc;
      mode_sh = sc == 0.0f ? 1 : 0;
      if (blockIdx.x == 0) {
        scale[0] = sc;
        flag_or(flags, s.has_nonfinite() ? QAT_FLAG_NONFINITE_INPUT : 0);
      }
    }
  } else if (threadIdx.x == 0) {
    const float sc = scale[0];
    s_sh = sc;
    const bool bad = isnan(sc) || isinf(sc) || sc < 0.0f;
    mode_sh = bad ? 2 : (sc == 0.0f ? 1 : 0);
    if (blockIdx.x == 0 && bad) flag_or(flags, QAT_FLAG_BAD_PARAMS);
  }
  __syncthreads();
  const float s = s_sh;
  const int mode = mode_sh;
  const float lim = __fmul_rn(kMaxF, s);
  const int lane = threadIdx.x & 31;
  const int64_t runs = (n + 31) / 32;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < runs;
       r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t i = r * 32 + lane;
    const bool present = i < n;
    uint32_t m = 0u;
    if (present) {
      const float xv = ua_load<T>(x, i);
      const bool nan = isnan(xv);
      uint32_t c = 0u;
      float yv = 0.0f;
      if (mode == 0) {
        const float t = __fdiv_rn(xv, s);
        const float g = SR ? ua_fp8_sr_value<FMT>(t, ua_draw(sr, i)) : t;
        c = ua_fp8_encode<FMT>(g);
        yv = __fmul_rn(ua_fp8_decode<FMT>(c), s);
      }
      if (mode != 2) {
        if (nan) c = 0x7fu;
        m = fabsf(xv) <= lim ? 1u : 0u;
      }
      if (y) {
        if (mode != 2 && nan)
          ua_store_nan<T>(y, i);
        else
          ua_store<T>(y, i, yv);
      }
      if (codes) codes[i] = (uint8_t)c;
    }
    const uint32_t w = __ballot_sync(kFull, m != 0u);
    if (mask && lane == 0) mask[r] = w;
  }
}

// dx = mask bit ? g : +0 (bit copy of g)
template <typename T>
__global__ void __launch_bounds__(kUaThreads)
    k_ua_ste(const void* __restrict__ g, int64_t n, const uint32_t* __restrict__ mask,
             void* __restrict__ dx) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool keep = (mask[i >> 5] >> (i & 31)) & 1u;
    if (T::BYTES == 4)
      static_cast<uint32_t*>(dx)[i] = keep ? static_cast<const uint32_t*>(g)[i] : 0u;
    else
      static_cast<uint16_t*>(dx)[i] = keep ? static_cast<const uint16_t*>(g)[i] : (uint16_t)0;
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int ua_grid(int64_t n) {
  const int64_t g = (n + kUaThreads - 1) / kUaThreads;
  const int64_t cap = (int64_t)device_info().sms * 8;
  return (int)(g > cap ? cap : (g < 1 ? 1 : g));
}

qat_status launch_ua_stats(qat_dtype dt, int mm, const void* x, int64_t n, void* ws, int grid,
                           cudaStream_t s) {
  uint4* part = static_cast<uint4*>(ws);
#define QAT_US(T, M) k_ua_stats<T, M><<<grid, kUaThreads, 0, s>>>(x, n, part)
  if (dt == QAT_F32) {
    if (mm == kMMKeys) QAT_US(F32, kMMKeys); else if (mm == kMMFloat) QAT_US(F32, kMMFloat); else QAT_US(F32, kMMNone);
  } else {
    if (mm == kMMKeys) QAT_US(BF16, kMMKeys); else if (mm == kMMFloat) QAT_US(BF16, kMMFloat); else QAT_US(BF16, kMMNone);
  }
#undef QAT_US
  count_launch(1);
  return launch_status();
}

template <typename T, int BITS, bool AFFINE, int MODE>
static void ua_int_t(bool stoch, const void* x, int64_t n, int64_t L, const void* ws, int nparts,
                     float* scale, int32_t* zp, const uint8_t* dead, const SrCtx& sr,
                     const CalOpts& co, void* y, void* codes, uint32_t* mask, int32_t* flags,
                     cudaStream_t s) {
  const int grid = ua_grid(n);
  const uint4* part = static_cast<const uint4*>(ws);
  if (stoch)
    k_ua_int_map<T, BITS, AFFINE, MODE, true><<<grid, kUaThreads, 0, s>>>(
        x, n, L, part, nparts, scale, zp, dead, sr, co, y, codes, mask, flags);
  else
    k_ua_int_map<T, BITS, AFFINE, MODE, false><<<grid, kUaThreads, 0, s>>>(
        x, n, L, part, nparts, scale, zp, dead, sr, co, y, codes, mask, flags);
}

qat_status launch_ua_int_map(qat_dtype dt, int bits, bool affine, int mode, bool stoch,
                             const void* x, int64_t n, int64_t L, const void* ws, int nparts,
                             float* scale, int32_t* zp, const uint8_t* dead, const SrCtx& sr,
                             const CalOpts& co, void* y, void* codes, uint32_t* mask,
                             int32_t* flags, cudaStream_t s) {
#define QAT_UM(T, B, A)                                                                        \
  do {                                                                                         \
    if (mode == 0) ua_int_t<T, B, A, 0>(stoch, x, n, L, ws, nparts, scale, zp, dead, sr, co, y, codes, mask, flags, s); \
    else if (mode == 1) ua_int_t<T, B, A, 1>(stoch, x, n, L, ws, nparts, scale, zp, dead, sr, co, y, codes, mask, flags, s); \
    else if (mode == 2) ua_int_t<T, B, A, 2>(stoch, x, n, L, ws, nparts, scale, zp, dead, sr, co, y, codes, mask, flags, s); \
    else ua_int_t<T, B, A, 3>(stoch, x, n, L, ws, nparts, scale, zp, dead, sr, co, y, codes, mask, flags, s); \
  } while (0)
  if (dt == QAT_F32) {
    if (bits == 8) { if (affine) QAT_UM(F32, 8, true); else QAT_UM(F32, 8, false); }
    else { if (affine) QAT_UM(F32, 4, true); else QAT_UM(F32, 4, false); }
  } else {
    if (bits == 8) { if (affine) QAT_UM(BF16, 8, true); else QAT_UM(BF16, 8, false); }
    else { if (affine) QAT_UM(BF16, 4, true); else QAT_UM(BF16, 4, false); }
  }
#undef QAT_UM
  count_launch(1);
  return launch_status();
}

template <typename T, int FMT>
static void ua_fp8_t(bool given, bool stoch, const void* x, int64_t n, const void* ws, int nparts,
                     float* scale, const SrCtx& sr, void* y, uint8_t* codes, uint32_t* mask,
                     int32_t* flags, cudaStream_t s) {
  const int grid = ua_grid(n);
  const uint4* part = static_cast<const uint4*>(ws);
#define QAT_UF(G, S) \
  k_ua_fp8_map<T, FMT, G, S><<<grid, kUaThreads, 0, s>>>(x, n, part, nparts, scale, sr, y, codes, mask, flags)
  if (given) { if (stoch) QAT_UF(true, true); else QAT_UF(true, false); }
  else { if (stoch) QAT_UF(false, true); else QAT_UF(false, false); }
#undef QAT_UF
}

qat_status launch_ua_fp8_map(qat_dtype dt, int fmt, bool given, bool stoch, const void* x,
                             int64_t n, const void* ws, int nparts, float* scale, const SrCtx& sr,
                             void* y, uint8_t* codes, uint32_t* mask, int32_t* flags,
                             cudaStream_t s) {
  if (dt == QAT_F32) {
    if (fmt == QAT_E4M3) ua_fp8_t<F32, QAT_E4M3>(given, stoch, x, n, ws, nparts, scale, sr, y, codes, mask, flags, s);
    else ua_fp8_t<F32, QAT_E5M2>(given, stoch, x, n, ws, nparts, scale, sr, y, codes, mask, flags, s);
  } else {
    if (fmt == QAT_E4M3) ua_fp8_t<BF16, QAT_E4M3>(given, stoch, x, n, ws, nparts, scale, sr, y, codes, mask, flags, s);
    else ua_fp8_t<BF16, QAT_E5M2>(given, stoch, x, n, ws, nparts, scale, sr, y, codes, mask, flags, s);
  }
  count_launch(1);
  return launch_status();
}

qat_status launch_ua_ste(qat_dtype dt, const void* g, int64_t n, const uint32_t* mask, void* dx,
                         cudaStream_t s) {
  const int grid = ua_grid(n);
  if (dt == QAT_F32)
    k_ua_ste<F32><<<grid, kUaThreads, 0, s>>>(g, n, mask, dx);
  else
    k_ua_ste<BF16><<<grid, kUaThreads, 0, s>>>(g, n, mask, dx);
  count_launch(1);
  return launch_status();
}

}  // namespace qat
