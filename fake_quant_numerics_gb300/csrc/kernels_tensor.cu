// kernels_tensor.cu -- per-tensor statistics, integer fake quant with one
// parameter set or per-unit parameter arrays, and the warp-per-unit fallback.
//
// Integer fake quant (optirs-gpu quantization.rs, module docs "Integer
// quantization", QuantParams::quantize / dequantize / real_min / real_max,
// fake_quant_int, fake_quant_int_per_channel, fake_quant_backward):
//   q = clamp(rne(x / scale) + zp, qmin, qmax), y = (q - zp) * scale,
//   mask = x in [(qmin - zp) * scale, (qmax - zp) * scale].
// Per-tensor calibration needs the whole tensor's statistics before the first
// element is quantized, so it is two passes: k_stats_tensor writes one
// partial per block, k_int_tensor re-reduces the partials in every block (an
// exact, order-free max/min) and streams the tensor a second time, in reverse
// tile order so the tail of the first pass is still in L2.
#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

#if !QAT_SR
// ---------------------------------------------------------------------------
// per-tensor statistics: one uint4 partial (Stats::pack) per block
// ---------------------------------------------------------------------------
template <typename T, int MM, bool FULL>
__device__ __forceinline__ void stats_tile(const void* __restrict__ x, int64_t n, int64_t tile,
                                           V32 (&v)[kTile / (32 * T::VEC)], bool have,
                                           int64_t next, Stats& st, int lane) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC);
  int cnt[SLOTS];
  tile_load<T, FULL>(x, n, tile, v, cnt, have, lane);
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) {
    if (MM == kMMNone) {
      st.add_absmax<T>(v[j]);  // absent tail elements read +0
    } else if (FULL) {
      stats_add_vec<T, MM>(st, v[j]);
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        if (e < cnt[j]) st.add<MM>(elem_bits<T>(v[j], e));
    }
    slot_prefetch<T>(x, next, j, v[j], lane);
  }
}

template <typename T, int MM>
__global__ void __launch_bounds__(512) k_stats_tensor(const void* __restrict__ x, int64_t n,
                                                      uint4* __restrict__ part) {
  __shared__ __align__(16) uint32_t red[4 * 16];
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t nfull = n / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  Stats st;
  st.init<MM>();
  V32 v[kTile / (32 * T::VEC)];
  bool have = false;
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < ntiles;
       t += wstride) {
    const int64_t next = -1;  // no rolling prefetch: occupancy matters more here
    if (t < nfull) stats_tile<T, MM, true>(x, n, t, v, have, next, st, lane);
    else stats_tile<T, MM, false>(x, n, t, v, have, next, st, lane);
    have = next >= 0;
  }
  pdl_trigger();  // the map may be scheduled as the blocks finish
  Stats b = block_reduce_stats<MM>(st, red);
  if (threadIdx.x == 0) part[blockIdx.x] = b.pack();
}

__global__ void __launch_bounds__(256) k_stats_finalize(const uint4* __restrict__ part, int nparts,
                                                        float* absmax, float* minv, float* maxv,
                                                        int32_t* flags) {
  __shared__ __align__(16) uint32_t red[4 * 8];
  Stats s = reduce_partials<kMMKeys>(part, nparts, red);
  if (threadIdx.x == 0) {
    if (absmax) absmax[0] = s.absmax_f();
    if (minv) minv[0] = s.min_f<kMMKeys>();
    if (maxv) maxv[0] = s.max_f<kMMKeys>();
    flag_or(flags, s.has_nonfinite() ? QAT_FLAG_NONFINITE_INPUT : 0);
  }
}

#endif  // !QAT_SR

// ---------------------------------------------------------------------------
// integer fake quant, one parameter set (calibrated from partials or given)
// ---------------------------------------------------------------------------
// OPT: the unit may come from a calibration with options (p.fast 2 or 3);
// without, only the plain reciprocal path is built, which keeps its registers.
template <typename T, int BITS, bool AFFINE, bool GIVEN, bool FULL, bool SR, bool OPT>
__device__ __forceinline__ void int_tile(const void* __restrict__ x, int64_t n, int64_t tile,
                                         V32 (&v)[kTile / (32 * T::VEC)], bool have, int64_t next,
                                         const IntParams& p, const SrCtx& sr,
                                         void* __restrict__ y, void* __restrict__ codes,
                                         uint32_t* __restrict__ mask, int lane) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC);
  const int64_t tb = tile * kTile;
  int cnt[SLOTS];
  tile_load<T, FULL>(x, n, tile, v, cnt, have, lane);
  uint32_t mw[SLOTS];
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) {
    int64_t base = tb + (int64_t)(j * 32 + lane) * VEC;
    OutVec<T> ov;
    CodeVec<BITS, VEC> cv;
    cv.clear();
    uint32_t mb = 0u;
    if (!GIVEN && p.fast) {
      if (SR) {
        if (OPT && p.fast == 3)
          int_vec_cal_sr<T, BITS, AFFINE, FULL, true>(v[j], p, cnt[j], sr, base, ov, cv, mb);
        else
          int_vec_cal_sr<T, BITS, AFFINE, FULL>(v[j], p, cnt[j], sr, base, ov, cv, mb);
      } else if (OPT && p.fast == 3) {
        int_vec_cal<T, BITS, AFFINE, FULL, 2>(v[j], p, cnt[j], ov, cv, mb);
      } else if (OPT && !AFFINE && p.fast == 2) {
        int_vec_cal<T, BITS, AFFINE, FULL, 1>(v[j], p, cnt[j], ov, cv, mb);
      } else {
        int_vec_cal<T, BITS, AFFINE, FULL>(v[j], p, cnt[j], ov, cv, mb);
      }
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
            int_elem_sr<GIVEN>(elem<T>(v[j], e), u[c], p, q, yv, m);
          else
            int_elem<GIVEN>(elem<T>(v[j], e), p, q, yv, m);
          ov.set(e, yv);
          if (FULL || e < cnt[j]) cv.set(e, q);
          mb |= m << e;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) ov.set(e, 0.0f);
    }
    slot_prefetch<T>(x, next, j, v[j], lane);
    if (!FULL) mb &= (cnt[j] >= 32) ? 0xffffffffu : ((1u << cnt[j]) - 1u);
    if (cnt[j] > 0) {
      if (y) store_vec<T>(y, base, ov.v, cnt[j]);
      if (codes) cv.store(codes, base, cnt[j]);
    }
    mw[j] = mask_word_of_slot<VEC>(mb, lane);
  }
  if (mask) {
    uint32_t w = gather_tile_word<VEC, SLOTS>(mw, lane);
    int64_t wi = tile * 32 + lane;
    if (FULL || wi < (n + 31) / 32) mask[wi] = w;
  }
}

template <typename T, int BITS, bool AFFINE, bool GIVEN, bool SR, bool OPT>
__global__ void __maxnreg__(SR ? 128 : 80) k_int_tensor(const void* __restrict__ x, int64_t n,
                                                    const uint4* __restrict__ part, int nparts,
                                                    float* scale, int32_t* zp, SrCtx sr,
                                                    CalOpts co, void* y, void* codes,
                                                    uint32_t* mask, int32_t* flags) {
  __shared__ __align__(16) uint32_t red[4 * 8];
  __shared__ IntParams sp;
  if (GIVEN) {
    if (threadIdx.x == 0) {
      int f = given_params<BITS, AFFINE>(scale[0], zp ? zp[0] : 0, sp);
      if (blockIdx.x == 0) flag_or(flags, f);
    }
  } else {
    constexpr int MM = AFFINE ? kMMFloat : kMMNone;
    // launched early (after the statistics pass): request the warp's first
    // tile into L2, then wait for the partials
    {
      const int64_t ntiles = (n + kTile - 1) / kTile;
      const int64_t t0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
      if (t0 < ntiles) prefetch_tile_l2<T>(x, n, ntiles - 1 - t0, threadIdx.x & 31);
    }
    pdl_wait();
    Stats st = reduce_partials<MM>(part, nparts, red);
    if (threadIdx.x == 0) {
      int f = calibrate<BITS, AFFINE, MM>(st, sp, OPT ? co : CalOpts{1.0f, 0, 0});
      if (blockIdx.x == 0) {
        scale[0] = sp.s;
        if (zp) zp[0] = sp.zp;
        flag_or(flags, f);
      }
    }
  }
  __syncthreads();
  const IntParams p = sp;
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t nfull = n / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  V32 v[kTile / (32 * T::VEC)];
  bool have = false;
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < ntiles;
       t += wstride) {
    // calibrated: reverse order, so the first tiles read are the ones the
    // statistics pass touched last (still in L2)
    const int64_t tile = GIVEN ? t : ntiles - 1 - t;
    const int64_t nt = t + wstride;
    const int64_t ntile = GIVEN ? nt : ntiles - 1 - nt;
    const int64_t next = (nt < ntiles && ntile < nfull) ? ntile : -1;
    if (tile < nfull)
      int_tile<T, BITS, AFFINE, GIVEN, true, SR, OPT>(x, n, tile, v, have, next, p, sr, y, codes,
                                                      mask, lane);
    else
      int_tile<T, BITS, AFFINE, GIVEN, false, SR, OPT>(x, n, tile, v, have, next, p, sr, y, codes,
                                                       mask, lane);
    have = next >= 0;
  }
}

// ---------------------------------------------------------------------------
// integer fake quant with per-unit parameter arrays, unit = element / L, or
// element % ucols for per-column units (ucols > 0): given per-row, per-group
// and per-column parameters, and the calibrated fallback for unit shapes the
// fused and column kernels do not cover
// ---------------------------------------------------------------------------
template <typename T, int BITS, bool AFFINE, bool GIVEN, bool SR>
__global__ void __maxnreg__(SR ? 128 : 80) k_int_units(const void* __restrict__ x, int64_t n, int64_t L,
                                                   int64_t ucols,
                                                   const float* __restrict__ scale,
                                                   const int32_t* __restrict__ zp,
                                                   const uint8_t* __restrict__ dead, SrCtx sr,
                                                   void* y, void* codes, uint32_t* mask,
                                                   int32_t* flags) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC);
  constexpr int qmin = QRange<BITS, AFFINE>::qmin, qmax = QRange<BITS, AFFINE>::qmax;
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t tile = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tile < ntiles;
       tile += wstride) {
    const int64_t tb = tile * kTile;
    uint32_t mw[SLOTS];
    int fl = 0;
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      int64_t base = tb + (int64_t)(j * 32 + lane) * VEC;
      int64_t c = n - base;
      int cnt = c >= VEC ? VEC : (c > 0 ? (int)c : 0);
      V32 v = load_vec<T>(x, cnt > 0 ? base : 0, cnt);
      OutVec<T> ov;
      CodeVec<BITS, VEC> cv;
      cv.clear();
      uint32_t mb = 0u;
      int64_t cur = -1;
      IntParams p;
      p.s = 1.0f;
      p.zp = 0;
      p.dead = 1;
      finish_params(p, qmin, qmax);
      float ud[VEC];  // stochastic-rounding draws of the vector's elements
#pragma unroll
      for (int g = 0; g < VEC / 4; ++g) {
        float w[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (SR) sr_draws4(sr, base / 4 + g, w);
#pragma unroll
        for (int c = 0; c < 4; ++c) ud[4 * g + c] = w[c];
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        int q = 0;
        float yv = 0.0f;
        uint32_t m = 0u;
        if (e < cnt) {
          int64_t u = ucols > 0 ? (base + e) % ucols : (base + e) / L;
          if (u != cur) {
            cur = u;
            if (GIVEN) {
              fl |= given_params<BITS, AFFINE>(scale[u], zp ? zp[u] : 0, p);
            } else {
              p.s = scale[u];
              p.zp = AFFINE ? zp[u] : 0;
              p.dead = dead[u];
              finish_params(p, qmin, qmax);
            }
          }
          if (!p.dead) {
            if (SR)
              int_elem_sr<GIVEN>(elem<T>(v, e), ud[e], p, q, yv, m);
            else
              int_elem<GIVEN>(elem<T>(v, e), p, q, yv, m);
          }
        }
        ov.set(e, yv);
        cv.set(e, q);
        mb |= m << e;
      }
      if (cnt > 0) {
        if (y) store_vec<T>(y, base, ov.v, cnt);
        if (codes) cv.store(codes, base, cnt);
      }
      mw[j] = mask_word_of_slot<VEC>(mb, lane);
    }
    if (mask) {
      uint32_t w = gather_tile_word<VEC, SLOTS>(mw, lane);
      int64_t wi = tile * 32 + lane;
      if (wi < (n + 31) / 32) mask[wi] = w;
    }
    warp_flag_or(flags, fl);
  }
}

#if !QAT_SR
// ---------------------------------------------------------------------------
// warp-per-unit statistics for any unit length (scalar loads)
//   MODE 0: absmax / minv / maxv per unit, QAT_FLAG_NONFINITE_INPUT
//   MODE 1: calibrated int params -> scale, zp, dead (per unit)
// ---------------------------------------------------------------------------
template <typename T, int MODE, int BITS, bool AFFINE>
__global__ void __launch_bounds__(256) k_unit_generic(const void* __restrict__ x, int64_t units,
                                                      int64_t L, float* absmax, float* minv,
                                                      float* maxv, float* scale, int32_t* zp,
                                                      uint8_t* dead, CalOpts co, int32_t* flags) {
  const int lane = threadIdx.x & 31;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units;
       u += wstride) {
    Stats st;
    st.init<kMMKeys>();
    const int64_t off = u * L;
    for (int64_t i = lane; i < L; i += 32) st.add<kMMKeys>(load_elem_bits<T>(x, off + i));
    st.reduce_lanes<kMMKeys>(32);
    if (lane == 0) {
      if (MODE == 0) {
        if (absmax) absmax[u] = st.absmax_f();
        if (minv) minv[u] = st.min_f<kMMKeys>();
        if (maxv) maxv[u] = st.max_f<kMMKeys>();
        flag_or(flags, st.has_nonfinite() ? QAT_FLAG_NONFINITE_INPUT : 0);
      } else {
        IntParams p;
        int f = calibrate<BITS, AFFINE, kMMKeys>(st, p, co);
        scale[u] = p.s;
        if (zp) zp[u] = p.zp;
        dead[u] = (uint8_t)p.dead;
        flag_or(flags, f);
      }
    }
  }
}

#endif  // !QAT_SR

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
#if !QAT_SR
int stats_grid(int64_t n) {
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t warps_per_block = 16;  // 512 threads
  int64_t g = (ntiles + warps_per_block - 1) / warps_per_block;
  int64_t cap = (int64_t)device_info().sms * 2;
  if (cap > kMaxPartials) cap = kMaxPartials;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

#endif  // !QAT_SR

static int map_grid(int64_t n, int per_sm) {
  const int64_t ntiles = (n + kTile - 1) / kTile;
  int64_t g = (ntiles + 7) / 8;  // 8 warps per 256-thread block
  int64_t cap = (int64_t)device_info().sms * per_sm;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

#if !QAT_SR
qat_status launch_stats_tensor(qat_dtype dt, const void* x, int64_t n, int mm, void* ws,
                               int grid, cudaStream_t s) {
  uint4* part = static_cast<uint4*>(ws);
#define QAT_ST(T, M) k_stats_tensor<T, M><<<grid, 512, 0, s>>>(x, n, part)
  if (dt == QAT_F32) {
    if (mm == kMMKeys) QAT_ST(F32, kMMKeys);
    else if (mm == kMMFloat) QAT_ST(F32, kMMFloat);
    else QAT_ST(F32, kMMNone);
  } else {
    if (mm == kMMKeys) QAT_ST(BF16, kMMKeys);
    else if (mm == kMMFloat) QAT_ST(BF16, kMMFloat);
    else QAT_ST(BF16, kMMNone);
  }
#undef QAT_ST
  count_launch(1);
  return launch_status();
}

qat_status launch_stats_finalize(const void* ws, int nparts, float* absmax, float* minv, float* maxv,
                                 int32_t* flags, cudaStream_t s) {
  k_stats_finalize<<<1, 256, 0, s>>>(static_cast<const uint4*>(ws), nparts, absmax, minv, maxv,
                                     flags);
  count_launch(1);
  return launch_status();
}

#endif  // !QAT_SR

template <typename T, int BITS, bool AFFINE>
static void int_tensor_t(bool given, const void* x, int64_t n, const void* ws, int nparts,
                         float* scale, int32_t* zp, const SrCtx& sr, const CalOpts& co, void* y,
                         void* codes, uint32_t* mask, int32_t* flags, cudaStream_t s, bool pdl) {
  const int grid = map_grid(n, 8);
  const uint4* part = static_cast<const uint4*>(ws);
  // calibration options as a compile-time switch (the plain build keeps its registers)
  const bool opt = co.clip != 1.0f || co.fp16 || co.clamp;
  if (given)
    k_int_tensor<T, BITS, AFFINE, true, QAT_SR, false>
        <<<grid, 256, 0, s>>>(x, n, part, nparts, scale, zp, sr, co, y, codes, mask, flags);
  else if (opt)
    launch_kernel(k_int_tensor<T, BITS, AFFINE, false, QAT_SR, true>, dim3(grid), dim3(256), 0, s,
                  pdl, x, n, part, nparts, scale, zp, sr, co, y, codes, mask, flags);
  else
    launch_kernel(k_int_tensor<T, BITS, AFFINE, false, QAT_SR, false>, dim3(grid), dim3(256), 0, s,
                  pdl, x, n, part, nparts, scale, zp, sr, co, y, codes, mask, flags);
}

qat_status QAT_SR_NAME(launch_int_tensor)(qat_dtype dt, int bits, bool affine, bool given,
                                          const void* x, int64_t n, const void* ws, int nparts,
                                          float* scale, int32_t* zp, const SrCtx& sr,
                                          const CalOpts& co, void* y, void* codes, uint32_t* mask,
                                          int32_t* flags, cudaStream_t s, bool pdl) {
#define QAT_IT(T, B, A) int_tensor_t<T, B, A>(given, x, n, ws, nparts, scale, zp, sr, co, y, codes, mask, flags, s, pdl)
  if (dt == QAT_F32) {
    if (bits == 8) { if (affine) QAT_IT(F32, 8, true); else QAT_IT(F32, 8, false); }
    else { if (affine) QAT_IT(F32, 4, true); else QAT_IT(F32, 4, false); }
  } else {
    if (bits == 8) { if (affine) QAT_IT(BF16, 8, true); else QAT_IT(BF16, 8, false); }
    else { if (affine) QAT_IT(BF16, 4, true); else QAT_IT(BF16, 4, false); }
  }
#undef QAT_IT
  count_launch(1);
  return launch_status();
}

template <typename T, int BITS, bool AFFINE>
static void int_units_t(bool given, const void* x, int64_t n, int64_t L, int64_t ucols,
                        const float* scale,
                        const int32_t* zp, const uint8_t* dead, const SrCtx& sr, void* y,
                        void* codes, uint32_t* mask, int32_t* flags, cudaStream_t s) {
  const int grid = map_grid(n, 8);
  if (given)
    k_int_units<T, BITS, AFFINE, true, QAT_SR>
        <<<grid, 256, 0, s>>>(x, n, L, ucols, scale, zp, dead, sr, y, codes, mask, flags);
  else
    k_int_units<T, BITS, AFFINE, false, QAT_SR>
        <<<grid, 256, 0, s>>>(x, n, L, ucols, scale, zp, dead, sr, y, codes, mask, flags);
}

qat_status QAT_SR_NAME(launch_int_units)(qat_dtype dt, int bits, bool affine, bool given,
                                         const void* x, int64_t n, int64_t L, int64_t ucols,
                                         const float* scale,
                                         const int32_t* zp, const uint8_t* dead, const SrCtx& sr,
                                         void* y, void* codes, uint32_t* mask, int32_t* flags,
                                         cudaStream_t s) {
#define QAT_IU(T, B, A) int_units_t<T, B, A>(given, x, n, L, ucols, scale, zp, dead, sr, y, codes, mask, flags, s)
  if (dt == QAT_F32) {
    if (bits == 8) { if (affine) QAT_IU(F32, 8, true); else QAT_IU(F32, 8, false); }
    else { if (affine) QAT_IU(F32, 4, true); else QAT_IU(F32, 4, false); }
  } else {
    if (bits == 8) { if (affine) QAT_IU(BF16, 8, true); else QAT_IU(BF16, 8, false); }
    else { if (affine) QAT_IU(BF16, 4, true); else QAT_IU(BF16, 4, false); }
  }
#undef QAT_IU
  count_launch(1);
  return launch_status();
}

#if !QAT_SR
template <typename T>
static void unit_generic_t(int mode, int bits, bool affine, const void* x, int64_t units, int64_t L,
                           float* absmax, float* minv, float* maxv, float* scale, int32_t* zp,
                           uint8_t* dead, const CalOpts& co, int32_t* flags, cudaStream_t s) {
  int64_t g = (units + 7) / 8;
  int64_t cap = (int64_t)device_info().sms * 8;
  int grid = (int)(g > cap ? cap : (g < 1 ? 1 : g));
#define QAT_UG(M, B, A) \
  k_unit_generic<T, M, B, A><<<grid, 256, 0, s>>>(x, units, L, absmax, minv, maxv, scale, zp, dead, co, flags)
  if (mode == 0) QAT_UG(0, 8, false);
  else if (bits == 8) { if (affine) QAT_UG(1, 8, true); else QAT_UG(1, 8, false); }
  else { if (affine) QAT_UG(1, 4, true); else QAT_UG(1, 4, false); }
#undef QAT_UG
}

qat_status launch_unit_generic(qat_dtype dt, int mode, int bits, bool affine, const void* x,
                               int64_t units, int64_t L, float* absmax, float* minv, float* maxv,
                               float* scale, int32_t* zp, uint8_t* dead, const CalOpts& co,
                               int32_t* flags, cudaStream_t s) {
  if (dt == QAT_F32)
    unit_generic_t<F32>(mode, bits, affine, x, units, L, absmax, minv, maxv, scale, zp, dead, co,
                        flags, s);
  else
    unit_generic_t<BF16>(mode, bits, affine, x, units, L, absmax, minv, maxv, scale, zp, dead, co,
                         flags, s);
  count_launch(1);
  return launch_status();
}

#endif  // !QAT_SR

}  // namespace qat
