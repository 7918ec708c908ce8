// kernels_fused.cu -- single-pass per-unit calibration + integer fake quant.
//
// A unit (one row, axis-0 channel of optirs-gpu quantization.rs
// per_channel_params; or one group of consecutive elements along the last
// dimension, cs349e 05_quantization_basics.py demo 3) is small enough to stay
// on chip, so its statistics and its quantization share one read of x:
//
//   k_int_groups: units of L = VEC * LPG elements (LPG = 2..32 lanes, a
//     power of two).  Each unit lives in LPG adjacent lanes of one warp tile;
//     its absmax / min / max is a shuffle reduction over those lanes.
//   k_int_rows:   units of L elements, L % 32 == 0, up to 256 * NV vectors.
//     One thread block per unit, statistics by a block reduction.
//
// Calibration follows QuantParams::from_absmax / from_minmax; the element map
// follows QuantParams::quantize / dequantize and the STE window of
// fake_quant_backward.  STATS_ONLY instantiations write the unit statistics
// (absmax, min, max) instead.
#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

// OPT: the calibration options apply (else the plain calibration, so that the
// plain kernel keeps the registers the options would take)
template <typename T, int BITS, bool AFFINE, int LPG, bool STATS_ONLY, bool FULL, bool SR, bool OPT>
__device__ __forceinline__ void group_tile(const void* __restrict__ x, int64_t n, int64_t tile,
                                           V32 (&v)[kTile / (32 * T::VEC)], bool have,
                                           int64_t next, float* scale, int32_t* zp, float* absmax,
                                           float* minv, float* maxv, const SrCtx& sr,
                                           const CalOpts& co, void* __restrict__ y,
                                           void* __restrict__ codes,
                                           uint32_t* __restrict__ mask, int lane, int& fl) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC);
  constexpr int L = VEC * LPG;
  constexpr int MM = STATS_ONLY ? kMMKeys : (AFFINE ? kMMFloat : kMMNone);
  const int64_t tb = tile * kTile;
  bool present[SLOTS];
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) {
    int64_t base = tb + (int64_t)(j * 32 + lane) * VEC;
    // n is a multiple of L, so a lane's vector is entirely present or absent
    present[j] = FULL || base < n;
    if (FULL) {
      if (!have) v[j] = ld_v32(static_cast<const char*>(x) + base * T::BYTES);
    } else if (present[j]) {
      v[j] = ld_v32(static_cast<const char*>(x) + base * T::BYTES);
    } else {
#pragma unroll
      for (int w = 0; w < 8; ++w) v[j].w[w] = 0u;
    }
  }
  uint32_t mw[SLOTS];
  // groups per slot and per tile; with at most 32 groups in a tile, lane i
  // calibrates group i once instead of every lane of every group
  constexpr int G = 32 / LPG, NG = SLOTS * G;
  if constexpr (!STATS_ONLY && NG <= 32) {
    Stats sj[SLOTS];
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      Stats& sr = sj[j];
      sr.init<MM>();
      if (present[j]) stats_add_vec<T, MM>(sr, v[j]);
      sr.reduce_lanes<MM>(LPG);
    }
    // group i lives in slot i / G on lanes (i % G) * LPG ...
    Stats g;
    g.init<MM>();
    const int src = (lane % G) * LPG;
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      Stats t;
      t.amax = __shfl_sync(kFull, sj[j].amax, src);
      t.nonfinite = __shfl_sync(kFull, sj[j].nonfinite, src);
      if (MM != kMMNone) {
        t.kmin = __shfl_sync(kFull, sj[j].kmin, src);
        t.kmax = __shfl_sync(kFull, sj[j].kmax, src);
      }
      if (lane / G == j) g = t;
    }
    IntParams q;
    const int f = calibrate<BITS, AFFINE, MM>(g, q, OPT ? co : CalOpts{1.0f, 0, 0});
    const int64_t ug = tb / L + lane;
    if (lane < NG && ug * L < n) {
      scale[ug] = q.s;
      if (zp) zp[ug] = q.zp;
      fl |= f;
    }
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      const int64_t base = tb + (int64_t)(j * 32 + lane) * VEC;
      const IntParams p = shfl_params<BITS, AFFINE>(q, j * G + lane / LPG);
      OutVec<T> ov;
      CodeVec<BITS, VEC> cv;
      uint32_t mb;
      int_map_vec<T, BITS, AFFINE, SR, OPT>(v[j], p, ov, cv, mb, sr, base);
      slot_prefetch<T>(x, next, j, v[j], lane);
      if (!present[j]) mb = 0u;
      if (present[j]) {
        if (y) st_v32(static_cast<char*>(y) + base * T::BYTES, ov.v);
        if (codes) cv.store(codes, base, VEC);
      }
      mw[j] = mask_word_of_slot<VEC>(mb, lane);
    }
  } else {
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      const int64_t base = tb + (int64_t)(j * 32 + lane) * VEC;
      const int64_t u = base / L;
      Stats st;
      st.init<MM>();
      if (present[j]) {
        stats_add_vec<T, MM>(st, v[j]);
      }
      st.reduce_lanes<MM>(LPG);
      const bool leader = present[j] && (lane % LPG) == 0;
      if (STATS_ONLY) {
        if (leader) {
          if (absmax) absmax[u] = st.absmax_f();
          if (minv) minv[u] = st.min_f<MM>();
          if (maxv) maxv[u] = st.max_f<MM>();
        }
        if (present[j] && st.has_nonfinite()) fl |= QAT_FLAG_NONFINITE_INPUT;
        mw[j] = 0u;
        slot_prefetch<T>(x, next, j, v[j], lane);
        continue;
      }
      IntParams p;
      int f = calibrate<BITS, AFFINE, MM>(st, p, OPT ? co : CalOpts{1.0f, 0, 0});
      if (leader) {
        scale[u] = p.s;
        if (zp) zp[u] = p.zp;
      }
      if (present[j]) fl |= f;
      OutVec<T> ov;
      CodeVec<BITS, VEC> cv;
      uint32_t mb;
      int_map_vec<T, BITS, AFFINE, SR, OPT>(v[j], p, ov, cv, mb, sr, base);
      slot_prefetch<T>(x, next, j, v[j], lane);
      if (!present[j]) mb = 0u;
      if (present[j]) {
        if (y) st_v32(static_cast<char*>(y) + base * T::BYTES, ov.v);
        if (codes) cv.store(codes, base, VEC);
      }
      mw[j] = mask_word_of_slot<VEC>(mb, lane);
    }
  }
  if (!STATS_ONLY && mask) {
    uint32_t w = gather_tile_word<VEC, SLOTS>(mw, lane);
    int64_t wi = tile * 32 + lane;
    if (FULL || wi < (n + 31) / 32) mask[wi] = w;
  }
}

// registers: bf16 nearest rounding 64 (four blocks of 256 per SM; 53.3 ->
// 49.4 us on the w4 weights against 80), stochastic rounding 80 (three),
// fp32 nearest rounding 96
template <typename T, int BITS, bool AFFINE, int LPG, bool STATS_ONLY, bool SR, bool OPT>
__global__ void __maxnreg__((T::BYTES == 4 && !SR) ? 96 : (SR ? 80 : 64))
    k_int_groups(const void* __restrict__ x, int64_t n, float* scale, int32_t* zp, float* absmax,
                 float* minv, float* maxv, SrCtx sr, CalOpts co, void* y, void* codes,
                 uint32_t* mask, int32_t* flags) {
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t nfull = n / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  int fl = 0;
  V32 v[kTile / (32 * T::VEC)];
  bool have = false;
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < ntiles;
       t += wstride) {
    const int64_t nt = t + wstride;
    // rolling prefetch of the next full tile (not with stochastic rounding,
    // whose draws need the registers)
    const int64_t next = (!SR && nt < nfull) ? nt : -1;
    if (t < nfull)
      group_tile<T, BITS, AFFINE, LPG, STATS_ONLY, true, SR, OPT>(x, n, t, v, have, next, scale, zp,
                                                             absmax, minv, maxv, sr, co, y, codes,
                                                             mask, lane, fl);
    else
      group_tile<T, BITS, AFFINE, LPG, STATS_ONLY, false, SR, OPT>(x, n, t, v, have, next, scale, zp,
                                                              absmax, minv, maxv, sr, co, y, codes,
                                                              mask, lane, fl);
    have = next >= 0;
  }
  warp_flag_or(flags, fl);
}

// ---------------------------------------------------------------------------
// one thread block (256 threads) per unit of L elements, NV vectors / thread
// ---------------------------------------------------------------------------
template <typename T, int BITS, bool AFFINE, int NV, bool STATS_ONLY, bool SR>
__global__ void __launch_bounds__(256, NV <= 2 ? 4 : 1)
    k_int_rows(const void* __restrict__ x, int64_t units, int64_t L, float* scale, int32_t* zp,
               float* absmax, float* minv, float* maxv, SrCtx sr, CalOpts co, void* y, void* codes,
               uint32_t* mask, int32_t* flags) {
  constexpr int VEC = T::VEC, NT = 256;
  constexpr int LPW = 32 / VEC;
  constexpr int MM = STATS_ONLY ? kMMKeys : (AFFINE ? kMMFloat : kMMNone);
  __shared__ __align__(16) uint32_t red[4 * 8];
  __shared__ IntParams sp;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = (int)(L / VEC);
  // The row's statistics are folded per warp (redux.sync), the 8 warp
  // partials by warp 0, whose lane 0 calibrates and publishes the parameters
  // in shared memory: once per row, not once per thread.  `red` and `sp` are
  // rewritten by the next row only after its first barrier, by which time
  // every thread has read them.
  // the next unit's vectors are requested before the current one is
  // processed, so each block keeps a unit's worth of loads in flight
  auto load_unit = [&](int64_t uu, V32 (&dst)[NV]) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vi = threadIdx.x + j * NT;
      if (uu < units && vi < nvec) {
        dst[j] = ld_v32(static_cast<const char*>(x) + (uu * L + (int64_t)vi * VEC) * T::BYTES);
      } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) dst[j].w[w] = 0u;
      }
    }
  };
  V32 v[NV];
  load_unit(blockIdx.x, v);
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t ub = u * L;
    V32 vn[NV];
    load_unit(u + gridDim.x, vn);
    Stats st;
    st.init<MM>();
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      int vi = threadIdx.x + j * NT;
      if (vi < nvec) {
        stats_add_vec<T, MM>(st, v[j]);
      }
    }
    st.reduce_lanes<MM>(32);
    if (lane == 0) reinterpret_cast<uint4*>(red)[warp] = st.pack();
    __syncthreads();
    if (warp == 0) {
      Stats b;
      b.init<MM>();
      if (lane < NT / 32) b.unpack(reinterpret_cast<const uint4*>(red)[lane]);
      b.reduce_lanes<MM>(NT / 32);
      if (lane == 0) {
        if (STATS_ONLY) {
          if (absmax) absmax[u] = b.absmax_f();
          if (minv) minv[u] = b.min_f<MM>();
          if (maxv) maxv[u] = b.max_f<MM>();
          flag_or(flags, b.has_nonfinite() ? QAT_FLAG_NONFINITE_INPUT : 0);
        } else {
          IntParams q;
          const int f = calibrate<BITS, AFFINE, MM>(b, q, co);
          sp = q;
          scale[u] = q.s;
          if (zp) zp[u] = q.zp;
          flag_or(flags, f);
        }
      }
    }
    if (STATS_ONLY) {
#pragma unroll
      for (int j = 0; j < NV; ++j) v[j] = vn[j];
      continue;
    }
    __syncthreads();
    const IntParams p = sp;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vi = threadIdx.x + j * NT;
      const bool present = vi < nvec;
      const int64_t base = ub + (int64_t)vi * VEC;
      OutVec<T> ov;
      CodeVec<BITS, VEC> cv;
      uint32_t mb;
      int_map_vec<T, BITS, AFFINE, SR>(v[j], p, ov, cv, mb, sr, base);
      if (present) {
        if (y) st_v32(static_cast<char*>(y) + base * T::BYTES, ov.v);
        if (codes) cv.store(codes, base, VEC);
      }
      // L % 32 == 0: the LPW lanes of a mask word are all present or all absent
      uint32_t w = mask_word_of_slot<VEC>(present ? mb : 0u, lane);
      if (mask && present && (lane % LPW) == 0) mask[base >> 5] = w;
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = vn[j];
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int lpg_of(qat_dtype dt, int64_t L) {
  const int vec = dt == QAT_F32 ? F32::VEC : BF16::VEC;
  for (int lpg = 2; lpg <= 32; lpg <<= 1)
    if (L == (int64_t)vec * lpg) return lpg;
  return 0;
}

static int nv_of(qat_dtype dt, int64_t L) {
  const int vec = dt == QAT_F32 ? F32::VEC : BF16::VEC;
  if (L % 32 != 0) return 0;
  int64_t nvec = L / vec;
  for (int nv = 1; nv <= 8; nv <<= 1)
    if (nvec <= 256 * nv) return nv;
  return 0;
}

#if !QAT_SR
bool fused_units_supported(qat_dtype dt, int64_t L) { return lpg_of(dt, L) || nv_of(dt, L); }
#endif

template <typename T, int BITS, bool AFFINE, bool SO>
static qat_status groups_t(int lpg, const void* x, int64_t n, float* scale, int32_t* zp,
                           float* absmax, float* minv, float* maxv, const SrCtx& sr,
                           const CalOpts& co, void* y, void* codes, uint32_t* mask, int32_t* flags,
                           cudaStream_t s) {
  const int64_t ntiles = (n + kTile - 1) / kTile;
  int64_t g = (ntiles + 7) / 8;
  int64_t cap = (int64_t)device_info().sms * 8;
  int grid = (int)(g > cap ? cap : (g < 1 ? 1 : g));
  // the options as a compile-time switch of the nearest-rounding build (the
  // stochastic build has the registers and always takes them at run time)
  const bool opt = QAT_SR || co.clip != 1.0f || co.fp16 || co.clamp;
#define QAT_G(LP)                                                                              \
  do {                                                                                         \
    if (opt)                                                                                   \
      k_int_groups<T, BITS, AFFINE, LP, SO, QAT_SR, true><<<grid, 256, 0, s>>>(                \
          x, n, scale, zp, absmax, minv, maxv, sr, co, y, codes, mask, flags);                 \
    else /* the stochastic build never gets here (opt is set): same instantiation */      \
      k_int_groups<T, BITS, AFFINE, LP, SO, QAT_SR, (QAT_SR != 0)><<<grid, 256, 0, s>>>(       \
          x, n, scale, zp, absmax, minv, maxv, sr, co, y, codes, mask, flags);                 \
  } while (0)
  switch (lpg) {
    case 2: QAT_G(2); break;
    case 4: QAT_G(4); break;
    case 8: QAT_G(8); break;
    case 16: QAT_G(16); break;
    default: QAT_G(32); break;
  }
#undef QAT_G
  return launch_status();
}

template <typename T, int BITS, bool AFFINE, bool SO>
static void rows_t(int nv, const void* x, int64_t units, int64_t L, float* scale, int32_t* zp,
                   float* absmax, float* minv, float* maxv, const SrCtx& sr, const CalOpts& co,
                   void* y, void* codes, uint32_t* mask, int32_t* flags, cudaStream_t s) {
  int64_t cap = (int64_t)device_info().sms * 8;
  int grid = (int)(units > cap ? cap : (units < 1 ? 1 : units));
#define QAT_R(NV)                                                                         \
  k_int_rows<T, BITS, AFFINE, NV, SO, QAT_SR><<<grid, 256, 0, s>>>(x, units, L, scale, zp,     \
                                                                   absmax, minv, maxv, sr, co, \
                                                                   y, codes, mask, flags)
  switch (nv) {
    case 1: QAT_R(1); break;
    case 2: QAT_R(2); break;
    case 4: QAT_R(4); break;
    default: QAT_R(8); break;
  }
#undef QAT_R
}

template <typename T, int BITS, bool AFFINE, bool SO>
static qat_status fused_t(const void* x, int64_t units, int64_t L, float* scale, int32_t* zp,
                          float* absmax, float* minv, float* maxv, const SrCtx& sr,
                          const CalOpts& co, void* y, void* codes, uint32_t* mask,
                          int32_t* flags, cudaStream_t s) {
  const qat_dtype dt = T::kDtype;
  int lpg = lpg_of(dt, L);
  if (lpg)
    return groups_t<T, BITS, AFFINE, SO>(lpg, x, units * L, scale, zp, absmax, minv, maxv, sr, co,
                                         y, codes, mask, flags, s);
  rows_t<T, BITS, AFFINE, SO>(nv_of(dt, L), x, units, L, scale, zp, absmax, minv, maxv, sr, co, y,
                              codes, mask, flags, s);
  return launch_status();
}

QAT_DECL_INT_FUSED(QAT_SR_NAME(launch_int_fused)) {
  if (!(lpg_of(dt, L) || nv_of(dt, L))) return QAT_ERR_UNSUPPORTED;
  qat_status st;
#define QAT_F(T, B, A, SO) \
  st = fused_t<T, B, A, SO>(x, units, L, scale, zp, absmax, minv, maxv, sr, co, y, codes, mask, flags, s)
  if (stats_only) {
#if QAT_SR
    return QAT_ERR_UNSUPPORTED;
#else
    if (dt == QAT_F32) QAT_F(F32, 8, false, true);
    else QAT_F(BF16, 8, false, true);
#endif
  } else if (dt == QAT_F32) {
    if (bits == 8) { if (affine) QAT_F(F32, 8, true, false); else QAT_F(F32, 8, false, false); }
    else { if (affine) QAT_F(F32, 4, true, false); else QAT_F(F32, 4, false, false); }
  } else {
    if (bits == 8) { if (affine) QAT_F(BF16, 8, true, false); else QAT_F(BF16, 8, false, false); }
    else { if (affine) QAT_F(BF16, 4, true, false); else QAT_F(BF16, 4, false, false); }
  }
#undef QAT_F
  if (st == QAT_OK) count_launch(1);
  return st;
}

}  // namespace qat
