// kernels_cols.cu -- per-column (channel axis 1) integer fake quant.
//
// optirs-gpu quantization.rs, per_channel_params / fake_quant_int_per_channel
// with the channel axis along the columns of a row-major [rows, cols] tensor:
// one scale (and zero point) per column, calibrated from that column's
// absmax (symmetric) or min / max (affine) exactly as a row is.
//
// A column's statistics need every row before its first element can be
// mapped, so the calibrated path is two passes over x.  In both kernels a
// lane takes 16 bytes of a row (4 fp32 or 8 bf16 columns), a warp a strip of
// 32 lanes, and the 8 warps of a block sit side by side (up to 8 strips, so
// the block reads up to 4 KiB of each row) and walk the rows of their chunk.
// When the row length is a multiple of 32 the rows come in through shared
// memory (bulk copies, several tiles in flight); otherwise through registers.
//   k_col_init      resets the per-column accumulators
//   k_col_stats*    fold the chunk into per-column partials and combine each
//                   block's partial into the accumulators with integer
//                   atomics (absmax bits and order keys are monotone as
//                   unsigned integers)
//   k_int_cols      calibrates its columns from the accumulators while its
//                   first tiles are in flight, keeps their parameters in
//                   registers and maps the rows of its chunk
//   k_col_finalize  the accumulators -> statistics outputs, or scale, zero
//                   point and dead byte for the unit-kernel fallback
// Row lengths that are not a multiple of 32 (mask words would straddle rows)
// and given parameters take the per-element unit kernel in column mode.
#include <atomic>

#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

constexpr int kColWarps = 8;    // warps per block, interleaved along rows
// columns per lane (16 bytes of a row) and per warp strip
template <typename T>
constexpr int kColLane = 16 / T::BYTES;
template <typename T>
constexpr int kColStrip = 32 * kColLane<T>;

// The parameters of one column as the map uses them: wlo is stored as -0
// when it is zero (the window test).
struct ColP {
  float s, rcp, wlo, whi, klof, khif;
  int zp;
  int st;  // bit 0 dead, bit 1 fast (scale in the reciprocal's safe range)
};

// Grid of both column kernels: `wc` warp strips side by side in a block (a
// power of two up to 8; the other 8 / wc warps interleave along rows), so a
// block covers wc * ws columns of every row it reads; strips of that width
// along x, chunks of `rchunk` rows along y (a multiple of `mult` chunks,
// trailing ones empty).
struct ColShape {
  int wc;
  int64_t strips, chunks, rchunk;
};

static ColShape col_shape(int64_t rows, int64_t cols, int64_t ws, int per_sm, int64_t min_rows,
                          int64_t mult) {
  ColShape g;
  const int64_t warps = (cols + ws - 1) / ws;
  g.wc = 1;
  while (g.wc < kColWarps && g.wc < warps) g.wc <<= 1;
  const int64_t sw = ws * g.wc;
  g.strips = (cols + sw - 1) / sw;
  const int64_t want = ((int64_t)device_info().sms * per_sm + g.strips - 1) / g.strips;
  const int64_t most = (rows + min_rows - 1) / min_rows;
  int64_t chunks = want < most ? want : most;
  if (chunks < 1) chunks = 1;
  if (chunks > 65535 - mult) chunks = 65535 - mult;
  g.rchunk = (rows + chunks - 1) / chunks;
  chunks = (rows + g.rchunk - 1) / g.rchunk;
  g.chunks = (chunks + mult - 1) / mult * mult;
  return g;
}

// 16 bytes of one row as loaded: four fp32 or eight bf16 values
struct Raw16 {
  uint32_t w[4];
};
__device__ __forceinline__ Raw16 load_raw16(const void* p) {
  const uint4 v = __ldg(static_cast<const uint4*>(p));
  return Raw16{{v.x, v.y, v.z, v.w}};
}
// element j of a lane's columns as fp32
template <typename T>
__device__ __forceinline__ float raw_elem(const Raw16& r, int j) {
  if (T::BYTES == 4) return __uint_as_float(r.w[j]);
  const uint32_t w = r.w[j >> 1];
  return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
}
// the lane's columns of row element offset i: one 16-byte load when the row
// is 16-byte aligned (vec) and all `have` columns exist, else element loads
// (absent ones read +0)
template <typename T>
__device__ __forceinline__ Raw16 load_lane(const void* x, int64_t i, int have, bool vec) {
  constexpr int NC = kColLane<T>;
  if (vec && have >= NC) return load_raw16(static_cast<const char*>(x) + i * T::BYTES);
  Raw16 r = {{0u, 0u, 0u, 0u}};
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    if (j < have) {
      const uint32_t b = load_elem_bits<T>(x, i + j);
      if (T::BYTES == 4)
        r.w[j] = b;
      else
        r.w[j >> 1] |= (j & 1) ? (b & 0xffff0000u) : (b >> 16);
    }
  }
  return r;
}

// ---------------------------------------------------------------------------
// staged row tiles: a block walks its chunk in tiles of `tr` rows of its
// strip, copied into shared memory by bulk copies (cp.async.bulk, one per
// row segment, or one per tile when the strip is the whole row) that complete
// on a per-stage mbarrier; kColStages tiles are in flight.  Every wait is
// bounded: when one runs out the block records QAT_FLAG_DEVICE_TIMEOUT,
// waits (bounded) for the copies it issued and leaves.
// ---------------------------------------------------------------------------
constexpr int kColStageBytes = 32768;
constexpr int kColStages = 3;
constexpr uint32_t kColWaitLimit = 1u << 24;  // try_wait polls of the drain before giving up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(b))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0u;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(b, parity)) return true;
  return false;
}

// The tiles of one block: rows [r0, r1) of the strip starting at column cs,
// `segc` columns wide (whole rows when contig), `tr` rows per tile.
struct ColTiles {
  const char* x;
  int64_t cols, cs, r0, r1;
  int segc, tr, tiles, bytes_per_elem;
  bool contig;
  uint32_t wait_limit;  // polls of a tile wait (the drain always takes kColWaitLimit)
  __device__ __forceinline__ uint32_t seg_bytes() const { return (uint32_t)segc * bytes_per_elem; }
  __device__ __forceinline__ int rows_of(int t) const {
    const int64_t left = r1 - r0 - (int64_t)t * tr;
    return left < tr ? (int)left : tr;
  }
  // thread 0: the copies of tile t into stage buffer `dst`, completing on `bar`
  __device__ __forceinline__ void issue(int t, char* dst, uint64_t* bar) const {
    const int nr = rows_of(t);
    const uint32_t sb = seg_bytes();
    const int64_t rs = r0 + (int64_t)t * tr;
    mbar_expect_tx(bar, (uint32_t)nr * sb);
    if (contig) {
      bulk_g2s(dst, x + rs * cols * bytes_per_elem, (uint32_t)nr * sb, bar);
    } else {
      for (int i = 0; i < nr; ++i)
        bulk_g2s(dst + (size_t)i * sb, x + ((rs + i) * cols + cs) * bytes_per_elem, sb, bar);
    }
  }
};

// The staged walk: issues the first tiles, runs prologue(), then calls
// body(tile_base, tile, rows_in_tile) for every tile of the block, with all
// threads; returns false (flag set, copies drained) when a wait ran out.  The caller provides kColStages * kColStageBytes bytes of
// dynamic shared memory at `stage` and kColStages mbarriers at `bars`.
template <typename Pro, typename Body>
__device__ __forceinline__ bool col_staged(const ColTiles& tl, char* stage, uint64_t* bars,
                                           int32_t* flags, Pro&& prologue, Body&& body) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < kColStages; ++s) mbar_init(bars + s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int s = 0; s < kColStages && s < tl.tiles; ++s)
      tl.issue(s, stage + s * kColStageBytes, bars + s);
  prologue();  // runs while the first tiles are in flight
  for (int t = 0; t < tl.tiles; ++t) {
    const int s = t % kColStages;
    const uint32_t par = (uint32_t)(t / kColStages) & 1u;
    const bool ok = mbar_wait(bars + s, par, tl.wait_limit);
    if (ok) body(stage + s * kColStageBytes, t, tl.rows_of(t));
    // every thread is done with stage s (or a wait ran out somewhere)
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        // drain the copies still in flight, then report
        for (int u = t; u < tl.tiles && u < t + kColStages; ++u)
          mbar_wait(bars + u % kColStages, (uint32_t)(u / kColStages) & 1u, kColWaitLimit);
        if (flags) atomicOr(flags, QAT_FLAG_DEVICE_TIMEOUT);
      }
      return false;
    }
    if (threadIdx.x == 0 && t + kColStages < tl.tiles) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tl.issue(t + kColStages, stage + s * kColStageBytes, bars + s);
    }
  }
  return true;
}

template <int BITS, bool AFFINE>
__device__ __forceinline__ ColP col_params(const IntParams& p) {
  ColP q;
  q.s = p.s;
  q.rcp = p.rcp;
  q.wlo = p.wlo == 0.0f ? -0.0f : p.wlo;
  q.whi = p.whi;
  q.klof = p.klof;
  q.khif = p.khif;
  q.zp = p.zp;
  // a unit whose quotients may overflow (fast == 3) takes the division path
  q.st = (p.dead ? 1 : 0) | ((p.fast == 1 || p.fast == 2) ? 2 : 0);
  return q;
}

#if !QAT_SR
// One element into a column's statistics.  With order keys the absmax is
// left to the finalisation (max(|min|, |max|)), so only min, max and the
// non-finite bit are folded.
template <int MM>
__device__ __forceinline__ void col_add(Stats& st, uint32_t u) {
  if (MM != kMMKeys) {
    st.add<MM>(u);
    return;
  }
  const bool fin = (u & 0x7fffffffu) < 0x7f800000u;
  const uint32_t k = order_key(u);
  st.nonfinite |= fin ? 0u : 1u;
  st.kmin = min(st.kmin, fin ? k : kKeyPosInf);
  st.kmax = max(st.kmax, fin ? k : kKeyNegInf);
}

__global__ void k_col_init(uint4* __restrict__ acc, int64_t cols) {
  pdl_trigger();
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c < cols) acc[c] = make_uint4(0u, 0u, kKeyPosInf, kKeyNegInf);
}

// After the fold: merge the warps that share a strip (red: the block's
// kColWarps x WW partials in shared memory) and combine the block's partial
// of each column into the accumulators.
template <typename T, int MM>
__device__ __forceinline__ void col_stats_combine(const Stats (&st)[kColLane<T>], uint4* red,
                                                  int wc, int64_t cols, uint4* __restrict__ acc) {
  constexpr int NC = kColLane<T>, WW = kColStrip<T>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nrw = kColWarps / wc;
  const int sw = WW * wc;
#pragma unroll
  for (int j = 0; j < NC; ++j) red[warp * WW + lane * NC + j] = st[j].pack();
  __syncthreads();
  if (nrw > 1) {
    for (int t = threadIdx.x; t < sw; t += blockDim.x) {
      const int ts = t / WW, tl = t % WW;
      Stats s;
      s.unpack(red[ts * WW + tl]);
      for (int w = 1; w < nrw; ++w) {
        Stats o;
        o.unpack(red[(w * wc + ts) * WW + tl]);
        s.merge<MM>(o);
      }
      red[ts * WW + tl] = s.pack();
    }
    __syncthreads();
  }
  for (int t = threadIdx.x; t < sw; t += blockDim.x) {
    const int64_t col = (int64_t)blockIdx.x * sw + t;
    if (col < cols) {
      Stats s;
      s.unpack(red[t]);
      uint32_t* a = reinterpret_cast<uint32_t*>(acc + col);
      if (MM == kMMKeys) {
        if (s.kmin != kKeyPosInf) atomicMin(a + 2, s.kmin);
        if (s.kmax != kKeyNegInf) atomicMax(a + 3, s.kmax);
      } else if (s.amax) {
        atomicMax(a + 0, s.amax);
      }
      if (s.nonfinite) atomicOr(a + 1, 1u);
    }
  }
}
#endif  // !QAT_SR

// A column's statistics from its accumulator; with order keys the finite
// absmax is max(|min|, |max|) (0 when the column has no finite value).
template <int MM>
__device__ __forceinline__ Stats col_acc_stats(const uint4& a) {
  Stats s;
  s.unpack(a);
  if (MM == kMMKeys) {
    const uint32_t am = max(key_to_bits(s.kmin) & 0x7fffffffu, key_to_bits(s.kmax) & 0x7fffffffu);
    s.amax = s.kmin <= s.kmax ? am : 0u;
  }
  return s;
}

#if !QAT_SR
// The accumulators of every column (one thread each).  MODE 0: absmax / min /
// max (finite values) and QAT_FLAG_NONFINITE_INPUT.  MODE 1: the integer
// calibration -> scale, zero point and dead byte (the unit-kernel fallback),
// and the calibration flags.
template <int MODE, int BITS, bool AFFINE>
__global__ void k_col_finalize(const uint4* __restrict__ acc, int64_t cols, float* out0,
                               float* out1, float* out2, int32_t* zp, uint8_t* dead, CalOpts co,
                               int32_t* flags) {
  constexpr int MM = (MODE == 0 || AFFINE) ? kMMKeys : kMMNone;
  pdl_wait();  // launched early: the accumulators come from the statistics kernel
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int f = 0;
  if (c < cols) {
    const Stats s = col_acc_stats<MM>(acc[c]);
    if (MODE == 0) {
      if (out0) out0[c] = s.absmax_f();
      if (out1) out1[c] = s.min_f<kMMKeys>();
      if (out2) out2[c] = s.max_f<kMMKeys>();
      f = s.has_nonfinite() ? QAT_FLAG_NONFINITE_INPUT : 0;
    } else {
      IntParams p;
      f = calibrate<BITS, AFFINE, MM>(s, p, co);
      out0[c] = p.s;
      if (zp) zp[c] = p.zp;
      dead[c] = (uint8_t)p.dead;
    }
  }
  warp_flag_or(flags, f);
}

// Column statistics (MM: kMMNone for the symmetric calibration, otherwise
// kMMKeys) for any row length (element loads where a row is not 16-byte
// aligned), the rows through registers: kColDepth loads in flight per warp.
constexpr int kColDepth = 4;

template <typename T, int MM>
__global__ void __launch_bounds__(256, 3)
    k_col_stats(const void* __restrict__ x, int64_t rows, int64_t cols, int wc, int64_t rchunk,
                uint4* __restrict__ acc) {
  constexpr int NC = kColLane<T>, WW = kColStrip<T>, D = kColDepth;
  __shared__ uint4 red[kColWarps * WW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = warp & (wc - 1), rw = warp / wc, nrw = kColWarps / wc;
  const int sw = WW * wc;
  const int64_t c = (int64_t)blockIdx.x * sw + sub * WW + lane * NC;
  const bool vec = cols % NC == 0;
  const int have = c < cols ? (cols - c >= NC ? NC : (int)(cols - c)) : 0;
  Stats st[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) st[j].template init<MM>();
  const int64_t r0 = (int64_t)blockIdx.y * rchunk + rw;
  const int64_t r1 = min(rows, (int64_t)blockIdx.y * rchunk + rchunk);
  const int64_t step = nrw;
  if (have > 0) {
    // rows r0, r0 + step, ...: D loads in flight, each row's load issued D
    // rows ahead of its fold
    Raw16 b[D];
#pragma unroll
    for (int k = 0; k < D; ++k) {
      const int64_t rk = r0 + k * step;
      if (rk < r1) b[k] = load_lane<T>(x, rk * cols + c, have, vec);
    }
    for (int64_t r = r0; r < r1; r += D * step) {
#pragma unroll
      for (int k = 0; k < D; ++k) {
        const int64_t rk = r + k * step;
        if (rk >= r1) break;
        const Raw16 cur = b[k];
        const int64_t rn = rk + D * step;
        if (rn < r1) b[k] = load_lane<T>(x, rn * cols + c, have, vec);
#pragma unroll
        for (int j = 0; j < NC; ++j)
          if (j < have) col_add<MM>(st[j], __float_as_uint(raw_elem<T>(cur, j)));
      }
    }
  }
  pdl_trigger();
  pdl_wait();  // launched early: the accumulators are set by k_col_init
  col_stats_combine<T, MM>(st, red, wc, cols, acc);
}

// The same statistics for row lengths that are a multiple of 32: the rows of
// the block's strip come in through the staged tiles (shared memory), so the
// loads in flight do not occupy registers.
template <typename T, int MM>
__global__ void __launch_bounds__(256, 2)
    k_col_stats_staged(const void* __restrict__ x, int64_t rows, int64_t cols, int wc,
                       int64_t rchunk, int tr, uint32_t wait_limit, uint4* __restrict__ acc,
                       int32_t* flags) {
  constexpr int NC = kColLane<T>, WW = kColStrip<T>;
  extern __shared__ __align__(128) char col_stage[];
  __shared__ __align__(8) uint64_t bars[kColStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = warp & (wc - 1), rw = warp / wc, nrw = kColWarps / wc;
  const int sw = WW * wc;
  ColTiles tl;
  tl.x = static_cast<const char*>(x);
  tl.cols = cols;
  tl.cs = (int64_t)blockIdx.x * sw;
  tl.segc = (int)(cols - tl.cs < sw ? cols - tl.cs : sw);
  tl.contig = tl.segc == cols;
  tl.bytes_per_elem = T::BYTES;
  tl.r0 = (int64_t)blockIdx.y * rchunk;
  tl.r1 = min(rows, tl.r0 + rchunk);
  tl.tr = tr;
  tl.wait_limit = wait_limit;
  tl.tiles = tl.r1 > tl.r0 ? (int)((tl.r1 - tl.r0 + tr - 1) / tr) : 0;
  const int cl = sub * WW + lane * NC;  // the lane's first column in the strip
  const bool active = cl < tl.segc;
  const int64_t c = tl.cs + cl;
  const uint32_t sb = tl.seg_bytes();
  // Raw folds over every value, non-finite ones included: the absmax bits
  // (symmetric) or the order keys of min and max, per column (fp32) or per
  // pair of columns in 16-bit halves (bf16).  A non-finite value pushes the
  // raw result past the finite range, and only then is the column folded
  // again, exactly, from global memory.
  constexpr int NW = T::BYTES == 4 ? NC : NC / 2;  // accumulator words
  uint32_t lo[NW], hi[NW];
#pragma unroll
  for (int k = 0; k < NW; ++k) {
    lo[k] = 0xffffffffu;  // min of keys
    hi[k] = 0u;           // max of keys, or of absmax bits
  }
  const bool ok = col_staged(tl, col_stage, bars, flags, [] {}, [&](const char* tile, int, int nr) {
    if (!active) return;
    for (int r = rw; r < nr; r += nrw) {
      const uint4 v = *reinterpret_cast<const uint4*>(tile + (size_t)r * sb + cl * T::BYTES);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (T::BYTES == 4) {
          if (MM == kMMKeys) {
            const uint32_t key = order_key(w[k]);
            lo[k] = min(lo[k], key);
            hi[k] = max(hi[k], key);
          } else {
            hi[k] = max(hi[k], w[k] & 0x7fffffffu);
          }
        } else if (MM == kMMKeys) {
          // 16-bit order keys of both halves: h ^ 0xffff when negative, h ^ 0x8000 otherwise
          const uint32_t key2 = w[k] ^ (((w[k] >> 15) & 0x00010001u) * 0x7fffu) ^ 0x80008000u;
          asm("min.u16x2 %0, %0, %1;" : "+r"(lo[k]) : "r"(key2));
          asm("max.u16x2 %0, %0, %1;" : "+r"(hi[k]) : "r"(key2));
        } else {
          asm("max.u16x2 %0, %0, %1;" : "+r"(hi[k]) : "r"(w[k] & 0x7fff7fffu));
        }
      }
    }
  });
  if (!ok) return;
  Stats st[NC];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    Stats& sj = st[j];
    sj.init<MM>();
    if (!active) continue;
    if (T::BYTES == 4) {
      if (MM == kMMKeys) {
        bad |= lo[j] <= kKeyNegInf || hi[j] >= kKeyPosInf;
        sj.kmin = lo[j];
        sj.kmax = hi[j];
      } else {
        bad |= hi[j] >= 0x7f800000u;
        sj.amax = hi[j];
      }
    } else {
      const int sh = (j & 1) ? 16 : 0;
      if (MM == kMMKeys) {
        // the fp32 key of a bf16 key: key << 16, low bits all ones when negative
        const uint32_t kl = (lo[j >> 1] >> sh) & 0xffffu, kh = (hi[j >> 1] >> sh) & 0xffffu;
        bad |= kl <= 0x007fu || kh >= 0xff80u;
        sj.kmin = (kl << 16) | (kl < 0x8000u ? 0xffffu : 0u);
        sj.kmax = (kh << 16) | (kh < 0x8000u ? 0xffffu : 0u);
      } else {
        const uint32_t a = (hi[j >> 1] >> sh) & 0xffffu;
        bad |= a >= 0x7f80u;
        sj.amax = a << 16;
      }
    }
  }
  if (bad) {
    // a non-finite value in one of the lane's columns: their exact statistics
    // over the lane's rows of the chunk, one 16-byte load per row, 4 in flight
#pragma unroll
    for (int j = 0; j < NC; ++j) st[j].template init<MM>();
    const int64_t step = nrw;
    for (int64_t r = tl.r0 + rw; r < tl.r1; r += 4 * step) {
      Raw16 b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (r + k * step < tl.r1) b[k] = load_lane<T>(x, (r + k * step) * cols + c, NC, true);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (r + k * step >= tl.r1) break;
#pragma unroll
        for (int j = 0; j < NC; ++j) st[j].template add<MM>(__float_as_uint(raw_elem<T>(b[k], j)));
      }
    }
  }
  pdl_trigger();
  pdl_wait();  // launched early: the accumulators are set by k_col_init
  col_stats_combine<T, MM>(st, reinterpret_cast<uint4*>(col_stage), wc, cols, acc);
}
#endif  // !QAT_SR

// ---------------------------------------------------------------------------
// the calibrated per-column map
// ---------------------------------------------------------------------------
// the fields of a record the fast path reads, held in registers per column
struct ColR {
  float s, rcp, wlo, whi, klof, khif;
  int zp;
};

// The IEEE-division path of one element of a calibrated column that is dead
// or has a scale outside the reciprocal's safe range.
template <int BITS, bool AFFINE, bool SR>
__device__ __forceinline__ void col_slow_elem(float x, float u, const ColR& c, bool dead, float& y,
                                              int& q, uint32_t& m) {
  constexpr int qmin = QRange<BITS, AFFINE>::qmin, qmax = QRange<BITS, AFFINE>::qmax;
  if (dead) {
    y = 0.0f;
    q = 0;
    m = 0u;
    return;
  }
  IntParams p;
  p.s = c.s;
  p.zp = c.zp;
  p.dead = 0;
  p.fast = 0;
  p.rcp = 0.0f;
  finish_params(p, qmin, qmax);
  if (SR)
    int_elem_sr<false>(x, u, p, q, y, m);
  else
    int_elem<false>(x, p, q, y, m);
}

// Two elements of two fast calibrated columns a, b (finite values): the
// exact quotient RN(x / s) (the Markstein step of quotient_rn2 with a
// reciprocal and a scale per element), rint by the magic constant (nearest)
// or the stochastic rounding with draws ua, ub, the clamp (affine, clampsym,
// and every stochastic rounding), y = k s, the code from the bits of k + M, and the
// out-of-window sign bits (whi - |x| symmetric; whi - x, x - wlo affine).
template <bool AFFINE, bool SR>
__device__ __forceinline__ void col_pair(float xa, float xb, const ColR& a, const ColR& b,
                                         float ua, float ub, bool clampsym, float& ya, float& yb,
                                         int& qa, int& qb, uint32_t& oa, uint32_t& ob) {
  float fa, fb, ra, rb, ta, tb;
  const float nsa = -a.s, nsb = -b.s;
  mul2(xa, xb, a.rcp, b.rcp, fa, fb);
  fma2(fa, fb, nsa, nsb, xa, xb, ra, rb);
  fma2(ra, rb, a.rcp, b.rcp, fa, fb, fa, fb);
  fma2(fa, fb, nsa, nsb, xa, xb, ra, rb);
  fma2(ra, rb, a.rcp, b.rcp, fa, fb, fa, fb);
  if (SR) {
    fa = fminf(fmaxf(sr_round(fa, ua), a.klof), a.khif);
    fb = fminf(fmaxf(sr_round(fb, ub), b.klof), b.khif);
    add2(fa, fb, kRintMagic, kRintMagic, ta, tb);
  } else {
    add2(fa, fb, kRintMagic, kRintMagic, ta, tb);
    sub2(ta, tb, kRintMagic, kRintMagic, fa, fb);
    if (AFFINE || clampsym) {
      fa = fminf(fmaxf(fa, a.klof), a.khif);
      fb = fminf(fmaxf(fb, b.klof), b.khif);
      add2(fa, fb, kRintMagic, kRintMagic, ta, tb);
    }
  }
  mul2(fa, fb, a.s, b.s, ya, yb);
  qa = (int)(__float_as_uint(ta) - kRintMagicBits) + (AFFINE ? a.zp : 0);
  qb = (int)(__float_as_uint(tb) - kRintMagicBits) + (AFFINE ? b.zp : 0);
  if (AFFINE) {
    float ha, hb, la, lb;
    sub2(a.whi, b.whi, xa, xb, ha, hb);
    sub2(xa, xb, a.wlo, b.wlo, la, lb);
    oa = (__float_as_uint(ha) | __float_as_uint(la)) >> 31;
    ob = (__float_as_uint(hb) | __float_as_uint(lb)) >> 31;
  } else {
    oa = __float_as_uint(__fsub_rn(a.whi, fabsf(xa))) >> 31;
    ob = __float_as_uint(__fsub_rn(b.whi, fabsf(xb))) >> 31;
  }
}

// One row of a lane's NC columns at element i: map, store y and the codes
// (packed as each pair is done), return the NC mask bits (bit j = column j).
// SLOW: columns whose bit is set in `slowm` take the IEEE path (dead ones,
// bit set in `deadm`, give zeros).
template <typename T, int BITS, bool AFFINE, bool SR, bool SLOW>
__device__ __forceinline__ uint32_t col_row(const Raw16& b, const ColR (&P)[kColLane<T>],
                                            uint32_t slowm, uint32_t deadm, bool clampsym,
                                            const SrCtx& sr, int64_t i, void* y, void* codes) {
  constexpr int NC = kColLane<T>;
  uint32_t yw[4];         // the y row as stored: 4 fp32, or 8 bf16 in pairs
  uint32_t cw[NC / 4];    // the codes as stored
  uint32_t mb = 0u;
#pragma unroll
  for (int k = 0; k < NC / 4; ++k) cw[k] = 0u;
#pragma unroll
  for (int g = 0; g < NC / 4; ++g) {
    float u[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (SR) sr_draws4(sr, i / 4 + g, u);
#pragma unroll
    for (int h = 0; h < 4; h += 2) {
      const int j = 4 * g + h;
      const float xa = raw_elem<T>(b, j), xb = raw_elem<T>(b, j + 1);
      float ya, yb;
      int qa, qb;
      uint32_t oa, ob;
      col_pair<AFFINE, SR>(xa, xb, P[j], P[j + 1], u[h], u[h + 1], clampsym, ya, yb, qa, qb, oa,
                           ob);
      uint32_t ma = oa ^ 1u, mbb = ob ^ 1u;
      if (SLOW) {
        if ((slowm >> j) & 1u)
          col_slow_elem<BITS, AFFINE, SR>(xa, u[h], P[j], (deadm >> j) & 1u, ya, qa, ma);
        if ((slowm >> (j + 1)) & 1u)
          col_slow_elem<BITS, AFFINE, SR>(xb, u[h + 1], P[j + 1], (deadm >> (j + 1)) & 1u, yb, qb,
                                          mbb);
      }
      mb |= (ma << j) | (mbb << (j + 1));
      if (T::BYTES == 4) {
        yw[j] = __float_as_uint(ya);
        yw[j + 1] = __float_as_uint(yb);
      } else {
        yw[j >> 1] = pack_bf16x2(ya, yb);
      }
      // int8: byte j = code j; int4: element 2m in the high nibble of byte m
      if (BITS == 8)
        cw[j >> 2] |= ((uint32_t)(qa & 0xff) << (8 * (j & 3))) |
                      ((uint32_t)(qb & 0xff) << (8 * ((j + 1) & 3)));
      else
        cw[j >> 3] |= (((uint32_t)(qa & 0xf) << 4) | (uint32_t)(qb & 0xf)) << (8 * ((j >> 1) & 3));
    }
  }
  if (y) *reinterpret_cast<uint4*>(static_cast<char*>(y) + i * T::BYTES) =
      make_uint4(yw[0], yw[1], yw[2], yw[3]);
  if (codes) {
    uint8_t* p = static_cast<uint8_t*>(codes) + (BITS == 8 ? i : i / 2);
    if (BITS == 8 && NC == 8)
      *reinterpret_cast<uint2*>(p) = make_uint2(cw[0], cw[1]);
    else if (BITS == 8 || NC == 8)
      *reinterpret_cast<uint32_t*>(p) = cw[0];
    else
      *reinterpret_cast<uint16_t*>(p) = (uint16_t)cw[0];
  }
  return mb;
}

// The rows rw, rw + nrw, ... of one staged tile (the tile's first row is rs):
// map, store, and assemble the mask words with shuffles (the loop is
// warp-uniform).  Requires cols % 32 == 0: every lane's columns are in the row
// and a warp's strip makes whole mask words.
template <typename T, int BITS, bool AFFINE, bool SR, bool SLOW>
__device__ __forceinline__ void col_map_tile(const char* tile, int nr, uint32_t sb, int cl, int rw,
                                             int nrw, int64_t rs, int64_t cols, int64_t c,
                                             bool active, const ColR (&P)[kColLane<T>],
                                             uint32_t slowm, uint32_t deadm, bool clampsym,
                                             const SrCtx& sr, void* y, void* codes,
                                             uint32_t* mask, int lane) {
  constexpr int NC = kColLane<T>, LPW = 32 / NC;  // LPW: lanes per mask word
  for (int r = rw; r < nr; r += nrw) {
    const int64_t i = (rs + r) * cols + c;
    uint32_t mb = 0u;
    if (active) {
      const uint4 v = *reinterpret_cast<const uint4*>(tile + (size_t)r * sb + cl * T::BYTES);
      const Raw16 cur = {{v.x, v.y, v.z, v.w}};
      mb = col_row<T, BITS, AFFINE, SR, SLOW>(cur, P, slowm, deadm, clampsym, sr, i, y, codes);
    }
    uint32_t w = mb << (NC * (lane & (LPW - 1)));
#pragma unroll
    for (int o = 1; o < LPW; o <<= 1) w |= __shfl_xor_sync(kFull, w, o);
    if (mask && active && (lane & (LPW - 1)) == 0) mask[i / 32] = w;
  }
}

// The calibrated per-column map (cols % 32 == 0): while its first tiles are
// in flight, each lane calibrates its columns from the accumulators and keeps
// their parameters in registers (blocks of the first row chunk write scale,
// zero point and the calibration flags); the rows of the block's strip come
// in through the staged tiles.
template <typename T, int BITS, bool AFFINE, bool SR>
__global__ void __launch_bounds__(256, 2)
    k_int_cols(const void* __restrict__ x, int64_t rows, int64_t cols, int wc, int64_t rchunk,
               int tr, uint32_t wait_limit, const uint4* __restrict__ acc, float* scale,
               int32_t* zp, SrCtx sr, CalOpts co, void* y, void* codes, uint32_t* mask,
               int32_t* flags) {
  constexpr int NC = kColLane<T>, WW = kColStrip<T>;
  constexpr int MM = AFFINE ? kMMKeys : kMMNone;
  extern __shared__ __align__(128) char col_stage[];
  __shared__ __align__(8) uint64_t bars[kColStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = warp & (wc - 1), rw = warp / wc, nrw = kColWarps / wc;
  const int sw = WW * wc;
  ColTiles tl;
  tl.x = static_cast<const char*>(x);
  tl.cols = cols;
  tl.cs = (int64_t)blockIdx.x * sw;
  tl.segc = (int)(cols - tl.cs < sw ? cols - tl.cs : sw);
  tl.contig = tl.segc == cols;
  tl.bytes_per_elem = T::BYTES;
  tl.r0 = (int64_t)blockIdx.y * rchunk;
  tl.r1 = min(rows, tl.r0 + rchunk);
  tl.tr = tr;
  tl.wait_limit = wait_limit;
  tl.tiles = tl.r1 > tl.r0 ? (int)((tl.r1 - tl.r0 + tr - 1) / tr) : 0;
  const int cl = sub * WW + lane * NC;
  const bool active = cl < tl.segc;
  const int64_t c = tl.cs + cl;
  const uint32_t sb = tl.seg_bytes();
  ColR P[NC];
  uint32_t slowm = 0u, deadm = 0u;
  bool slow = false;
  const auto calibrate_columns = [&] {
    pdl_wait();  // launched early: the accumulators come from the statistics kernel
    int f = 0;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      IntParams p;
      p.s = 1.0f;
      p.zp = 0;
      p.dead = 1;
      p.fast = 0;
      p.rcp = 0.0f;
      if (active) {
        f |= calibrate<BITS, AFFINE, MM>(col_acc_stats<MM>(acc[c + j]), p, co);
        // one writer per column (the warps of other row phases share it)
        if (blockIdx.y == 0 && rw == 0) {
          scale[c + j] = p.s;
          if (zp) zp[c + j] = p.zp;
        }
      } else {
        finish_params(p, QRange<BITS, AFFINE>::qmin, QRange<BITS, AFFINE>::qmax);
      }
      const ColP q = col_params<BITS, AFFINE>(p);
      P[j] = ColR{q.s, q.rcp, q.wlo, q.whi, q.klof, q.khif, q.zp};
      slowm |= (q.st & 2) ? 0u : (1u << j);
      deadm |= (q.st & 1) ? (1u << j) : 0u;
    }
    if (!active) slowm = deadm = 0u;
    warp_flag_or(flags, (blockIdx.y == 0 && rw == 0) ? f : 0);
    // a warp with a dead column or a scale outside the reciprocal's safe
    // range also runs the IEEE path for those columns
    slow = __any_sync(kFull, slowm != 0u);
  };
  const bool clampsym = co.clamp || co.clip != 1.0f || co.fp16;
  col_staged(tl, col_stage, bars, flags, calibrate_columns, [&](const char* tile, int t, int nr) {
    const int64_t rs = tl.r0 + (int64_t)t * tr;
    if (slow)
      col_map_tile<T, BITS, AFFINE, SR, true>(tile, nr, sb, cl, rw, nrw, rs, cols, c, active, P,
                                              slowm, deadm, clampsym, sr, y, codes, mask, lane);
    else
      col_map_tile<T, BITS, AFFINE, SR, false>(tile, nr, sb, cl, rw, nrw, rs, cols, c, active, P,
                                               0u, 0u, clampsym, sr, y, codes, mask, lane);
  });
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
constexpr int kColStagedBytes = kColStages * kColStageBytes;

// rows per staged tile of a strip of `sw` columns
static int col_tile_rows(int64_t sw, int bytes) {
  const int64_t tr = kColStageBytes / (sw * bytes);
  return (int)(tr < 1 ? 1 : tr);
}

// The dynamic shared memory of a staged kernel, raised once per kernel and
// device (a failure shows as a launch error).
template <auto Kernel>
static void col_staged_smem() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 63;
  const uint64_t bit = uint64_t{1} << dev;
  if (done.load(std::memory_order_acquire) & bit) return;
  if (cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kColStagedBytes) == cudaSuccess)
    done.fetch_or(bit, std::memory_order_acq_rel);
}

#if !QAT_SR
template <typename T>
static void col_stats_t(bool keys, const void* x, int64_t rows, int64_t cols, uint4* acc,
                        int32_t* flags, cudaStream_t s) {
  const bool staged = cols % 32 == 0;
  // one wave: 2 staged blocks per SM (shared memory), else 3 (registers)
  const ColShape g = col_shape(rows, cols, kColStrip<T>, staged ? 2 : 3, 8, 1);
  const int tr = col_tile_rows((int64_t)kColStrip<T> * g.wc, T::BYTES);
  const uint32_t limit = device_wait_limit();
  k_col_init<<<(unsigned)((cols + 255) / 256), 256, 0, s>>>(acc, cols);
  const dim3 grid((unsigned)g.strips, (unsigned)g.chunks);
#define QAT_CS(M)                                                                               \
  do {                                                                                          \
    if (staged) {                                                                               \
      col_staged_smem<k_col_stats_staged<T, M>>();                                              \
      launch_kernel(k_col_stats_staged<T, M>, grid, dim3(256), kColStagedBytes, s, true, x, rows, \
                    cols, g.wc, g.rchunk, tr, limit, acc, flags);                               \
    } else {                                                                                    \
      launch_kernel(k_col_stats<T, M>, grid, dim3(256), 0, s, true, x, rows, cols, g.wc,        \
                    g.rchunk, acc);                                                             \
    }                                                                                           \
  } while (0)
  if (keys) QAT_CS(kMMKeys);
  else QAT_CS(kMMNone);
#undef QAT_CS
}

qat_status launch_col_stats(qat_dtype dt, bool keys, const void* x, int64_t rows, int64_t cols,
                            void* ws, int32_t* flags, cudaStream_t s) {
  uint4* acc = col_ws(ws, cols).acc;
  if (dt == QAT_F32)
    col_stats_t<F32>(keys, x, rows, cols, acc, flags, s);
  else
    col_stats_t<BF16>(keys, x, rows, cols, acc, flags, s);
  count_launch(2);
  return launch_status();
}

qat_status launch_col_finalize(int mode, int bits, bool affine, void* ws, int64_t cols, float* out0,
                               float* out1, float* out2, int32_t* zp, const CalOpts& co,
                               int32_t* flags, cudaStream_t s) {
  const ColWs w = col_ws(ws, cols);
  const unsigned g = (unsigned)((cols + 255) / 256);
#define QAT_CF(M, B, A)                                                                        \
  launch_kernel(k_col_finalize<M, B, A>, dim3(g), dim3(256), 0, s, true, w.acc, cols, out0, out1, \
                out2, zp, w.dead, co, flags)
  if (mode == 0) QAT_CF(0, 8, false);
  else if (bits == 8) { if (affine) QAT_CF(1, 8, true); else QAT_CF(1, 8, false); }
  else { if (affine) QAT_CF(1, 4, true); else QAT_CF(1, 4, false); }
#undef QAT_CF
  count_launch(1);
  return launch_status();
}
#endif  // !QAT_SR

template <typename T, int BITS, bool AFFINE>
static void int_cols_t(const void* x, int64_t rows, int64_t cols, const uint4* acc, float* scale,
                       int32_t* zp, const SrCtx& sr, const CalOpts& co, void* y, void* codes,
                       uint32_t* mask, int32_t* flags, cudaStream_t s) {
  // one wave of 2 blocks per SM (their staged tiles fill the shared memory)
  const ColShape g = col_shape(rows, cols, kColStrip<T>, 2, 8, 1);
  const int tr = col_tile_rows((int64_t)kColStrip<T> * g.wc, T::BYTES);
  const dim3 grid((unsigned)g.strips, (unsigned)g.chunks);
  col_staged_smem<k_int_cols<T, BITS, AFFINE, QAT_SR>>();
  launch_kernel(k_int_cols<T, BITS, AFFINE, QAT_SR>, grid, dim3(256), kColStagedBytes, s, true, x,
                rows, cols, g.wc, g.rchunk, tr, device_wait_limit(), acc, scale, zp, sr, co, y,
                codes, mask, flags);
}

qat_status QAT_SR_NAME(launch_int_cols)(qat_dtype dt, int bits, bool affine, const void* x,
                                        int64_t rows, int64_t cols, const void* ws, float* scale,
                                        int32_t* zp, const SrCtx& sr, const CalOpts& co, void* y,
                                        void* codes, uint32_t* mask, int32_t* flags,
                                        cudaStream_t s) {
  const uint4* acc = col_ws(const_cast<void*>(ws), cols).acc;
#define QAT_IC(T, B, A) \
  int_cols_t<T, B, A>(x, rows, cols, acc, scale, zp, sr, co, y, codes, mask, flags, s)
  if (dt == QAT_F32) {
    if (bits == 8) { if (affine) QAT_IC(F32, 8, true); else QAT_IC(F32, 8, false); }
    else { if (affine) QAT_IC(F32, 4, true); else QAT_IC(F32, 4, false); }
  } else {
    if (bits == 8) { if (affine) QAT_IC(BF16, 8, true); else QAT_IC(BF16, 8, false); }
    else { if (affine) QAT_IC(BF16, 4, true); else QAT_IC(BF16, 4, false); }
  }
#undef QAT_IC
  count_launch(1);
  return launch_status();
}

}  // namespace qat
