// kernels_cols.cu -- per-column (channel axis 1) integer fake quant.
//
// optirs-gpu quantization.rs, per_channel_params / fake_quant_int_per_channel
// with the channel axis along the columns of a row-major [rows, cols] tensor:
// one scale (and zero point) per column, calibrated from that column's
// absmax (symmetric) or min / max (affine) exactly as a row is.
//
// A column's statistics need every row before its first element can be
// mapped, so the calibrated path is two passes over x:
//   k_col_init   the per-column accumulators (16 bytes per column)
//   k_col_stats  a block takes a strip of 128 columns and a chunk of rows;
//                each lane folds 4 consecutive columns down its rows, the
//                block merges its 8 warps in shared memory and combines into
//                the accumulators with integer atomics (the absmax bits and
//                order keys are monotone as unsigned integers)
//   k_int_cols   the same strips: the block calibrates its 128 columns into
//                shared memory, each lane keeps the parameters of its 4
//                columns in registers and maps its rows
// The second read of x hits L2 when the tensor fits in it.  Shapes whose
// row length is not a multiple of 32 (mask words would straddle rows) and
// given parameters take the per-element unit kernel in column mode.
#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

constexpr int kColStrip = 128;  // columns per block strip (4 per lane)
constexpr int kColWarps = 8;    // warps per block, one row each at a time

// four consecutive elements of one row as fp32 bits; scalar loads when the
// row length is not a multiple of 4 (unaligned rows) or at the row's end
template <typename T>
__device__ __forceinline__ void load4(const void* x, int64_t i, int have, bool vec,
                                      uint32_t (&b)[4]) {
  if (vec && have >= 4) {
    if (T::BYTES == 4) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const float*>(x) + i));
      b[0] = v.x;
      b[1] = v.y;
      b[2] = v.z;
      b[3] = v.w;
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + i));
      b[0] = v.x << 16;
      b[1] = v.x & 0xffff0000u;
      b[2] = v.y << 16;
      b[3] = v.y & 0xffff0000u;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) b[j] = j < have ? load_elem_bits<T>(x, i + j) : 0u;
}

#if !QAT_SR
__global__ void k_col_init(uint4* __restrict__ acc, int64_t cols) {
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c < cols) acc[c] = make_uint4(0u, 0u, kKeyPosInf, kKeyNegInf);
}

// MM: kMMNone (absmax and the non-finite bit) or kMMKeys (also min / max)
template <typename T, int MM>
__global__ void __launch_bounds__(256) k_col_stats(const void* __restrict__ x, int64_t rows,
                                                   int64_t cols, int64_t rchunk,
                                                   uint4* __restrict__ acc) {
  __shared__ uint4 red[kColWarps][kColStrip];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * kColStrip + lane * 4;
  const bool vec = (cols & 3) == 0;
  const int have = c < cols ? (cols - c >= 4 ? 4 : (int)(cols - c)) : 0;
  Stats st[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) st[j].init<MM>();
  const int64_t r0 = (int64_t)blockIdx.y * rchunk;
  const int64_t r1 = min(rows, r0 + rchunk);
  if (have > 0) {
    // four rows per step, their loads issued before the folds
    for (int64_t r = r0 + warp; r < r1; r += 4 * kColWarps) {
      uint32_t b[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t rk = r + k * kColWarps;
        if (rk < r1) load4<T>(x, rk * cols + c, have, vec, b[k]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (r + k * kColWarps < r1) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j < have) st[j].add<MM>(b[k][j]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) red[warp][lane * 4 + j] = st[j].pack();
  __syncthreads();
  if (threadIdx.x < kColStrip) {
    const int64_t col = (int64_t)blockIdx.x * kColStrip + threadIdx.x;
    if (col < cols) {
      Stats s;
      s.unpack(red[0][threadIdx.x]);
#pragma unroll
      for (int w = 1; w < kColWarps; ++w) {
        Stats o;
        o.unpack(red[w][threadIdx.x]);
        s.merge<MM>(o);
      }
      uint32_t* a = reinterpret_cast<uint32_t*>(acc + col);
      atomicMax(a + 0, s.amax);
      if (s.nonfinite) atomicOr(a + 1, 1u);
      if (MM == kMMKeys) {
        atomicMin(a + 2, s.kmin);
        atomicMax(a + 3, s.kmax);
      }
    }
  }
}

// accumulators -> per-column absmax / min / max and the non-finite flag
__global__ void k_col_finalize(const uint4* __restrict__ acc, int64_t cols, float* absmax,
                               float* minv, float* maxv, int32_t* flags) {
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int f = 0;
  if (c < cols) {
    Stats s;
    s.unpack(acc[c]);
    if (absmax) absmax[c] = s.absmax_f();
    if (minv) minv[c] = s.min_f<kMMKeys>();
    if (maxv) maxv[c] = s.max_f<kMMKeys>();
    f = s.has_nonfinite() ? QAT_FLAG_NONFINITE_INPUT : 0;
  }
  warp_flag_or(flags, f);
}

// accumulators -> scale, zero point and the dead byte of every column (the
// unit-kernel fallback)
template <int BITS, bool AFFINE>
__global__ void k_col_params(const uint4* __restrict__ acc, int64_t cols, float* scale,
                             int32_t* zp, uint8_t* dead, int32_t* flags) {
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int f = 0;
  if (c < cols) {
    Stats s;
    s.unpack(acc[c]);
    IntParams p;
    f = calibrate<BITS, AFFINE, kMMKeys>(s, p);
    scale[c] = p.s;
    if (zp) zp[c] = p.zp;
    dead[c] = (uint8_t)p.dead;
  }
  warp_flag_or(flags, f);
}
#endif  // !QAT_SR

// ---------------------------------------------------------------------------
// the calibrated per-column map
// ---------------------------------------------------------------------------
// The parameters of one column as the map keeps them (32 bytes in shared
// memory): wlo is stored as -0 when it is zero (the window test below).
struct ColP {
  float s, rcp, wlo, whi, klof, khif;
  int zp;
  int st;  // bit 0 dead, bit 1 fast (scale in the reciprocal's safe range)
};

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
  q.st = (p.dead ? 1 : 0) | (p.fast ? 2 : 0);
  return q;
}

// The IEEE-division path of one element of a calibrated column that is dead
// or has a scale outside the reciprocal's safe range.
template <int BITS, bool AFFINE, bool SR>
__device__ __forceinline__ void col_slow_elem(float x, float u, const ColP& c, float& y, int& q,
                                              uint32_t& m) {
  constexpr int qmin = QRange<BITS, AFFINE>::qmin, qmax = QRange<BITS, AFFINE>::qmax;
  if (c.st & 1) {
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
// or the stochastic rounding with draws ua, ub, the clamp (affine, and every
// stochastic rounding), y = k s, the code from the bits of k + M, and the
// out-of-window sign bits (whi - |x| symmetric; whi - x, x - wlo affine).
template <bool AFFINE, bool SR>
__device__ __forceinline__ void col_pair(float xa, float xb, const ColP& a, const ColP& b,
                                         float ua, float ub, float& ya, float& yb, int& qa,
                                         int& qb, uint32_t& oa, uint32_t& ob) {
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
    if (AFFINE) {
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

// One row of a lane's four columns: map, store y and the codes, return the
// four mask bits (bit j = column j).
template <typename T, int BITS, bool AFFINE, bool SR>
__device__ __forceinline__ uint32_t col_row(const uint32_t (&b)[4], const ColP (&P)[4], bool slow,
                                            const SrCtx& sr, int64_t i, void* y, void* codes) {
  float u[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (SR) sr_draws4(sr, i / 4, u);
  float yv[4];
  int q[4];
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; j += 2)
    col_pair<AFFINE, SR>(__uint_as_float(b[j]), __uint_as_float(b[j + 1]), P[j], P[j + 1], u[j],
                         u[j + 1], yv[j], yv[j + 1], q[j], q[j + 1], o[j], o[j + 1]);
  uint32_t mb = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) mb |= (o[j] ^ 1u) << j;
  if (slow) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!(P[j].st & 2)) {
        uint32_t m;
        col_slow_elem<BITS, AFFINE, SR>(__uint_as_float(b[j]), u[j], P[j], yv[j], q[j], m);
        mb = (mb & ~(1u << j)) | (m << j);
      }
    }
  }
  if (y) {
    if (T::BYTES == 4)
      *reinterpret_cast<uint4*>(static_cast<float*>(y) + i) =
          make_uint4(__float_as_uint(yv[0]), __float_as_uint(yv[1]), __float_as_uint(yv[2]),
                     __float_as_uint(yv[3]));
    else
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + i) =
          make_uint2(pack_bf16x2(yv[0], yv[1]), pack_bf16x2(yv[2], yv[3]));
  }
  if (codes) {
    if (BITS == 8)
      *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(codes) + i) =
          (uint32_t)(q[0] & 0xff) | ((uint32_t)(q[1] & 0xff) << 8) |
          ((uint32_t)(q[2] & 0xff) << 16) | ((uint32_t)(q[3] & 0xff) << 24);
    else  // element 2j in the high nibble of byte j
      *reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(codes) + i / 2) =
          (uint16_t)(((q[0] & 0xf) << 4) | (q[1] & 0xf) | ((q[2] & 0xf) << 12) |
                     ((q[3] & 0xf) << 8));
  }
  return mb;
}

// Requires cols % 32 == 0: every lane's four columns are in the row and a
// warp's 128 columns make four whole mask words.
template <typename T, int BITS, bool AFFINE, bool SR>
__global__ void __launch_bounds__(256) k_int_cols(const void* __restrict__ x, int64_t rows,
                                                  int64_t cols, int64_t rchunk,
                                                  const uint4* __restrict__ acc, float* scale,
                                                  int32_t* zp, SrCtx sr, void* y, void* codes,
                                                  uint32_t* mask, int32_t* flags) {
  __shared__ ColP sp[kColStrip];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t cb = (int64_t)blockIdx.x * kColStrip;
  int f = 0;
  if (threadIdx.x < kColStrip) {
    const int64_t col = cb + threadIdx.x;
    IntParams p;
    p.s = 1.0f;
    p.zp = 0;
    p.dead = 1;
    p.fast = 0;
    p.rcp = 0.0f;
    if (col < cols) {
      Stats s;
      s.unpack(acc[col]);
      f = calibrate<BITS, AFFINE, kMMKeys>(s, p);
      if (blockIdx.y == 0) {
        scale[col] = p.s;
        if (zp) zp[col] = p.zp;
      } else {
        f = 0;
      }
    } else {
      finish_params(p, QRange<BITS, AFFINE>::qmin, QRange<BITS, AFFINE>::qmax);
    }
    sp[threadIdx.x] = col_params<BITS, AFFINE>(p);
  }
  warp_flag_or(flags, f);
  __syncthreads();
  const int64_t c = cb + lane * 4;
  const bool active = c < cols;
  ColP P[4];
  bool slow = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    P[j] = sp[lane * 4 + j];
    slow |= !(P[j].st & 2);
  }
  const int64_t r0 = (int64_t)blockIdx.y * rchunk;
  const int64_t r1 = min(rows, r0 + rchunk);
  // two rows per step, both loads issued first; the row loop is warp-uniform
  // (the mask words are assembled with shuffles)
  for (int64_t r = r0 + warp; r < r1; r += 2 * kColWarps) {
    const int64_t rb = r + kColWarps;
    const bool hb = rb < r1;
    uint32_t b0[4], b1[4];
    if (active) {
      load4<T>(x, r * cols + c, 4, true, b0);
      if (hb) load4<T>(x, rb * cols + c, 4, true, b1);
    }
    uint32_t m0 = 0u, m1 = 0u;
    if (active) {
      m0 = col_row<T, BITS, AFFINE, SR>(b0, P, slow, sr, r * cols + c, y, codes);
      if (hb) m1 = col_row<T, BITS, AFFINE, SR>(b1, P, slow, sr, rb * cols + c, y, codes);
    }
    // mask word k of the warp's 128 columns: lanes 8k .. 8k + 7, 4 bits each
    uint32_t w0 = m0 << (4 * (lane & 7)), w1 = m1 << (4 * (lane & 7));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      w0 |= __shfl_xor_sync(kFull, w0, o);
      w1 |= __shfl_xor_sync(kFull, w1, o);
    }
    if (mask && active && (lane & 7) == 0) {
      mask[(r * cols + c) / 32] = w0;
      if (hb) mask[(rb * cols + c) / 32] = w1;
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
// Row chunks per column strip: about `per_sm` blocks per SM in all, each
// chunk at least `min_rows` rows.
static int64_t col_chunk(int64_t rows, int64_t cols, int per_sm, int64_t min_rows) {
  const int64_t strips = (cols + kColStrip - 1) / kColStrip;
  int64_t want = ((int64_t)device_info().sms * per_sm + strips - 1) / strips;
  int64_t most = (rows + min_rows - 1) / min_rows;
  int64_t chunks = want < most ? want : most;
  if (chunks < 1) chunks = 1;
  if (chunks > 65535) chunks = 65535;
  return (rows + chunks - 1) / chunks;
}

#if !QAT_SR
qat_status launch_col_stats(qat_dtype dt, const void* x, int64_t rows, int64_t cols, int mm,
                            void* ws, cudaStream_t s) {
  uint4* acc = static_cast<uint4*>(ws);
  k_col_init<<<(unsigned)((cols + 255) / 256), 256, 0, s>>>(acc, cols);
  const int64_t rchunk = col_chunk(rows, cols, 8, 32);
  const dim3 grid((unsigned)((cols + kColStrip - 1) / kColStrip),
                  (unsigned)((rows + rchunk - 1) / rchunk));
#define QAT_CS(T, M) k_col_stats<T, M><<<grid, 256, 0, s>>>(x, rows, cols, rchunk, acc)
  if (dt == QAT_F32) {
    if (mm == kMMKeys) QAT_CS(F32, kMMKeys); else QAT_CS(F32, kMMNone);
  } else {
    if (mm == kMMKeys) QAT_CS(BF16, kMMKeys); else QAT_CS(BF16, kMMNone);
  }
#undef QAT_CS
  count_launch(2);
  return launch_status();
}

qat_status launch_col_finalize(const void* ws, int64_t cols, float* absmax, float* minv,
                               float* maxv, int32_t* flags, cudaStream_t s) {
  k_col_finalize<<<(unsigned)((cols + 255) / 256), 256, 0, s>>>(static_cast<const uint4*>(ws), cols,
                                                                absmax, minv, maxv, flags);
  count_launch(1);
  return launch_status();
}

qat_status launch_col_params(int bits, bool affine, const void* ws, int64_t cols, float* scale,
                             int32_t* zp, uint8_t* dead, int32_t* flags, cudaStream_t s) {
  const uint4* acc = static_cast<const uint4*>(ws);
  const unsigned g = (unsigned)((cols + 255) / 256);
  if (bits == 8) {
    if (affine) k_col_params<8, true><<<g, 256, 0, s>>>(acc, cols, scale, zp, dead, flags);
    else k_col_params<8, false><<<g, 256, 0, s>>>(acc, cols, scale, zp, dead, flags);
  } else {
    if (affine) k_col_params<4, true><<<g, 256, 0, s>>>(acc, cols, scale, zp, dead, flags);
    else k_col_params<4, false><<<g, 256, 0, s>>>(acc, cols, scale, zp, dead, flags);
  }
  count_launch(1);
  return launch_status();
}
#endif  // !QAT_SR

qat_status QAT_SR_NAME(launch_int_cols)(qat_dtype dt, int bits, bool affine, const void* x,
                                        int64_t rows, int64_t cols, const void* ws, float* scale,
                                        int32_t* zp, const SrCtx& sr, void* y, void* codes,
                                        uint32_t* mask, int32_t* flags, cudaStream_t s) {
  const uint4* acc = static_cast<const uint4*>(ws);
  const int64_t rchunk = col_chunk(rows, cols, 6, 64);
  const dim3 grid((unsigned)((cols + kColStrip - 1) / kColStrip),
                  (unsigned)((rows + rchunk - 1) / rchunk));
#define QAT_IC(T, B, A)                                                                       \
  k_int_cols<T, B, A, QAT_SR><<<grid, 256, 0, s>>>(x, rows, cols, rchunk, acc, scale, zp, sr, y, \
                                                   codes, mask, flags)
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
