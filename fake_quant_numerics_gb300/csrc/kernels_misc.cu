// kernels_misc.cu -- straight-through-estimator backward and the two-level
// 4-bit block format.
//
// STE (optirs-gpu quantization.rs, fake_quant_backward): the incoming
// gradient passes where the forward input lay inside the clamp window and is
// zero elsewhere.  The forward kernels already evaluated the window into a
// packed bit mask, so the backward pass is one read of grad + mask and one
// write of grad_in.
//
// Two-level 4-bit (aprender-train double_quant.rs, quantize_4bit_double,
// reconstruct_scales, dequantize_4bit_double): 64-element absmax blocks with
// 4-bit codes (two per byte, even element in the high nibble) and scale
// absmax / 7; every 256 block scales are re-quantized to uint8 against their
// maximum (the fp32 super-scale, floored at 1e-8).  One thread block handles
// one super-block of 256 * 64 = 16384 elements; the codes never depend on the
// super-scale, so they are written as soon as their block scale is known, and
// only the optional fused round trip waits for the super-scale.
#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

// ---------------------------------------------------------------------------
// STE backward
// ---------------------------------------------------------------------------
template <typename T, bool FULL>
__device__ __forceinline__ void ste_tile(const void* __restrict__ g, int64_t n, int64_t tile,
                                         V32 (&v)[kTile / (32 * T::VEC)], uint32_t& word,
                                         bool have, int64_t next, const uint32_t* __restrict__ mask,
                                         void* __restrict__ dx, int lane) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC), LPW = 32 / VEC;
  const int64_t tb = tile * kTile;
  const int64_t nwords = (n + 31) / 32;
  const int64_t wi = tile * 32 + lane;
  if (!FULL || !have) word = (FULL || wi < nwords) ? __ldg(mask + wi) : 0u;
  int cnt[SLOTS];
  tile_load<T, FULL>(g, n, tile, v, cnt, have, lane);
  const uint32_t cur = word;
  if (next >= 0) word = __ldg(mask + next * 32 + lane);
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) {
    const int64_t base = tb + (int64_t)(j * 32 + lane) * VEC;
    const uint32_t w = __shfl_sync(kFull, cur, j * VEC + lane / LPW);
    const uint32_t bits = (w >> ((lane % LPW) * VEC)) & ((1u << VEC) - 1u);
    V32 o;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t sel;
      if (T::BYTES == 4) {
        sel = ((bits >> k) & 1u) ? 0xffffffffu : 0u;
      } else {
        sel = (((bits >> (2 * k)) & 1u) ? 0x0000ffffu : 0u) |
              (((bits >> (2 * k + 1)) & 1u) ? 0xffff0000u : 0u);
      }
      o.w[k] = v[j].w[k] & sel;
    }
    slot_prefetch<T>(g, next, j, v[j], lane);
    if (cnt[j] > 0) store_vec<T>(dx, base, o, cnt[j]);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) k_ste(const void* __restrict__ g, int64_t n,
                                             const uint32_t* __restrict__ mask, void* dx) {
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t nfull = n / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  V32 v[kTile / (32 * T::VEC)];
  uint32_t word = 0u;
  bool have = false;
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < ntiles;
       t += wstride) {
    const int64_t next = -1;  // no rolling prefetch: occupancy matters more here
    if (t < nfull) ste_tile<T, true>(g, n, t, v, word, have, next, mask, dx, lane);
    else ste_tile<T, false>(g, n, t, v, word, have, next, mask, dx, lane);
    have = next >= 0;
  }
}

qat_status launch_ste(qat_dtype dt, const void* g, int64_t n, const uint32_t* mask, void* dx,
                      cudaStream_t s) {
  const int64_t ntiles = (n + kTile - 1) / kTile;
  int64_t gr = (ntiles + 7) / 8;
  int64_t cap = (int64_t)device_info().sms * 8;
  int grid = (int)(gr > cap ? cap : (gr < 1 ? 1 : gr));
  if (dt == QAT_F32) k_ste<F32><<<grid, 256, 0, s>>>(g, n, mask, dx);
  else k_ste<BF16><<<grid, 256, 0, s>>>(g, n, mask, dx);
  count_launch(1);
  return launch_status();
}

// ---------------------------------------------------------------------------
// two-level 4-bit quantization
// ---------------------------------------------------------------------------
constexpr int kQ4Block = 64;
constexpr int kQ4Super = 256;                       // block scales per super-block
constexpr int kQ4SuperElems = kQ4Block * kQ4Super;  // 16384
constexpr int kQ4Threads = 512;
// each lane holds 16 elements (two 32-byte vectors) of one 64-element block,
// four lanes per block; a thread covers kQ4Pairs such blocks per super-block
constexpr int kQ4Pairs = kQ4SuperElems / (kQ4Threads * 16);  // 2

// code = clamp(round_half_away(x / s), -8, 7); s == 0 or NaN -> 0
__device__ __forceinline__ int q4_code(float x, float s) {
  if (s == 0.0f) return 0;
  float r = roundf(__fdiv_rn(x, s));
  int k = __float2int_rz(r);  // r is integral; NaN -> 0
  return min(max(k, -8), 7);
}

// y = code * rs for the 8 codes of one 32-bit word (element e in byte e / 2,
// even element in the high nibble).  The code k of a nibble u is (u ^ 8) - 8,
// and the float bits 0x4b400000 | (u ^ 8) are the value M + k + 8 with
// M = 1.5 * 2^23, so subtracting M + 8 gives k exactly without an
// integer-to-float conversion; y = RN(k * rs).  A NaN product (only possible
// when rs is inf or NaN: 0 * inf, x * NaN) is written as the canonical quiet
// NaN 0x7fc00000.
__device__ __forceinline__ V32 dequant8(uint32_t packed, float rs) {
  constexpr float kBias = 12582920.0f;  // M + 8
  const uint32_t w = packed ^ 0x88888888u;
  V32 o;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int sh = (e >> 1) * 8;
    const float ta = __uint_as_float(((w >> (sh + 4)) & 0xfu) | 0x4b400000u);
    const float tb = __uint_as_float(((w >> sh) & 0xfu) | 0x4b400000u);
    float ka, kb, ya, yb;
    sub2(ta, tb, kBias, kBias, ka, kb);
    mul2(ka, kb, rs, rs, ya, yb);
    o.w[e] = __float_as_uint(ya);
    o.w[e + 1] = __float_as_uint(yb);
  }
  if (!isfinite(rs)) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (isnan(__uint_as_float(o.w[e]))) o.w[e] = 0x7fc00000u;
  }
  return o;
}

// Level 1 of one lane's 16 elements (block scale s, 4-bit codes in two
// words, element 8h + e of the lane in word h).  For a block scale in the
// safe range the quotient is the IEEE RN(x/s) (quotient_rn2, exact), rounded
// to nearest even by the magic constant; the definition rounds half away from
// zero, so an exact half-integer quotient (and a NaN element, code 0) sends
// the lane through the element-wise code of q4_code.  Absent tail elements
// read +0 and give code 0.
__device__ __forceinline__ void q4_codes16(const V32 (&v)[2], float s, bool has_nan, bool full,
                                           const int (&cnt)[2], uint32_t (&w)[2]) {
  if (quot_scale_ok(s)) {
    const float rcp = __frcp_rn(s), ns = -s;
    bool fix = has_nan;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t pk = 0u;
#pragma unroll
      for (int e = 6; e >= 0; e -= 2) {
        float qa, qb, ta, tb, fa, fb, da, db;
        quotient_rn2(__uint_as_float(v[h].w[e]), __uint_as_float(v[h].w[e + 1]), rcp, ns, qa, qb);
        add2(qa, qb, kRintMagic, kRintMagic, ta, tb);
        sub2(ta, tb, kRintMagic, kRintMagic, fa, fb);
        sub2(qa, qb, fa, fb, da, db);  // exact
        fix |= (fabsf(da) == 0.5f) | (fabsf(db) == 0.5f);
        // |x/s| <= 7 (1 + 2^-23): k = rint(q) in [-7, 7], the low nibble of
        // the two's complement k is the code
        pk = pack_s4x2((int)(__float_as_uint(ta) - kRintMagicBits),
                       (int)(__float_as_uint(tb) - kRintMagicBits), pk);
      }
      w[h] = pk;
    }
    if (fix) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = __uint_as_float(v[h].w[e]);
          const float q = quotient_rn(x, rcp, ns);
          if (isnan(x) || fabsf(__fsub_rn(q, rintf(q))) == 0.5f) {
            const int sh = (e >> 1) * 8 + ((e & 1) ? 0 : 4);
            w[h] = (w[h] & ~(0xfu << sh)) | (((uint32_t)q4_code(x, s) & 0xfu) << sh);
          }
        }
      }
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t pk = 0u;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = (full || e < cnt[h]) ? q4_code(__uint_as_float(v[h].w[e]), s) : 0;
        pk |= ((uint32_t)c & 0xfu) << ((e >> 1) * 8 + ((e & 1) ? 0 : 4));
      }
      w[h] = pk;
    }
  }
}

// UA: x and y hold whole elements but may be off the 32-byte grid (element
// loads and stores, no prefetch of the next super-block)
template <bool ROUNDTRIP, bool UA>
__global__ void __launch_bounds__(kQ4Threads, 2) k_q4_quant(const float* __restrict__ x, int64_t n,
                                                         uint8_t* __restrict__ data,
                                                         uint8_t* __restrict__ qscales,
                                                         float* __restrict__ sup,
                                                         float* __restrict__ y) {
  __shared__ float s_scale[kQ4Super];
  __shared__ float s_q[kQ4Super];
  __shared__ float s_red[kQ4Threads / 32];
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t nsuper = (n + kQ4SuperElems - 1) / kQ4SuperElems;
  const int64_t nblocks = (n + kQ4Block - 1) / kQ4Block;
  const int64_t nbytes = (n + 1) / 2;
  // thread tid, pair j: elements e0 + j * 8192 + 16 tid .. + 15, block
  // j * 128 + tid / 4 of the super-block.  The vectors of the next
  // super-block are requested as soon as the level-1 codes of the current one
  // are computed, so they are in flight while level 2 (two block barriers)
  // and the stores run.
  V32 v[kQ4Pairs][2];
  bool have = false;  // v already holds this super-block (a full one)
  for (int64_t sb = blockIdx.x; sb < nsuper; sb += gridDim.x) {
    const int64_t e0 = sb * kQ4SuperElems;
    const bool full = e0 + kQ4SuperElems <= n;
    int cnt[kQ4Pairs][2];
#pragma unroll
    for (int j = 0; j < kQ4Pairs; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t base = e0 + (int64_t)j * (kQ4Threads * 16) + tid * 16 + h * 8;
        if (full && !UA) {
          cnt[j][h] = 8;
          if (!have) v[j][h] = ld_v32(x + base);
        } else {
          const int64_t c = n - base;
          cnt[j][h] = c >= 8 ? 8 : (c > 0 ? (int)c : 0);
          v[j][h] = load_vec<F32, UA>(x, cnt[j][h] > 0 ? base : 0, cnt[j][h]);
        }
      }
    }
    uint32_t packed[kQ4Pairs][2];
#pragma unroll
    for (int j = 0; j < kQ4Pairs; ++j) {
      // level 1: absmax over the 64-element block = 4 lanes x 16 elements.
      // max.NaN flags a NaN in the lane's elements; the definition's fold
      // (fmaxf: NaN ignored, +inf kept) is then redone element by element.
      float m = 0.0f;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmax_nan(m, fabsf(__uint_as_float(v[j][h].w[e])));
      const bool has_nan = isnan(m);
      if (has_nan) {
        m = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(__uint_as_float(v[j][h].w[e])));
      }
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
      const float s = __fdiv_rn(m, 7.0f);
      q4_codes16(v[j], s, has_nan, full, cnt[j], packed[j]);
      const int64_t base = e0 + (int64_t)j * (kQ4Threads * 16) + tid * 16;
      if (full) {
        *reinterpret_cast<uint2*>(data + base / 2) = make_uint2(packed[j][0], packed[j][1]);
      } else {
#pragma unroll
        for (int b = 0; b < 8; ++b)
          if (base / 2 + b < nbytes) data[base / 2 + b] = (uint8_t)(packed[j][b >> 2] >> (8 * (b & 3)));
      }
      if ((tid & 3) == 0) s_scale[j * (kQ4Threads / 4) + (tid >> 2)] = base < n ? s : 0.0f;
    }
    {
      const int64_t nsb = sb + gridDim.x;
      have = !UA && nsb < nsuper && nsb * kQ4SuperElems + kQ4SuperElems <= n;
      if (have) {
#pragma unroll
        for (int j = 0; j < kQ4Pairs; ++j)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            v[j][h] = ld_v32(x + nsb * kQ4SuperElems + (int64_t)j * (kQ4Threads * 16) + tid * 16 +
                             h * 8);
      }
    }
    __syncthreads();
    // level 2: super = max(max scale, 1e-8); q = clamp(round(scale / super * 255), 0, 255)
    const int64_t b0 = sb * kQ4Super;
    float sc = 0.0f, mm = 0.0f;
    if (tid < kQ4Super) {
      sc = s_scale[tid];
      mm = sc;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFull, mm, o));
    if (lane == 0) s_red[tid >> 5] = mm;
    __syncthreads();
    float mx = 0.0f;
#pragma unroll
    for (int w = 0; w < kQ4Super / 32; ++w) mx = fmaxf(mx, s_red[w]);
    const float super = fmaxf(mx, 1e-8f);
    if (tid < kQ4Super) {
      float r = roundf(__fmul_rn(__fdiv_rn(sc, super), 255.0f));
      int q = __float2int_rz(r);  // NaN (inf / inf) -> 0
      q = min(max(q, 0), 255);
      if (b0 + tid < nblocks) qscales[b0 + tid] = (uint8_t)q;
      s_q[tid] = (float)q;
    }
    if (tid == 0) sup[sb] = super;
    if (ROUNDTRIP) {
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kQ4Pairs; ++j) {
        const float rs =
            __fmul_rn(__fdiv_rn(s_q[j * (kQ4Threads / 4) + (tid >> 2)], 255.0f), super);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const V32 o = dequant8(packed[j][h], rs);
          const int64_t base = e0 + (int64_t)j * (kQ4Threads * 16) + tid * 16 + h * 8;
          if (cnt[j][h] > 0) store_vec<F32, UA>(y, base, o, cnt[j][h]);
        }
      }
    }
    __syncthreads();  // shared arrays are reused by the next super-block
  }
}

qat_status launch_q4_quant(const float* x, int64_t n, uint8_t* data, uint8_t* qscales, float* sup,
                           float* y, bool ua, cudaStream_t s) {
  const int64_t nsuper = (n + kQ4SuperElems - 1) / kQ4SuperElems;
  int64_t cap = (int64_t)device_info().sms * 4;
  int grid = (int)(nsuper > cap ? cap : (nsuper < 1 ? 1 : nsuper));
  if (ua) {
    if (y) k_q4_quant<true, true><<<grid, kQ4Threads, 0, s>>>(x, n, data, qscales, sup, y);
    else k_q4_quant<false, true><<<grid, kQ4Threads, 0, s>>>(x, n, data, qscales, sup, y);
  } else {
    if (y) k_q4_quant<true, false><<<grid, kQ4Threads, 0, s>>>(x, n, data, qscales, sup, y);
    else k_q4_quant<false, false><<<grid, kQ4Threads, 0, s>>>(x, n, data, qscales, sup, y);
  }
  count_launch(1);
  return launch_status();
}

// ---------------------------------------------------------------------------
// two-level 4-bit dequantization: a warp step is 128 octets (1024 elements,
// 16 blocks, inside one super-block); lane l takes octets 32 k + l (k < 4),
// so each 32-byte store instruction of the warp covers 1 KiB of contiguous
// output.  Loads per lane and step: four code words (128 contiguous bytes per
// warp instruction), the step's 16 block scales as one broadcast 16-byte
// load, and the super-scale.  The next step's loads are issued before the
// current step's arithmetic and stores (rolling prefetch).  RN(q / 255)
// comes from a 256-entry table of the same correctly rounded quotients.
// ---------------------------------------------------------------------------
struct Q4Step {
  uint32_t pk[4];
  uint4 q;  // block scales 16 st .. 16 st + 15, byte b of word w = block 16 st + 4 w + b
  float sup;
};

__device__ __forceinline__ void q4_step_full(const uint8_t* __restrict__ data,
                                             const uint8_t* __restrict__ qscales,
                                             const float* __restrict__ sup, int64_t st, int lane,
                                             Q4Step& d) {
  const uint32_t* words = reinterpret_cast<const uint32_t*>(data) + st * 128 + lane;
#pragma unroll
  for (int k = 0; k < 4; ++k) d.pk[k] = __ldg(words + 32 * k);
  d.q = __ldg(reinterpret_cast<const uint4*>(qscales) + st);
  d.sup = __ldg(sup + (st >> 4));
}

// UA: y holds whole elements but may be off the 32-byte grid (element stores)
template <bool UA>
__global__ void __launch_bounds__(256) k_q4_dequant(const uint8_t* __restrict__ data,
                                                    const uint8_t* __restrict__ qscales,
                                                    const float* __restrict__ sup, int64_t n,
                                                    float* __restrict__ y) {
  __shared__ float s_inv255[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) s_inv255[i] = __fdiv_rn((float)i, 255.0f);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t nsteps = (n + 1023) / 1024;
  const int64_t nfull = n / 1024;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  Q4Step cur, nxt;
  bool have = false;
  for (int64_t st = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); st < nsteps;
       st += wstride) {
    if (st >= nfull) {
      // the partial last step: element-wise bounds
      const int64_t nbytes = (n + 1) / 2;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t e0 = (st * 128 + k * 32 + lane) * 8;
        if (e0 >= n) continue;
        uint32_t pk = 0u;
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (e0 / 2 + b < nbytes) pk |= (uint32_t)data[e0 / 2 + b] << (8 * b);
        const float rs = __fmul_rn(s_inv255[qscales[e0 / kQ4Block]], sup[e0 / kQ4SuperElems]);
        const int64_t c = n - e0;
        store_vec<F32, UA>(y, e0, dequant8(pk, rs), c >= 8 ? 8 : (int)c);
      }
      continue;
    }
    if (have)
      cur = nxt;
    else
      q4_step_full(data, qscales, sup, st, lane, cur);
    const int64_t ns = st + wstride;
    have = ns < nfull;
    if (have) q4_step_full(data, qscales, sup, ns, lane, nxt);
    const int qb = 8 * (lane >> 3);  // octet 32 k + l lies in block 16 st + 4 k + l / 8
    const uint32_t qw[4] = {cur.q.x, cur.q.y, cur.q.z, cur.q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float rs = __fmul_rn(s_inv255[(qw[k] >> qb) & 0xffu], cur.sup);
      if (UA)
        store_vec<F32, true>(y, (st * 128 + k * 32 + lane) * 8, dequant8(cur.pk[k], rs), 8);
      else
        st_v32(y + (st * 128 + k * 32 + lane) * 8, dequant8(cur.pk[k], rs));
    }
  }
}

qat_status launch_q4_dequant(const uint8_t* data, const uint8_t* qscales, const float* sup,
                             int64_t n, float* y, bool ua, cudaStream_t s) {
  const int64_t nsteps = (n + 1023) / 1024;
  int64_t g = (nsteps + 7) / 8;
  int64_t cap = (int64_t)device_info().sms * 8;
  int grid = (int)(g > cap ? cap : (g < 1 ? 1 : g));
  if (ua)
    k_q4_dequant<true><<<grid, 256, 0, s>>>(data, qscales, sup, n, y);
  else
    k_q4_dequant<false><<<grid, 256, 0, s>>>(data, qscales, sup, n, y);
  count_launch(1);
  return launch_status();
}

}  // namespace qat
