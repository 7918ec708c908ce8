// kernels_pct.cu -- percentile calibration of a whole tensor.
//
// optirs-gpu quantization.rs, QuantParams::per_tensor_percentile: the values
// in the total order (-0 before +0), the nearest-rank quantiles at ranks
// lo = floor(c * (n - 1)) and hi = min(ceil((1 - c) * (n - 1)), n - 1) (the
// host computes both in binary64 as printed), then from_minmax: symmetric
// from_absmax(max(|lo|, |hi|)), affine the min / max calibration.  A
// non-finite value anywhere is the module's calibration error.
//
// The two order statistics come from a radix select on the order keys of the
// values (monotone unsigned integers, -0 below +0), most significant digit
// first: three passes of 11, 11 and 10 bits.  Each pass reads x (a warp loads
// a whole 1024-element tile at once, as the statistics pass does), histograms
// the digit of the elements whose higher bits match a target's prefix so far
// (one block-wide histogram in shared memory per target, a shared atomic per
// counted element), and the last block of the pass to finish scans the
// histograms, extends each target's prefix by the bin that holds its
// remaining rank and subtracts the counts below it.  After the
// last pass the prefixes are the keys of the two quantiles, and the last block
// writes the one statistics partial the per-tensor map calibrates from.
#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

constexpr int kPctBins = 2048;
constexpr int kPctPasses = 3;
__host__ __device__ constexpr int pct_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__host__ __device__ constexpr int pct_bits(int pass) { return pass == 2 ? 10 : 11; }

struct PctState {
  uint32_t prefix[2];  // known high bits of each target's key
  uint32_t known[2];   // mask of those bits
  unsigned long long rank[2];  // rank within the elements that match the prefix
  uint32_t nonfinite;  // a NaN or Inf was seen
  uint32_t shared;     // the two prefixes are equal (one histogram serves both)
  uint32_t done[4];    // blocks of each pass that have added their counts
};

struct PctWs {
  uint4* part;                 // the statistics partial for the map (offset 0)
  PctState* st;
  unsigned long long* hist;    // [2][kPctBins]
};
static PctWs pct_ws(void* ws) {
  char* p = static_cast<char*>(ws);
  return PctWs{reinterpret_cast<uint4*>(p), reinterpret_cast<PctState*>(p + 64),
               reinterpret_cast<unsigned long long*>(p + 1024)};
}

__global__ void k_pct_init(PctState* st, unsigned long long* hist, unsigned long long rank_lo,
                           unsigned long long rank_hi) {
  pdl_trigger();
  for (int i = threadIdx.x; i < 2 * kPctBins; i += blockDim.x) hist[i] = 0ull;
  if (threadIdx.x == 0) {
    st->prefix[0] = st->prefix[1] = 0u;
    st->known[0] = st->known[1] = 0u;
    st->rank[0] = rank_lo;
    st->rank[1] = rank_hi;
    st->nonfinite = 0u;
    st->shared = 1u;
    for (int p = 0; p < 4; ++p) st->done[p] = 0u;
  }
}

// Inclusive scan of one value per thread over a block of 256 threads.
__device__ __forceinline__ unsigned long long block_scan256(unsigned long long v,
                                                            unsigned long long* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  unsigned long long before = 0ull;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  __syncthreads();
  return v + before;
}

// A target's prefix on the raw bits: after the first pass the known bits hold
// the sign, which fixes the key's flip (order_key: ~u for a negative value,
// u with the sign bit set for a positive one), so (order_key(u) & km) == pf
// exactly when (u & km) == pct_raw_target(pf, km).
__device__ __forceinline__ uint32_t pct_raw_target(uint32_t pf, uint32_t km) {
  return (pf ^ ((pf & 0x80000000u) ? 0x80000000u : 0xffffffffu)) & km;
}

// One vector's elements into the block histograms.  PASS 0 counts every
// element in h0 (both targets share the empty prefix); later passes count the
// elements that match a target's prefix (raw-bit targets rp0 / rp1), one warp
// vote per vector first, so that the usual vector, with no match in the warp,
// costs a masked compare per element.  cnt: the vector's elements present
// (FULL: all of them).
template <typename T, int PASS, bool SHARED, bool FULL>
__device__ __forceinline__ void pct_fold(const V32& v, int cnt, uint32_t rp0, uint32_t km0,
                                         uint32_t rp1, uint32_t km1, uint32_t* h0, uint32_t* h1) {
  constexpr int SHIFT = pct_shift(PASS);
  constexpr uint32_t DMASK = (1u << pct_bits(PASS)) - 1u;
  if (PASS == 0) {
#pragma unroll
    for (int e = 0; e < T::VEC; ++e) {
      const uint32_t bin = (order_key(elem_bits<T>(v, e)) >> SHIFT) & DMASK;
      if (FULL || e < cnt) atomicAdd(h0 + bin, 1u);
    }
    return;
  }
  bool any = false;
#pragma unroll
  for (int e = 0; e < T::VEC; ++e) {
    const uint32_t u = elem_bits<T>(v, e);
    const bool m = (u & km0) == rp0 || (!SHARED && (u & km1) == rp1);
    any |= m && (FULL || e < cnt);
  }
  if (!__any_sync(kFull, any)) return;
#pragma unroll
  for (int e = 0; e < T::VEC; ++e) {
    const uint32_t u = elem_bits<T>(v, e);
    const uint32_t bin = (order_key(u) >> SHIFT) & DMASK;
    if ((FULL || e < cnt) && (u & km0) == rp0) atomicAdd(h0 + bin, 1u);
    if (!SHARED && (FULL || e < cnt) && (u & km1) == rp1) atomicAdd(h1 + bin, 1u);
  }
}

// The block's share of x: warp w takes the 1024-element tiles w, w + W, ...
// (W warps in the grid), each lane loading its SLOTS vectors of a tile at
// once, so a warp has a whole tile in flight (the loop is warp-uniform, for
// the votes).
template <typename T, int PASS, bool SHARED>
__device__ __forceinline__ void pct_walk(const void* __restrict__ x, int64_t n, uint32_t rp0,
                                         uint32_t km0, uint32_t rp1, uint32_t km1, uint32_t* h0,
                                         uint32_t* h1, uint32_t& bad) {
  constexpr int VEC = T::VEC, SLOTS = kTile / (32 * VEC);
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t nfull = n / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  V32 v[SLOTS];
  int cnt[SLOTS];
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < ntiles;
       t += wstride) {
    const bool full = t < nfull;
    if (full)
      tile_load<T, true>(x, n, t, v, cnt, false, lane);
    else
      tile_load<T, false>(x, n, t, v, cnt, false, lane);
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) {
      if (PASS == 0) {
        // a NaN or Inf in the vector (absent elements read +0)
        Stats probe;
        if (probe.vec_absmax_nan<T>(v[j]) >= 0x7f800000u) bad = 1u;
      }
      if (full)
        pct_fold<T, PASS, SHARED, true>(v[j], VEC, rp0, km0, rp1, km1, h0, h1);
      else
        pct_fold<T, PASS, SHARED, false>(v[j], cnt[j], rp0, km0, rp1, km1, h0, h1);
    }
  }
}

// One pass: every block histograms its share of x; the last block to finish
// (a counter per pass) picks each target's bin, extends its prefix, clears the
// histograms and, after the last pass, writes the map's partial.
template <typename T, bool AFFINE, int PASS>
__global__ void __launch_bounds__(256, 4) k_pct_pass(const void* __restrict__ x, int64_t n,
                                                  PctState* st, unsigned long long* hist,
                                                  uint4* part) {
  constexpr int PER = kPctBins / 256;  // bins per thread in the pick
  constexpr int pass = PASS;
  __shared__ uint32_t h[2][kPctBins];
  __shared__ unsigned long long warp_tot[8];
  __shared__ uint32_t pick_bin[2];
  __shared__ unsigned long long pick_below[2];
  __shared__ int last;
  // launched early (after the previous kernel of the call): clear the block
  // histograms and request the warp's first tile into L2 while that kernel
  // finishes, then wait for its state
  for (int i = threadIdx.x; i < 2 * kPctBins; i += blockDim.x) (&h[0][0])[i] = 0u;
  const int lane = threadIdx.x & 31;
  {
    const int64_t t0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t0 * kTile < n) prefetch_tile_l2<T>(x, n, t0, lane);
  }
  pdl_wait();
  __syncthreads();
  const int shift = pct_shift(pass);
  const uint32_t dmask = (1u << pct_bits(pass)) - 1u;
  const uint32_t km0 = st->known[0], km1 = st->known[1];
  const uint32_t rp0 = pct_raw_target(st->prefix[0], km0);
  const uint32_t rp1 = pct_raw_target(st->prefix[1], km1);
  const bool shared = st->shared != 0u;
  uint32_t bad = 0u;
  if (PASS == 0 || shared)
    pct_walk<T, PASS, true>(x, n, rp0, km0, rp1, km1, h[0], h[1], bad);
  else
    pct_walk<T, PASS, false>(x, n, rp0, km0, rp1, km1, h[0], h[1], bad);
  if (pass == 0 && __reduce_or_sync(kFull, bad) && lane == 0) atomicOr(&st->nonfinite, 1u);
  pdl_trigger();  // the next kernel may be scheduled as the blocks finish
  __syncthreads();
  for (int i = threadIdx.x; i < 2 * kPctBins; i += blockDim.x) {
    const uint32_t c = (&h[0][0])[i];
    if (c) atomicAdd(hist + i, (unsigned long long)c);
  }
  // the last block of the pass picks
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&st->done[pass], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int t = 0; t < 2; ++t) {
    const unsigned long long* hh = hist + (shared ? 0 : t) * kPctBins;
    const int b0 = PER * threadIdx.x;
    unsigned long long c[PER], sum = 0ull;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      c[j] = __ldcg(hh + b0 + j);
      sum += c[j];
    }
    const unsigned long long incl = block_scan256(sum, warp_tot);
    unsigned long long below = incl - sum;
    const unsigned long long r = __ldcg(&st->rank[t]);
    if (r >= below && r < incl) {
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        if (r < below + c[j]) {
          pick_bin[t] = (uint32_t)(b0 + j);
          pick_below[t] = below;
          break;
        }
        below += c[j];
      }
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < 2 * kPctBins; i += blockDim.x) hist[i] = 0ull;
  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      st->prefix[t] |= pick_bin[t] << shift;
      st->known[t] |= dmask << shift;
      st->rank[t] -= pick_below[t];
    }
    st->shared = st->prefix[0] == st->prefix[1];
    if (pass == kPctPasses - 1) {
      // the quantiles' values; a non-finite tensor gives the zero interval
      // (the scale written is then 0, as for the module's error)
      const uint32_t nf = __ldcg(&st->nonfinite);
      const float lo = nf ? 0.0f : __uint_as_float(key_to_bits(st->prefix[0]));
      const float hi = nf ? 0.0f : __uint_as_float(key_to_bits(st->prefix[1]));
      const float a = fmaxf(fabsf(lo), fabsf(hi));
      // the per-tensor map's partial: absmax bits (symmetric) or the min and
      // max as float bits (affine), and the non-finite bit
      *part = make_uint4(__float_as_uint(a), nf, AFFINE ? __float_as_uint(lo) : 0u,
                         AFFINE ? __float_as_uint(hi) : 0u);
    }
  }
}

size_t pct_ws_bytes() { return 1024 + 2 * kPctBins * sizeof(unsigned long long); }

qat_status launch_percentile(qat_dtype dt, const void* x, int64_t n, bool affine,
                             unsigned long long rank_lo, unsigned long long rank_hi, void* ws,
                             cudaStream_t s) {
  const PctWs w = pct_ws(ws);
  k_pct_init<<<1, 1024, 0, s>>>(w.st, w.hist, rank_lo, rank_hi);
  const int64_t ntiles = (n + kTile - 1) / kTile;
  int64_t g = (ntiles + 7) / 8;  // at least a tile per warp
  // the resident blocks: 4 per SM (64 registers, 16 KiB of shared memory),
  // every warp with a whole tile in flight
  const int64_t cap = (int64_t)device_info().sms * 4;
  const int grid = (int)(g > cap ? cap : (g < 1 ? 1 : g));
#define QAT_PP(T, A, P)                                                                       \
  launch_kernel(k_pct_pass<T, A, P>, dim3(grid), dim3(256), 0, s, true, x, n, w.st, w.hist, w.part)
#define QAT_PPS(T, A) QAT_PP(T, A, 0); QAT_PP(T, A, 1); QAT_PP(T, A, 2)
  static_assert(kPctPasses == 3, "three radix-select passes");
  if (dt == QAT_F32) {
    if (affine) { QAT_PPS(F32, true); } else { QAT_PPS(F32, false); }
  } else {
    if (affine) { QAT_PPS(BF16, true); } else { QAT_PPS(BF16, false); }
  }
#undef QAT_PPS
#undef QAT_PP
  count_launch(1 + kPctPasses);
  return launch_status();
}

}  // namespace qat
