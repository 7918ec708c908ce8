// kernels_onchip.cu -- per-tensor integer fake quant of a tensor that fits in
// the registers of the whole GPU, in one launch.
//
// optirs-gpu quantization.rs: per_tensor_minmax (the tensor's absmax, or its
// min and max, over finite values), QuantParams::from_absmax / from_minmax,
// then quantize / dequantize and the fake_quant_backward window for every
// element.  The calibration needs every element before the first one can be
// mapped; for a tensor larger than on-chip storage that is two passes over x
// (k_stats_tensor, then k_int_tensor).  Here each thread loads its vectors of
// x once and keeps them in registers: the blocks publish partial statistics,
// meet at a grid-wide barrier (a cooperative launch, so every block is
// resident), each block reduces all partials (max / min are exact and
// order-free, so every block gets the same bits) and calibrates, then maps
// the vectors it holds.  One read of x, one launch.
//
// The barrier is an arrival counter in the caller's workspace, cleared by the
// launcher just before the kernel.  Its wait is bounded: a block whose wait
// runs out sets QAT_FLAG_DEVICE_TIMEOUT and returns without writing outputs.
#include <atomic>

#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

constexpr int kOnchipThreads = 512;
// the partials take workspace slots [0, blocks); the barrier counter the last
// slot of the per-tensor workspace
constexpr int kOnchipBarrierSlot = kMaxPartials - 1;
constexpr int kOnchipMaxBlocks = kMaxPartials - 1;
// larger tensors do not fit the registers of a current GPU at 4 vectors per
// thread; the exact bound is the resident-block check of the launcher
constexpr int64_t kOnchipMaxElems = INT64_C(1) << 26;

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One vector of a calibrated unit (plain calibration: fast is 0 or 1); FULL
// == false: elements e >= cnt are absent and get no code and no mask bit.
template <typename T, int BITS, bool AFFINE, bool FULL>
__device__ __forceinline__ void onchip_vec(const V32& v, const IntParams& p, int cnt, OutVec<T>& ov,
                                           CodeVec<BITS, T::VEC>& cv, uint32_t& mb) {
  constexpr int VEC = T::VEC;
  cv.clear();
  mb = 0u;
  if (p.fast) {
    int_vec_cal<T, BITS, AFFINE, FULL>(v, p, cnt, ov, cv, mb);
  } else if (!p.dead) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      int q;
      float yv;
      uint32_t m;
      int_elem<false>(elem<T>(v, e), p, q, yv, m);
      ov.set(e, yv);
      if (FULL || e < cnt) cv.set(e, q);
      mb |= m << e;
    }
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) ov.set(e, 0.0f);
  }
  if (!FULL) mb &= cnt >= 32 ? 0xffffffffu : ((1u << cnt) - 1u);
}

// NV vectors of VEC elements per thread; vector k of the tensor is held by
// thread k % (grid * blockDim) of the grid, in slot k / (grid * blockDim), so
// a warp's loads and stores are contiguous.  part: gridDim.x partials;
// arrive: the barrier counter (zero at launch).
template <typename T, int BITS, bool AFFINE, int NV>
__global__ void __launch_bounds__(kOnchipThreads)
    k_int_tensor_onchip(const void* __restrict__ x, int64_t n, uint4* __restrict__ part,
                        uint32_t* __restrict__ arrive, uint32_t wait_limit, float* scale,
                        int32_t* zp, void* __restrict__ y, void* __restrict__ codes,
                        uint32_t* __restrict__ mask, int32_t* flags) {
  constexpr int VEC = T::VEC, LPW = 32 / VEC;
  constexpr int MM = AFFINE ? kMMFloat : kMMNone;
  __shared__ __align__(16) uint32_t red[4 * (kOnchipThreads / 32)];
  __shared__ IntParams sp;
  __shared__ int timed_out;
  const int lane = threadIdx.x & 31;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  V32 v[NV];
  int cnt[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int64_t base = (t0 + j * nthr) * VEC;
    const int64_t c = n - base;
    cnt[j] = c >= VEC ? VEC : (c > 0 ? (int)c : 0);
    v[j] = load_vec<T>(x, cnt[j] > 0 ? base : 0, cnt[j]);
  }
  // absent elements read +0, which leaves the absmax and min(m, 0) /
  // max(M, 0) of the affine calibration unchanged
  Stats st;
  st.init<MM>();
#pragma unroll
  for (int j = 0; j < NV; ++j)
    if (cnt[j] > 0) stats_add_vec<T, MM>(st, v[j]);
  const Stats b = block_reduce_stats<MM>(st, red);
  if (threadIdx.x == 0) {
    part[blockIdx.x] = b.pack();
    __threadfence();
    atomicAdd(arrive, 1u);
    int ok = 0;
    for (uint32_t i = 0; i < wait_limit; ++i) {
      if (ld_acquire_gpu(arrive) >= gridDim.x) {
        ok = 1;
        break;
      }
      __nanosleep(8);
    }
    timed_out = !ok;
    if (!ok && flags) atomicOr(flags, QAT_FLAG_DEVICE_TIMEOUT);
  }
  __syncthreads();
  if (timed_out) return;
  // every block: all partials (from L2), one calibration
  Stats s;
  s.init<MM>();
  for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) {
    Stats o;
    o.unpack(__ldcg(part + i));
    s.merge<MM>(o);
  }
  s = block_reduce_stats<MM>(s, red);
  if (threadIdx.x == 0) {
    IntParams q;
    const int f = calibrate<BITS, AFFINE, MM>(s, q);
    sp = q;
    if (blockIdx.x == 0) {
      scale[0] = q.s;
      if (zp) zp[0] = q.zp;
      flag_or(flags, f);
    }
  }
  __syncthreads();
  const IntParams p = sp;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int64_t base = (t0 + j * nthr) * VEC;
    OutVec<T> ov;
    CodeVec<BITS, VEC> cv;
    uint32_t mb;
    if (cnt[j] == VEC)
      onchip_vec<T, BITS, AFFINE, true>(v[j], p, VEC, ov, cv, mb);
    else
      onchip_vec<T, BITS, AFFINE, false>(v[j], p, cnt[j], ov, cv, mb);
    if (cnt[j] > 0) {
      if (y) store_vec<T>(y, base, ov.v, cnt[j]);
      if (codes) cv.store(codes, base, cnt[j]);
    }
    // the LPW lanes of a mask word hold consecutive vectors; the first one
    // stores the word when it is inside the tensor
    const uint32_t w = mask_word_of_slot<VEC>(mb, lane);
    if (mask && (lane % LPW) == 0 && cnt[j] > 0) mask[base >> 5] = w;
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
// Resident blocks per SM of one instantiation, looked up once per device.
template <auto Kernel>
static int onchip_occupancy() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];  // 0 = unknown, -1 = none
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  int occ = dev < kMaxDev ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (occ == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, Kernel, kOnchipThreads, 0) !=
            cudaSuccess ||
        occ <= 0) {
      cudaGetLastError();
      occ = -1;
    }
    if (dev < kMaxDev) cache[dev].store(occ, std::memory_order_relaxed);
  }
  return occ;
}

// Launches with NV vectors per thread when the tensor then takes at most
// `per_sm` blocks per SM (0: as many as are resident).
template <typename T, int BITS, bool AFFINE, int NV>
static qat_status onchip_launch(const void* x, int64_t n, void* ws, float* scale, int32_t* zp,
                                void* y, void* codes, uint32_t* mask, int32_t* flags,
                                cudaStream_t s, int per_sm, bool* done) {
  constexpr auto K = k_int_tensor_onchip<T, BITS, AFFINE, NV>;
  const int occ = onchip_occupancy<K>();
  if (occ <= 0) return QAT_OK;
  const int64_t per_block = (int64_t)kOnchipThreads * NV * T::VEC;
  const int64_t blocks = (n + per_block - 1) / per_block;
  const int64_t cap = (int64_t)(per_sm > 0 && per_sm < occ ? per_sm : occ) * device_info().sms;
  if (blocks > cap || blocks > kOnchipMaxBlocks) return QAT_OK;
  uint4* part = static_cast<uint4*>(ws);
  uint32_t* arrive = reinterpret_cast<uint32_t*>(part + kOnchipBarrierSlot);
  if (cudaMemsetAsync(arrive, 0, sizeof(uint4), s) != cudaSuccess) return QAT_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kOnchipThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint32_t limit = device_wait_limit();
  if (cudaLaunchKernelEx(&cfg, K, x, n, part, arrive, limit, scale, zp, y, codes, mask, flags) !=
      cudaSuccess) {
    cudaGetLastError();
    return QAT_ERR_CUDA;
  }
  *done = true;
  count_launch(1);
  return QAT_OK;
}

template <typename T, int BITS, bool AFFINE>
static qat_status onchip_t(const void* x, int64_t n, void* ws, float* scale, int32_t* zp, void* y,
                           void* codes, uint32_t* mask, int32_t* flags, cudaStream_t s,
                           bool* done) {
  // the fewest vectors per thread with at most one block per SM (the barrier
  // waits for the slowest block, and a second block on an SM is one), else
  // four vectors per thread with every resident block
  qat_status st = onchip_launch<T, BITS, AFFINE, 1>(x, n, ws, scale, zp, y, codes, mask, flags, s,
                                                    1, done);
  if (st || *done) return st;
  st = onchip_launch<T, BITS, AFFINE, 2>(x, n, ws, scale, zp, y, codes, mask, flags, s, 1, done);
  if (st || *done) return st;
  return onchip_launch<T, BITS, AFFINE, 4>(x, n, ws, scale, zp, y, codes, mask, flags, s, 0, done);
}

qat_status launch_int_tensor_onchip(qat_dtype dt, int bits, bool affine, const void* x, int64_t n,
                                    void* ws, float* scale, int32_t* zp, void* y, void* codes,
                                    uint32_t* mask, int32_t* flags, cudaStream_t s, bool* done) {
  *done = false;
  if (n > kOnchipMaxElems) return QAT_OK;
#define QAT_OC(T, B, A) return onchip_t<T, B, A>(x, n, ws, scale, zp, y, codes, mask, flags, s, done)
  if (dt == QAT_F32) {
    if (bits == 8) { if (affine) QAT_OC(F32, 8, true); else QAT_OC(F32, 8, false); }
    else { if (affine) QAT_OC(F32, 4, true); else QAT_OC(F32, 4, false); }
  } else {
    if (bits == 8) { if (affine) QAT_OC(BF16, 8, true); else QAT_OC(BF16, 8, false); }
    else { if (affine) QAT_OC(BF16, 4, true); else QAT_OC(BF16, 4, false); }
  }
#undef QAT_OC
}

}  // namespace qat
