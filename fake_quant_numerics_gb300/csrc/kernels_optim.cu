// kernels_optim.cu -- the master-weight update of the QAT optimizer step.
//
// optirs-gpu quantization.rs, QatOptimizer::step: per element
//   m = beta1 m + (1 - beta1) g;  v = beta2 v + (1 - beta2) g g;
//   m_hat = m / bc1;  v_hat = v / bc2;
//   w -= lr wd w (when wd != 0, decoupled AdamW);  w -= lr m_hat / (sqrt(v_hat) + eps)
// in binary32, every operation rounded once in the printed order (IEEE
// division and square root), then QatOptimizer::requantize re-derives the
// fake-quant view from the new master.  The view needs the per-tensor
// statistics of the new master before its first element, so the update pass
// also folds them into per-block partials (like k_stats_tensor) and the view
// is the per-tensor map that re-reduces them (k_int_tensor), or for an FP8
// target the unscaled cast (k_fp8_tensor with scale 1, written here).
#include "qat_device.cuh"
#include "qat_launch.h"

namespace qat {

// The Adam step of one element.  Every product that feeds a sum is a scalar
// __fmul_rn: the code generator may fuse a packed mul.rn.f32x2 feeding an
// add.rn.f32x2 into one fused multiply-add (one rounding instead of two),
// which would change the result.
__device__ __forceinline__ void adam_elem(float& w, float g, float& m, float& v, const AdamHp& hp) {
  m = __fadd_rn(__fmul_rn(hp.beta1, m), __fmul_rn(hp.omb1, g));
  v = __fadd_rn(__fmul_rn(hp.beta2, v), __fmul_rn(__fmul_rn(hp.omb2, g), g));
  if (hp.decay) w = __fsub_rn(w, __fmul_rn(hp.lrwd, w));  // decoupled decay
  const float mh = __fdiv_rn(m, hp.bc1), vh = __fdiv_rn(v, hp.bc2);
  const float den = __fadd_rn(__fsqrt_rn(vh), hp.eps);
  w = __fsub_rn(w, __fdiv_rn(__fmul_rn(hp.lr, mh), den));
}

// the Adam step of the 8 fp32 elements of one 32-byte vector
__device__ __forceinline__ void adam_vec(V32& w, const V32& g, V32& m, V32& v, const AdamHp& hp) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float we = __uint_as_float(w.w[e]), me = __uint_as_float(m.w[e]), ve = __uint_as_float(v.w[e]);
    adam_elem(we, __uint_as_float(g.w[e]), me, ve, hp);
    w.w[e] = __float_as_uint(we);
    m.w[e] = __float_as_uint(me);
    v.w[e] = __float_as_uint(ve);
  }
}

// Grid-stride over 1024-element tiles (a warp per tile, 4 vectors per lane);
// STATS folds the new master into one partial per block (min / max mode MM).
template <int MM, bool STATS>
__global__ void __launch_bounds__(512) k_adam(float* __restrict__ w, const float* __restrict__ g,
                                              float* __restrict__ m, float* __restrict__ v,
                                              int64_t n, AdamHp hp, uint4* __restrict__ part,
                                              float* scale_one) {
  __shared__ __align__(16) uint32_t red[4 * 16];
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  Stats st;
  st.init<MM>();
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < ntiles;
       t += wstride) {
#pragma unroll
    for (int j = 0; j < kTile / (32 * 8); ++j) {
      const int64_t base = t * kTile + (int64_t)(j * 32 + lane) * 8;
      const int64_t c = n - base;
      const int cnt = c >= 8 ? 8 : (c > 0 ? (int)c : 0);
      if (cnt == 0) continue;
      V32 wv = load_vec<F32>(w, base, cnt), gv = load_vec<F32>(g, base, cnt);
      V32 mv = load_vec<F32>(m, base, cnt), vv = load_vec<F32>(v, base, cnt);
      adam_vec(wv, gv, mv, vv, hp);
      store_vec<F32>(w, base, wv, cnt);
      store_vec<F32>(m, base, mv, cnt);
      store_vec<F32>(v, base, vv, cnt);
      if (STATS) {
        // absent tail elements count as +0 (the update of zeros can be NaN when
        // eps = 0): a 0 takes no part in absmax and cannot move the affine
        // range, which always includes 0
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e >= cnt) wv.w[e] = 0u;
        stats_add_vec<F32, MM>(st, wv);
      }
    }
  }
  pdl_trigger();  // the view may be scheduled as the blocks finish
  if (STATS) {
    const Stats b = block_reduce_stats<MM>(st, red);
    if (threadIdx.x == 0) part[blockIdx.x] = b.pack();
  } else if (scale_one && blockIdx.x == 0 && threadIdx.x == 0) {
    *scale_one = 1.0f;
  }
}

qat_status launch_adam(float* w, const float* g, float* m, float* v, int64_t n, const AdamHp& hp,
                       int mm, bool stats, void* ws, int grid, float* scale_one, cudaStream_t s) {
  uint4* part = static_cast<uint4*>(ws);
  if (!stats)
    k_adam<kMMNone, false><<<grid, 512, 0, s>>>(w, g, m, v, n, hp, part, scale_one);
  else if (mm == kMMFloat)
    k_adam<kMMFloat, true><<<grid, 512, 0, s>>>(w, g, m, v, n, hp, part, scale_one);
  else
    k_adam<kMMNone, true><<<grid, 512, 0, s>>>(w, g, m, v, n, hp, part, scale_one);
  count_launch(1);
  return launch_status();
}

}  // namespace qat
