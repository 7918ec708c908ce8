// qat_launch.h -- host-side launchers shared by the library's translation
// units (internal; not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "qat.h"
#include "qat_sr.h"

namespace qat {

// An NVTX range around one C-ABI call, so a profiler's timeline shows which
// entry point issued which kernels (header-only NVTX: without a tool attached
// a push / pop is a check of a function pointer).
struct NvtxScope {
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
  NvtxScope(const NvtxScope&) = delete;
  NvtxScope& operator=(const NvtxScope&) = delete;
};

// Launch a kernel, with programmatic dependent launch when pdl is set: the
// kernel may then be scheduled while the previous kernel of the stream (the
// call's own previous kernel) finishes, and must call pdl_wait() before it
// reads anything that kernel wrote.  Only a call's second and later kernels
// are launched so.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

struct Dev {
  int sms;  // streaming multiprocessors of the current device
};
Dev device_info();           // cached per device
void count_launch(int k);    // diagnostic launch counter
qat_status launch_status();  // QAT_OK or QAT_ERR_CUDA after a <<<>>> launch

// Grid for a per-tensor statistics pass (<= kMaxPartials blocks).
int stats_grid(int64_t n);

// Polls a bounded device wait makes before it gives up (QAT_FLAG_DEVICE_TIMEOUT);
// the default, or the value set by qat_debug_set_wait_limit.
uint32_t device_wait_limit();

// Element-per-lane kernels for tensors aligned to their element but not to
// 32-byte vectors (kernels_unaligned.cu).  ua_stats: per-tensor partials
// (grid blocks) in ws.  ua_int_map mode 0: per tensor calibrated from the
// nparts partials in ws; 1: per tensor given (scale[0], zp[0]); 2: per unit
// (unit = i / L) with arrays calibrated by launch_unit_generic (dead); 3: per
// unit given.  ua_fp8_map: per tensor, calibrated from the partials or given.
qat_status launch_ua_stats(qat_dtype dt, int mm, const void* x, int64_t n, void* ws, int grid,
                           cudaStream_t s);
qat_status launch_ua_int_map(qat_dtype dt, int bits, bool affine, int mode, bool stoch,
                             const void* x, int64_t n, int64_t L, const void* ws, int nparts,
                             float* scale, int32_t* zp, const uint8_t* dead, const SrCtx& sr,
                             const CalOpts& co, void* y, void* codes, uint32_t* mask,
                             int32_t* flags, cudaStream_t s);
qat_status launch_ua_fp8_map(qat_dtype dt, int fmt, bool given, bool stoch, const void* x,
                             int64_t n, const void* ws, int nparts, float* scale, const SrCtx& sr,
                             void* y, uint8_t* codes, uint32_t* mask, int32_t* flags,
                             cudaStream_t s);
qat_status launch_ua_ste(qat_dtype dt, const void* g, int64_t n, const uint32_t* mask, void* dx,
                         cudaStream_t s);

// Calibrated per-tensor integer fake quant (nearest rounding, plain
// calibration) of a tensor that fits in the registers of the resident blocks,
// in one cooperative launch; *done = false (nothing launched) when it does not
// fit.  ws: the per-tensor workspace.
qat_status launch_int_tensor_onchip(qat_dtype dt, int bits, bool affine, const void* x, int64_t n,
                                    void* ws, float* scale, int32_t* zp, void* y, void* codes,
                                    uint32_t* mask, int32_t* flags, cudaStream_t s, bool* done);

// per-tensor statistics -> workspace partials (uint4 per block); mm is the
// min / max mode of Stats (kMMNone, kMMFloat, kMMKeys)
qat_status launch_stats_tensor(qat_dtype dt, const void* x, int64_t n, int mm, void* ws,
                               int grid, cudaStream_t s);
// partials -> absmax / min / max (one thread block)
qat_status launch_stats_finalize(const void* ws, int nparts, float* absmax, float* minv, float* maxv,
                                 int32_t* flags, cudaStream_t s);

// Launchers whose rounding can be stochastic come in two builds: the plain
// name rounds to nearest (sr ignored), the *_sr name rounds stochastically
// with the draws of sr.

// integer fake quant, one parameter set for the whole tensor
#define QAT_DECL_INT_TENSOR(name)                                                               \
  qat_status name(qat_dtype dt, int bits, bool affine, bool given, const void* x, int64_t n,    \
                  const void* ws, int nparts, float* scale, int32_t* zp, const SrCtx& sr,       \
                  const CalOpts& co, void* y, void* codes, uint32_t* mask, int32_t* flags,      \
                  cudaStream_t s, bool pdl)
QAT_DECL_INT_TENSOR(launch_int_tensor);
QAT_DECL_INT_TENSOR(launch_int_tensor_sr);

// integer fake quant with per-unit parameter arrays (unit = i / L, or
// i % ucols for per-column units when ucols > 0)
#define QAT_DECL_INT_UNITS(name)                                                                \
  qat_status name(qat_dtype dt, int bits, bool affine, bool given, const void* x, int64_t n,    \
                  int64_t L, int64_t ucols, const float* scale, const int32_t* zp, const uint8_t* dead,        \
                  const SrCtx& sr, void* y, void* codes, uint32_t* mask, int32_t* flags,        \
                  cudaStream_t s)
QAT_DECL_INT_UNITS(launch_int_units);
QAT_DECL_INT_UNITS(launch_int_units_sr);

// warp-per-unit statistics / calibration for any unit length (fallback)
// mode 0: absmax/minv/maxv outputs; mode 1: int params -> scale, zp, dead
qat_status launch_unit_generic(qat_dtype dt, int mode, int bits, bool affine, const void* x,
                               int64_t units, int64_t L, float* absmax, float* minv, float* maxv,
                               float* scale, int32_t* zp, uint8_t* dead, const CalOpts& co,
                               int32_t* flags, cudaStream_t s);

// fused single-pass per-unit calibration + fake quant (or statistics only)
// for units of L elements.  Returns QAT_ERR_UNSUPPORTED when L does not fit
// either fused kernel (the caller then takes the fallback).
bool fused_units_supported(qat_dtype dt, int64_t L);
#define QAT_DECL_INT_FUSED(name)                                                                \
  qat_status name(qat_dtype dt, int bits, bool affine, bool stats_only, const void* x,          \
                  int64_t units, int64_t L, float* scale, int32_t* zp, float* absmax,           \
                  float* minv, float* maxv, const SrCtx& sr, const CalOpts& co, void* y,        \
                  void* codes, uint32_t* mask, int32_t* flags, cudaStream_t s)
QAT_DECL_INT_FUSED(launch_int_fused);
QAT_DECL_INT_FUSED(launch_int_fused_sr);  // stats_only unsupported

// per-column units of a row-major [rows, cols] tensor.  Workspace layout:
// one 16-byte statistics accumulator per column, then the unit-kernel
// fallback's dead bytes and zero points (each array rounded up to 16 bytes).
struct ColWs {
  uint4* acc;
  uint8_t* dead;
  int32_t* zp;
};
inline int64_t col_r16(int64_t b) { return (b + 15) / 16 * 16; }
inline size_t col_ws_bytes(int64_t cols) {
  return (size_t)(cols * 16 + col_r16(cols) + col_r16(cols * 4));
}
inline ColWs col_ws(void* ws, int64_t cols) {
  char* p = static_cast<char*>(ws);
  ColWs w;
  w.acc = reinterpret_cast<uint4*>(p);
  p += cols * 16;
  w.dead = reinterpret_cast<uint8_t*>(p);
  p += col_r16(cols);
  w.zp = reinterpret_cast<int32_t*>(p);
  return w;
}
// Column statistics into the accumulators (two launches; keys: min / max
// order keys, else the absmax alone).  flags receives
// QAT_FLAG_DEVICE_TIMEOUT if a staged copy wait runs out.
qat_status launch_col_stats(qat_dtype dt, bool keys, const void* x, int64_t rows, int64_t cols,
                            void* ws, int32_t* flags, cudaStream_t s);
// Accumulators -> mode 0: absmax / min / max into out0 / out1 / out2 (each
// nullable) and QAT_FLAG_NONFINITE_INPUT; mode 1: the calibration of the int
// grid (bits, affine): scale into out0, zero points into zp (nullable), the
// dead bytes into the workspace, the calibration flags.
qat_status launch_col_finalize(int mode, int bits, bool affine, void* ws, int64_t cols, float* out0,
                               float* out1, float* out2, int32_t* zp, const CalOpts& co,
                               int32_t* flags, cudaStream_t s);
// The calibrated per-column map (cols % 32 == 0) from the accumulators: it
// calibrates every column itself and writes scale and zero point (nullable)
#define QAT_DECL_INT_COLS(name)                                                                 \
  qat_status name(qat_dtype dt, int bits, bool affine, const void* x, int64_t rows,             \
                  int64_t cols, const void* ws, float* scale, int32_t* zp, const SrCtx& sr,     \
                  const CalOpts& co, void* y, void* codes, uint32_t* mask, int32_t* flags,      \
                  cudaStream_t s)
QAT_DECL_INT_COLS(launch_int_cols);
QAT_DECL_INT_COLS(launch_int_cols_sr);

// Percentile calibration of a whole tensor (radix select of the two
// nearest-rank quantiles): leaves at offset 0 of the workspace the one
// statistics partial the per-tensor map calibrates from (absmax, or min and
// max, of the quantiles; the non-finite bit).  pct_ws_bytes: its workspace.
size_t pct_ws_bytes();
qat_status launch_percentile(qat_dtype dt, const void* x, int64_t n, bool affine,
                             unsigned long long rank_lo, unsigned long long rank_hi, void* ws,
                             cudaStream_t s);

// block-scaled floating point (fmt: qat_elem_format, kind: qat_block_scale,
// block 16 or 32); ws / nparts: the tensor statistics partials (E4M3 kind)
qat_status launch_block_fq(qat_dtype dt, int fmt, int kind, int64_t block, const void* x,
                           int64_t n, const void* ws, int nparts, float* tensor_scale, void* y,
                           uint8_t* codes, void* bscales, uint32_t* mask, int32_t* flags,
                           cudaStream_t s);

// FP8
#define QAT_DECL_FP8_TENSOR(name)                                                               \
  qat_status name(qat_dtype dt, qat_fp8_format fmt, bool given, const void* x, int64_t n,       \
                  const void* ws, int nparts, float* scale, const SrCtx& sr, void* y,           \
                  uint8_t* codes, uint32_t* mask, int32_t* flags, cudaStream_t s, bool pdl)
QAT_DECL_FP8_TENSOR(launch_fp8_tensor);
QAT_DECL_FP8_TENSOR(launch_fp8_tensor_sr);

// QAT optimizer step, the master update (binary32 hyper-parameters; omb =
// 1 - beta, lrwd = lr * wd, decay = (wd != 0), bc = the bias corrections)
struct AdamHp {
  float lr, beta1, beta2, eps, omb1, omb2, lrwd, bc1, bc2;
  int decay;
};
// the update of w, m, v in place; with `stats`, one partial of the new w per
// block into ws (min / max mode mm, grid <= kMaxPartials); otherwise block 0
// writes 1.0f to *scale_one when it is not null
qat_status launch_adam(float* w, const float* g, float* m, float* v, int64_t n, const AdamHp& hp,
                       int mm, bool stats, void* ws, int grid, float* scale_one, cudaStream_t s);

// STE backward
qat_status launch_ste(qat_dtype dt, const void* g, int64_t n, const uint32_t* mask, void* dx,
                      cudaStream_t s);

// two-level 4-bit
qat_status launch_q4_quant(const float* x, int64_t n, uint8_t* data, uint8_t* qscales, float* sup,
                           float* y, bool ua, cudaStream_t s);
qat_status launch_q4_dequant(const uint8_t* data, const uint8_t* qscales, const float* sup,
                             int64_t n, float* y, bool ua, cudaStream_t s);

}  // namespace qat
