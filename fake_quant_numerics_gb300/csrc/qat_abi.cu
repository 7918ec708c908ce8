// qat_abi.cu -- the exported C entry points: argument validation, path
// selection and kernel launches.  See include/qat.h for the contract.
#include <atomic>
#include <cstdint>

#include "qat_device.cuh"
#include <cmath>

#include "qat_launch.h"

namespace qat {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int k) { g_launches.fetch_add((uint64_t)k, std::memory_order_relaxed); }

qat_status launch_status() { return cudaGetLastError() == cudaSuccess ? QAT_OK : QAT_ERR_CUDA; }

// bounded device waits: polls before giving up (negative: the default)
constexpr uint32_t kDefaultWaitLimit = 1u << 24;
static std::atomic<int64_t> g_wait_limit{-1};
uint32_t device_wait_limit() {
  const int64_t v = g_wait_limit.load(std::memory_order_relaxed);
  if (v < 0) return kDefaultWaitLimit;
  return v > INT64_C(0xffffffff) ? 0xffffffffu : (uint32_t)v;
}

Dev device_info() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];  // 0 = unknown
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  Dev d{0};
  if (dev < kMaxDev) d.sms = cache[dev].load(std::memory_order_relaxed);
  if (d.sms <= 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      sms = 1;
    d.sms = sms;
    if (dev < kMaxDev) cache[dev].store(sms, std::memory_order_relaxed);
  }
  return d;
}

}  // namespace qat

using namespace qat;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// x, y, grad, grad_in: 32-byte vectors; codes, mask, data, qscales, workspace: 16 bytes
constexpr uintptr_t kAlignVec = 32;
constexpr uintptr_t kAlignBuf = 16;

bool valid_dtype(qat_dtype d) { return d == QAT_F32 || d == QAT_BF16; }

// x, y, grad, grad_in must hold whole elements; off the 32-byte vector grid
// they take the element-per-lane kernels (kernels_unaligned.cu)
bool elem_aligned(const void* p, qat_dtype d) { return aligned(p, d == QAT_F32 ? 4 : 2); }

// number of elements with overflow / sign checks
bool elems(int64_t rows, int64_t cols, int64_t* n) {
  if (rows < 0 || cols < 0) return false;
  if (cols != 0 && rows > (INT64_C(1) << 50) / cols) return false;
  *n = rows * cols;
  return true;
}

// Longest row of a per-column call: the column kernels' grids take one
// block per 128 (statistics, map) or 256 (set-up) columns in x.
constexpr int64_t kMaxColumns = INT64_C(1) << 36;

size_t ws_bytes_for(int64_t rows, int64_t cols, qat_granularity g, int64_t group) {
  if (g == QAT_PER_TENSOR) return (size_t)kMaxPartials * sizeof(uint4);
  int64_t n;
  if (!elems(rows, cols, &n)) return 0;
  const auto r16 = [](int64_t b) { return (b + 15) / 16 * 16; };
  if (g == QAT_PER_COLUMN) return col_ws_bytes(cols);
  int64_t units = 0;
  if (g == QAT_PER_ROW) units = rows;
  else if (g == QAT_PER_GROUP && group > 0) units = n / group;
  return (size_t)(r16(units) + r16(units * 4));
}

// The fallback's per-unit arrays inside the workspace: the dead bytes, then
// the zero points (used when the caller passes no zero-point array).
static uint8_t* ws_dead(void* ws, int64_t cols, qat_granularity g) {
  return g == QAT_PER_COLUMN ? col_ws(ws, cols).dead : static_cast<uint8_t*>(ws);
}
static int32_t* ws_zp(void* ws, int64_t cols, qat_granularity g, int64_t units) {
  return g == QAT_PER_COLUMN ? col_ws(ws, cols).zp
                             : reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) +
                                                          (units + 15) / 16 * 16);
}

// Unit length and count of a granularity; false on an invalid combination.
bool unit_shape(int64_t rows, int64_t cols, qat_granularity g, int64_t group, int64_t* L,
                int64_t* units) {
  int64_t n = rows * cols;
  if (g == QAT_PER_TENSOR) {
    *L = n;
    *units = n > 0 ? 1 : 0;
    return true;
  }
  if (g == QAT_PER_ROW) {
    *L = cols;
    *units = rows;
    return true;
  }
  if (g == QAT_PER_GROUP) {
    if (group <= 0 || cols % group != 0) return false;
    *L = group;
    *units = n / group;
    return true;
  }
  if (g == QAT_PER_COLUMN) {
    *L = rows;
    *units = n > 0 ? cols : 0;
    return true;
  }
  return false;
}

}  // namespace

extern "C" {

const char* qat_status_string(qat_status s) {
  switch (s) {
    case QAT_OK: return "ok";
    case QAT_ERR_INVALID_ARGUMENT: return "invalid argument";
    case QAT_ERR_DIMENSION_MISMATCH: return "dimension mismatch";
    case QAT_ERR_UNSUPPORTED: return "unsupported (bit width, dtype, scheme or format)";
    case QAT_ERR_CUDA: return "CUDA launch failed";
    case QAT_ERR_MISALIGNED: return "misaligned pointer";
    case QAT_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

uint64_t qat_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void qat_debug_set_wait_limit(int64_t polls) {
  g_wait_limit.store(polls, std::memory_order_relaxed);
}

size_t qat_workspace_bytes(int64_t rows, int64_t cols, qat_granularity g, int64_t group) {
  return ws_bytes_for(rows, cols, g, group);
}

qat_status qat_amax_stats(const void* x, qat_dtype dtype, int64_t rows, int64_t cols,
                          qat_granularity g, int64_t group, float* absmax, float* minv, float* maxv,
                          int32_t* flags, void* ws, size_t ws_bytes, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_amax_stats");
  if (!valid_dtype(dtype)) return QAT_ERR_UNSUPPORTED;
  int64_t n, L, units;
  if (!elems(rows, cols, &n)) return QAT_ERR_INVALID_ARGUMENT;
  if (!unit_shape(rows, cols, g, group, &L, &units)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!x) return QAT_ERR_INVALID_ARGUMENT;
  if (!elem_aligned(x, dtype) || (absmax && !aligned(absmax, 4)) || (minv && !aligned(minv, 4)) ||
      (maxv && !aligned(maxv, 4)))
    return QAT_ERR_MISALIGNED;
  const bool ua = !aligned(x, kAlignVec);
  if (ua && g == QAT_PER_COLUMN) return QAT_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (g == QAT_PER_TENSOR) {
    if (!ws || ws_bytes < ws_bytes_for(rows, cols, g, group)) return QAT_ERR_WORKSPACE;
    if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
    int grid = stats_grid(n);
    qat_status st = ua ? launch_ua_stats(dtype, kMMKeys, x, n, ws, grid, s)
                       : launch_stats_tensor(dtype, x, n, kMMKeys, ws, grid, s);
    if (st) return st;
    return launch_stats_finalize(ws, grid, absmax, minv, maxv, flags, s);
  }
  if (g == QAT_PER_COLUMN) {
    if (cols > kMaxColumns) return QAT_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ws_bytes_for(rows, cols, g, group)) return QAT_ERR_WORKSPACE;
    if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
    qat_status st = launch_col_stats(dtype, true, x, rows, cols, ws, flags, s);
    if (st) return st;
    return launch_col_finalize(0, 8, false, ws, cols, absmax, minv, maxv, nullptr, kCalPlain, flags,
                               s);
  }
  if (!ua && fused_units_supported(dtype, L))
    return launch_int_fused(dtype, 8, false, true, x, units, L, nullptr, nullptr, absmax, minv, maxv,
                            SrCtx{}, kCalPlain, nullptr, nullptr, nullptr, flags, s);
  return launch_unit_generic(dtype, 0, 8, false, x, units, L, absmax, minv, maxv, nullptr, nullptr,
                             nullptr, kCalPlain, flags, s);
}

// The integer and FP8 entry points share one body; sr == nullptr rounds to
// nearest, otherwise stochastically with the call's draws.
static qat_status fake_quant_int_impl(const void* x, qat_dtype dtype, int64_t rows, int64_t cols,
                                      int bits, qat_scheme scheme, qat_granularity g,
                                      int64_t group, int params_given, float* scale, int32_t* zp,
                                      const SrCtx* sr, const CalOpts& co, void* y, void* codes,
                                      uint32_t* mask, int32_t* flags, void* ws, size_t ws_bytes,
                                      qat_stream_t stream) {
  if (!valid_dtype(dtype)) return QAT_ERR_UNSUPPORTED;
  if (bits != 8 && bits != 4) return QAT_ERR_UNSUPPORTED;
  if (scheme != QAT_SYMMETRIC && scheme != QAT_AFFINE) return QAT_ERR_UNSUPPORTED;
  const bool affine = scheme == QAT_AFFINE;
  int64_t n, L, units;
  if (!elems(rows, cols, &n)) return QAT_ERR_INVALID_ARGUMENT;
  if (!unit_shape(rows, cols, g, group, &L, &units)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (g == QAT_PER_COLUMN && cols > kMaxColumns) return QAT_ERR_UNSUPPORTED;
  if (!x || !scale) return QAT_ERR_INVALID_ARGUMENT;
  if (params_given && affine && !zp) return QAT_ERR_INVALID_ARGUMENT;
  if (!elem_aligned(x, dtype) || (y && !elem_aligned(y, dtype)) ||
      (codes && !aligned(codes, kAlignBuf)) || (mask && !aligned(mask, kAlignBuf)) ||
      !aligned(scale, 4) || (zp && !aligned(zp, 4)))
    return QAT_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const SrCtx c = sr ? *sr : SrCtx{};
  if (!aligned(x, kAlignVec) || (y && !aligned(y, kAlignVec))) {
    // element-aligned tensors off the vector grid: per tensor, rows, groups
    if (g == QAT_PER_COLUMN) return QAT_ERR_MISALIGNED;
    if (params_given)
      return launch_ua_int_map(dtype, bits, affine, g == QAT_PER_TENSOR ? 1 : 3, sr != nullptr, x,
                               n, L, nullptr, 0, scale, zp, nullptr, c, co, y, codes, mask, flags,
                               s);
    if (!ws || ws_bytes < ws_bytes_for(rows, cols, g, group)) return QAT_ERR_WORKSPACE;
    if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
    if (g == QAT_PER_TENSOR) {
      const int grid = stats_grid(n);
      qat_status st = launch_ua_stats(dtype, affine ? kMMFloat : kMMNone, x, n, ws, grid, s);
      if (st) return st;
      return launch_ua_int_map(dtype, bits, affine, 0, sr != nullptr, x, n, n, ws, grid, scale,
                               zp, nullptr, c, co, y, codes, mask, flags, s);
    }
    uint8_t* dead = ws_dead(ws, cols, g);
    int32_t* zpu = (affine && !zp) ? ws_zp(ws, cols, g, units) : zp;
    qat_status st = launch_unit_generic(dtype, 1, bits, affine, x, units, L, nullptr, nullptr,
                                        nullptr, scale, zpu, dead, co, flags, s);
    if (st) return st;
    return launch_ua_int_map(dtype, bits, affine, 2, sr != nullptr, x, n, L, nullptr, 0, scale,
                             zpu, dead, c, co, y, codes, mask, flags, s);
  }
  auto map_tensor = sr ? launch_int_tensor_sr : launch_int_tensor;
  auto map_units = sr ? launch_int_units_sr : launch_int_units;
  auto map_fused = sr ? launch_int_fused_sr : launch_int_fused;
  if (g == QAT_PER_TENSOR) {
    if (params_given)
      return map_tensor(dtype, bits, affine, true, x, n, nullptr, 0, scale, zp, c, co, y, codes, mask,
                        flags, s, false);
    if (!ws || ws_bytes < ws_bytes_for(rows, cols, g, group)) return QAT_ERR_WORKSPACE;
    if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
    const bool plain = co.clip == 1.0f && !co.fp16 && !co.clamp;
    if (!sr && plain) {
      // a tensor that fits on chip: statistics and map in one launch
      bool done = false;
      qat_status st = launch_int_tensor_onchip(dtype, bits, affine, x, n, ws, scale, zp, y, codes,
                                               mask, flags, s, &done);
      if (st || done) return st;
    }
    int grid = stats_grid(n);
    qat_status st = launch_stats_tensor(dtype, x, n, affine ? kMMFloat : kMMNone, ws, grid, s);
    if (st) return st;
    return map_tensor(dtype, bits, affine, false, x, n, ws, grid, scale, zp, c, co, y, codes, mask,
                      flags, s, true);
  }
  const bool col = g == QAT_PER_COLUMN;
  const int64_t ucols = col ? cols : 0;
  if (params_given)
    return map_units(dtype, bits, affine, true, x, n, L, ucols, scale, zp, nullptr, c, y, codes,
                     mask, flags, s);
  if (!col && fused_units_supported(dtype, L))
    return map_fused(dtype, bits, affine, false, x, units, L, scale, zp, nullptr, nullptr, nullptr,
                     c, co, y, codes, mask, flags, s);
  if (!ws || ws_bytes < ws_bytes_for(rows, cols, g, group)) return QAT_ERR_WORKSPACE;
  if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
  uint8_t* dead = ws_dead(ws, cols, g);
  int32_t* zpu = (affine && !zp) ? ws_zp(ws, cols, g, units) : zp;
  qat_status st;
  if (col) {
    // column statistics, then the strip map that calibrates its columns
    // (whole mask words per warp row), or the calibration and the unit kernel
    st = launch_col_stats(dtype, affine, x, rows, cols, ws, flags, s);
    if (st) return st;
    if (cols % 32 == 0) {
      auto map_cols = sr ? launch_int_cols_sr : launch_int_cols;
      return map_cols(dtype, bits, affine, x, rows, cols, ws, scale, zp, c, co, y, codes, mask,
                      flags, s);
    }
    st = launch_col_finalize(1, bits, affine, ws, cols, scale, nullptr, nullptr, zpu, co, flags, s);
    if (st) return st;
  } else {
    // fallback: calibrate every unit, then the flat map with per-unit arrays
    st = launch_unit_generic(dtype, 1, bits, affine, x, units, L, nullptr, nullptr, nullptr, scale,
                             zpu, dead, co, flags, s);
    if (st) return st;
  }
  return map_units(dtype, bits, affine, false, x, n, L, ucols, scale, zpu, dead, c, y, codes, mask,
                   flags, s);
}

qat_status qat_fake_quant_int(const void* x, qat_dtype dtype, int64_t rows, int64_t cols, int bits,
                              qat_scheme scheme, qat_granularity g, int64_t group, int params_given,
                              float* scale, int32_t* zp, void* y, void* codes, uint32_t* mask,
                              int32_t* flags, void* ws, size_t ws_bytes, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_fake_quant_int");
  return fake_quant_int_impl(x, dtype, rows, cols, bits, scheme, g, group, params_given, scale, zp,
                             nullptr, kCalPlain, y, codes, mask, flags, ws, ws_bytes, stream);
}

static SrCtx sr_ctx(uint64_t seed, uint64_t offset) {
  SrCtx c;
  c.k0 = (uint32_t)seed;
  c.k1 = (uint32_t)(seed >> 32);
  c.offset = offset;
  sr_set_round_keys(c);
  return c;
}

qat_status qat_fake_quant_int_sr(const void* x, qat_dtype dtype, int64_t rows, int64_t cols,
                                 int bits, qat_scheme scheme, qat_granularity g, int64_t group,
                                 int params_given, float* scale, int32_t* zp, uint64_t seed,
                                 uint64_t offset, void* y, void* codes, uint32_t* mask,
                                 int32_t* flags, void* ws, size_t ws_bytes, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_fake_quant_int_sr");
  const SrCtx c = sr_ctx(seed, offset);
  return fake_quant_int_impl(x, dtype, rows, cols, bits, scheme, g, group, params_given, scale, zp,
                             &c, kCalPlain, y, codes, mask, flags, ws, ws_bytes, stream);
}

qat_status qat_fake_quant_int_opts(const void* x, qat_dtype dtype, int64_t rows, int64_t cols,
                                   int bits, qat_scheme scheme, qat_granularity g, int64_t group,
                                   const qat_calib_options* options, int stochastic, uint64_t seed,
                                   uint64_t offset, float* scale, int32_t* zp, void* y, void* codes,
                                   uint32_t* mask, int32_t* flags, void* ws, size_t ws_bytes,
                                   qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_fake_quant_int_opts");
  CalOpts co = kCalPlain;
  if (options) {
    if (!(options->clip > 0.0f && options->clip <= 1.0f)) return QAT_ERR_INVALID_ARGUMENT;
    co.clip = options->clip;
    co.fp16 = options->scale_fp16 ? 1 : 0;
  }
  const SrCtx c = sr_ctx(seed, offset);
  return fake_quant_int_impl(x, dtype, rows, cols, bits, scheme, g, group, 0, scale, zp,
                             stochastic ? &c : nullptr, co, y, codes, mask, flags, ws, ws_bytes,
                             stream);
}

size_t qat_percentile_workspace_bytes(void) { return pct_ws_bytes(); }

qat_status qat_fake_quant_int_percentile(const void* x, qat_dtype dtype, int64_t n, int bits,
                                         qat_scheme scheme, double clip_fraction, int stochastic,
                                         uint64_t seed, uint64_t offset, float* scale, int32_t* zp,
                                         void* y, void* codes, uint32_t* mask, int32_t* flags,
                                         void* ws, size_t ws_bytes, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_fake_quant_int_percentile");
  if (!valid_dtype(dtype)) return QAT_ERR_UNSUPPORTED;
  if (bits != 8 && bits != 4) return QAT_ERR_UNSUPPORTED;
  if (scheme != QAT_SYMMETRIC && scheme != QAT_AFFINE) return QAT_ERR_UNSUPPORTED;
  if (!(clip_fraction >= 0.0 && clip_fraction < 0.5)) return QAT_ERR_INVALID_ARGUMENT;
  if (n < 0 || n > (INT64_C(1) << 40)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!x || !scale) return QAT_ERR_INVALID_ARGUMENT;
  if (!aligned(x, kAlignVec) || (y && !aligned(y, kAlignVec)) ||
      (codes && !aligned(codes, kAlignBuf)) || (mask && !aligned(mask, kAlignBuf)) ||
      !aligned(scale, 4) || (zp && !aligned(zp, 4)))
    return QAT_ERR_MISALIGNED;
  if (!ws || ws_bytes < pct_ws_bytes()) return QAT_ERR_WORKSPACE;
  if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
  // QuantParams::per_tensor_percentile: the index products in binary64
  const int64_t last = n - 1;
  int64_t lo = (int64_t)floor(clip_fraction * (double)last);
  int64_t hi = (int64_t)ceil((1.0 - clip_fraction) * (double)last);
  if (lo > last) lo = last;
  if (hi > last) hi = last;
  const bool affine = scheme == QAT_AFFINE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  qat_status st = launch_percentile(dtype, x, n, affine, (unsigned long long)lo,
                                    (unsigned long long)hi, ws, s);
  if (st) return st;
  // the per-tensor map from the one partial; values beyond the quantiles
  // clamp to the end codes
  const CalOpts co{1.0f, 0, 1};
  const SrCtx c = sr_ctx(seed, offset);
  auto map = stochastic ? launch_int_tensor_sr : launch_int_tensor;
  return map(dtype, bits, affine, false, x, n, ws, 1, scale, zp, c, co, y, codes, mask, flags, s,
             true);
}

qat_status qat_fake_quant_block(const void* x, qat_dtype dtype, int64_t n, qat_elem_format elem,
                                int64_t block, qat_block_scale kind, float* tensor_scale, void* y,
                                uint8_t* codes, void* bscales, uint32_t* mask, int32_t* flags,
                                void* ws, size_t ws_bytes, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_fake_quant_block");
  if (!valid_dtype(dtype)) return QAT_ERR_UNSUPPORTED;
  if (elem < QAT_ELEM_E4M3 || elem > QAT_ELEM_E2M1) return QAT_ERR_UNSUPPORTED;
  if (kind < QAT_BLOCK_SCALE_E8M0 || kind > QAT_BLOCK_SCALE_FP32) return QAT_ERR_UNSUPPORTED;
  if (block != 16 && block != 32) return QAT_ERR_UNSUPPORTED;
  if (n < 0 || n > (INT64_C(1) << 50) || n % block != 0) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!x) return QAT_ERR_INVALID_ARGUMENT;
  if (!aligned(x, kAlignVec) || (y && !aligned(y, kAlignVec)) ||
      (codes && !aligned(codes, kAlignBuf)) || (mask && !aligned(mask, kAlignBuf)) ||
      (bscales && !aligned(bscales, 4)) || (tensor_scale && !aligned(tensor_scale, 4)))
    return QAT_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int grid = 0;
  if (kind == QAT_BLOCK_SCALE_E4M3) {
    if (!ws || ws_bytes < ws_bytes_for(1, n, QAT_PER_TENSOR, 0)) return QAT_ERR_WORKSPACE;
    if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
    grid = stats_grid(n);
    qat_status st = launch_stats_tensor(dtype, x, n, kMMNone, ws, grid, s);
    if (st) return st;
  }
  return launch_block_fq(dtype, elem, kind, block, x, n, ws, grid, tensor_scale, y, codes,
                         bscales, mask, flags, s);
}

static qat_status fake_quant_fp8_impl(const void* x, qat_dtype dtype, int64_t n,
                                      qat_fp8_format fmt, int scale_given, float* scale,
                                      const SrCtx* sr, void* y, uint8_t* codes, uint32_t* mask,
                                      int32_t* flags, void* ws, size_t ws_bytes,
                                      qat_stream_t stream) {
  if (!valid_dtype(dtype)) return QAT_ERR_UNSUPPORTED;
  if (fmt != QAT_E4M3 && fmt != QAT_E5M2) return QAT_ERR_UNSUPPORTED;
  if (n < 0 || n > (INT64_C(1) << 50)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!x || !y || !scale) return QAT_ERR_INVALID_ARGUMENT;
  if (!elem_aligned(x, dtype) || !elem_aligned(y, dtype) ||
      (codes && !aligned(codes, kAlignBuf)) || (mask && !aligned(mask, kAlignBuf)) ||
      !aligned(scale, 4))
    return QAT_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const SrCtx c = sr ? *sr : SrCtx{};
  if (!aligned(x, kAlignVec) || !aligned(y, kAlignVec)) {
    // element-aligned tensors off the vector grid
    if (scale_given)
      return launch_ua_fp8_map(dtype, fmt, true, sr != nullptr, x, n, nullptr, 0, scale, c, y,
                               codes, mask, flags, s);
    if (!ws || ws_bytes < ws_bytes_for(1, n, QAT_PER_TENSOR, 0)) return QAT_ERR_WORKSPACE;
    if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
    const int grid = stats_grid(n);
    qat_status st = launch_ua_stats(dtype, kMMNone, x, n, ws, grid, s);
    if (st) return st;
    return launch_ua_fp8_map(dtype, fmt, false, sr != nullptr, x, n, ws, grid, scale, c, y, codes,
                             mask, flags, s);
  }
  auto map = sr ? launch_fp8_tensor_sr : launch_fp8_tensor;
  if (scale_given)
    return map(dtype, fmt, true, x, n, nullptr, 0, scale, c, y, codes, mask, flags, s, false);
  if (!ws || ws_bytes < ws_bytes_for(1, n, QAT_PER_TENSOR, 0)) return QAT_ERR_WORKSPACE;
  if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
  int grid = stats_grid(n);
  qat_status st = launch_stats_tensor(dtype, x, n, kMMNone, ws, grid, s);
  if (st) return st;
  return map(dtype, fmt, false, x, n, ws, grid, scale, c, y, codes, mask, flags, s, true);
}

qat_status qat_fake_quant_fp8(const void* x, qat_dtype dtype, int64_t n, qat_fp8_format fmt,
                              int scale_given, float* scale, void* y, uint8_t* codes,
                              uint32_t* mask, int32_t* flags, void* ws, size_t ws_bytes,
                              qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_fake_quant_fp8");
  return fake_quant_fp8_impl(x, dtype, n, fmt, scale_given, scale, nullptr, y, codes, mask, flags,
                             ws, ws_bytes, stream);
}

qat_status qat_fake_quant_fp8_sr(const void* x, qat_dtype dtype, int64_t n, qat_fp8_format fmt,
                                 int scale_given, float* scale, uint64_t seed, uint64_t offset,
                                 void* y, uint8_t* codes, uint32_t* mask, int32_t* flags,
                                 void* ws, size_t ws_bytes, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_fake_quant_fp8_sr");
  const SrCtx c = sr_ctx(seed, offset);
  return fake_quant_fp8_impl(x, dtype, n, fmt, scale_given, scale, &c, y, codes, mask, flags, ws,
                             ws_bytes, stream);
}

qat_status qat_optimizer_step(float* master, const float* grad, float* exp_avg, float* exp_avg_sq,
                              int64_t n, const qat_adam_hparams* hp, int bits, qat_scheme scheme,
                              qat_fp8_format format, int stochastic, uint64_t seed,
                              uint64_t offset, float* view, void* codes, uint32_t* mask,
                              float* scale, int32_t* zp, int32_t* flags, void* ws,
                              size_t ws_bytes, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_optimizer_step");
  if (!hp) return QAT_ERR_INVALID_ARGUMENT;
  if (bits != 0 && bits != 4 && bits != 8) return QAT_ERR_UNSUPPORTED;
  if (bits == 0 && format != QAT_E4M3 && format != QAT_E5M2) return QAT_ERR_UNSUPPORTED;
  if (bits != 0 && scheme != QAT_SYMMETRIC && scheme != QAT_AFFINE) return QAT_ERR_UNSUPPORTED;
  if (n < 0 || n > (INT64_C(1) << 50)) return QAT_ERR_INVALID_ARGUMENT;
  const float bc1 = hp->bias_correction1, bc2 = hp->bias_correction2;
  if (!(bc1 > 0.0f) || !(bc2 > 0.0f) || isinf(bc1) || isinf(bc2)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!master || !grad || !exp_avg || !exp_avg_sq || !view || !scale)
    return QAT_ERR_INVALID_ARGUMENT;
  if (!aligned(master, kAlignVec) || !aligned(grad, kAlignVec) || !aligned(exp_avg, kAlignVec) ||
      !aligned(exp_avg_sq, kAlignVec) || !aligned(view, kAlignVec) ||
      (codes && !aligned(codes, kAlignBuf)) || (mask && !aligned(mask, kAlignBuf)) ||
      !aligned(scale, 4) || (zp && !aligned(zp, 4)))
    return QAT_ERR_MISALIGNED;
  const bool int_view = bits != 0;
  if (int_view) {
    if (!ws || ws_bytes < ws_bytes_for(1, n, QAT_PER_TENSOR, 0)) return QAT_ERR_WORKSPACE;
    if (!aligned(ws, kAlignBuf)) return QAT_ERR_MISALIGNED;
  }
  AdamHp a;
  a.lr = hp->lr;
  a.beta1 = hp->beta1;
  a.beta2 = hp->beta2;
  a.eps = hp->eps;
  a.omb1 = 1.0f - hp->beta1;
  a.omb2 = 1.0f - hp->beta2;
  a.lrwd = hp->lr * hp->weight_decay;
  a.bc1 = bc1;
  a.bc2 = bc2;
  a.decay = hp->weight_decay != 0.0f;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool affine = int_view && scheme == QAT_AFFINE;
  const int grid = stats_grid(n);
  qat_status st = launch_adam(master, grad, exp_avg, exp_avg_sq, n, a,
                              affine ? kMMFloat : kMMNone, int_view, ws, grid,
                              int_view ? nullptr : scale, s);
  if (st) return st;
  const SrCtx c = sr_ctx(seed, offset);
  if (int_view) {
    auto map = stochastic ? launch_int_tensor_sr : launch_int_tensor;
    return map(QAT_F32, bits, affine, false, master, n, ws, grid, scale, zp, c, kCalPlain, view,
               codes, mask, flags, s, true);
  }
  auto map = stochastic ? launch_fp8_tensor_sr : launch_fp8_tensor;
  return map(QAT_F32, format, true, master, n, nullptr, 0, scale, c, view,
             static_cast<uint8_t*>(codes), mask, flags, s, true);
}

qat_status qat_ste_backward(const void* grad, qat_dtype dtype, int64_t n, const uint32_t* mask,
                            void* grad_in, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_ste_backward");
  if (!valid_dtype(dtype)) return QAT_ERR_UNSUPPORTED;
  if (n < 0 || n > (INT64_C(1) << 50)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!grad || !mask || !grad_in) return QAT_ERR_INVALID_ARGUMENT;
  if (!elem_aligned(grad, dtype) || !elem_aligned(grad_in, dtype) || !aligned(mask, kAlignBuf))
    return QAT_ERR_MISALIGNED;
  if (!aligned(grad, kAlignVec) || !aligned(grad_in, kAlignVec))
    return launch_ua_ste(dtype, grad, n, mask, grad_in, reinterpret_cast<cudaStream_t>(stream));
  return launch_ste(dtype, grad, n, mask, grad_in, reinterpret_cast<cudaStream_t>(stream));
}

qat_status qat_quant4_double(const float* x, int64_t n, uint8_t* data, uint8_t* qscales,
                             float* super_scales, float* y, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_quant4_double");
  if (n < 0 || n > (INT64_C(1) << 50)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!x || !data || !qscales || !super_scales) return QAT_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 4) || !aligned(data, kAlignBuf) || !aligned(qscales, kAlignBuf) ||
      !aligned(super_scales, 4) || (y && !aligned(y, 4)))
    return QAT_ERR_MISALIGNED;
  const bool ua = !aligned(x, kAlignVec) || (y && !aligned(y, kAlignVec));
  return launch_q4_quant(x, n, data, qscales, super_scales, y, ua,
                         reinterpret_cast<cudaStream_t>(stream));
}

qat_status qat_dequant4_double(const uint8_t* data, const uint8_t* qscales, const float* super_scales,
                               int64_t n, float* y, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_dequant4_double");
  if (n < 0 || n > (INT64_C(1) << 50)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!data || !qscales || !super_scales || !y) return QAT_ERR_INVALID_ARGUMENT;
  if (!aligned(data, kAlignBuf) || !aligned(qscales, kAlignBuf) || !aligned(super_scales, 4) ||
      !aligned(y, 4))
    return QAT_ERR_MISALIGNED;
  return launch_q4_dequant(data, qscales, super_scales, n, y, !aligned(y, kAlignVec),
                           reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
