// qat_noalloc.cu -- per-tensor FP8 fake quant for callers that cannot
// allocate device memory.
//
// The regular qat_fake_quant_fp8 takes a caller-supplied workspace for the
// cross-block partial statistics of its amax pass.  Some callers have no way
// to provide one: code embedded in a host framework that owns every device
// allocation and hands the library only the tensors it works on, or a
// latency-critical loop that must not call cudaMalloc (which can synchronise
// the device).  qat_fake_quant_fp8_noalloc keeps that scratch in a fixed
// file-scope device array instead, so the caller passes only inputs and
// outputs and nothing is allocated.
//
// The array holds kNoAllocSlots partials of 16 bytes (16 KiB), as many as the
// statistics pass can ever use (its grid is capped at kMaxPartials blocks).
// Every GPU that loads the library reserves it until the process exits.  All
// calls share it: two calls whose kernels overlap on the GPU (different
// streams, or different host threads on the same device) race on it and must
// be ordered by the caller.  Every slot a call reads is first written by the
// same call, so the contents left by the previous call never matter and
// nothing is cleared.
//
// In host code the array's name is only a host-side stand-in.  Each call looks
// up the array's device address with cudaGetSymbolAddress in the context that
// is current at the call (the address belongs to a context: another context
// on the same device, or the primary context created again after
// cudaDeviceReset, holds its own copy), checks the result and passes it to
// the kernels.  After the first call in a context the lookup is a host-side
// table search; the first call may also load the library's device code into
// the context, so it should be made before any stream capture begins.
#include "qat_device.cuh"
#include "qat_launch.h"

namespace {

constexpr int kNoAllocSlots = qat::kMaxPartials;  // 1024 x 16 B = 16 KiB
static_assert(kNoAllocSlots >= qat::kMaxPartials,
              "the scratch must hold every partial the statistics pass can write");

static __device__ __align__(256) uint4 g_noalloc_partials[kNoAllocSlots];

// Device address of the scratch array in the current context.
qat_status scratch_of_current_context(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr) {
    cudaGetLastError();  // clear it, so a later launch check does not report it again
    return QAT_ERR_CUDA;
  }
  *out = p;
  return QAT_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" qat_status qat_fake_quant_fp8_noalloc(const void* x, qat_dtype dtype, int64_t n,
                                                 qat_fp8_format fmt, int scale_given, float* scale,
                                                 void* y, uint8_t* codes, uint32_t* mask,
                                                 int32_t* flags, qat_stream_t stream) {
  qat::NvtxScope nvtx("qat_fake_quant_fp8_noalloc");
  if (dtype != QAT_F32 && dtype != QAT_BF16) return QAT_ERR_UNSUPPORTED;
  if (fmt != QAT_E4M3 && fmt != QAT_E5M2) return QAT_ERR_UNSUPPORTED;
  if (n < 0 || n > (INT64_C(1) << 50)) return QAT_ERR_INVALID_ARGUMENT;
  if (n == 0) return QAT_OK;
  if (!x || !y || !scale) return QAT_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 32) || !aligned(y, 32) || (codes && !aligned(codes, 16)) ||
      (mask && !aligned(mask, 16)) || !aligned(scale, 4))
    return QAT_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (scale_given)
    return qat::launch_fp8_tensor(dtype, fmt, true, x, n, nullptr, 0, scale, qat::SrCtx{}, y, codes,
                                  mask, flags, s, false);
  const int grid = qat::stats_grid(n);  // at most kMaxPartials = kNoAllocSlots
  void* ws = nullptr;
  qat_status st = scratch_of_current_context(&ws);
  if (st) return st;
  st = qat::launch_stats_tensor(dtype, x, n, qat::kMMNone, ws, grid, s);
  if (st) return st;
  return qat::launch_fp8_tensor(dtype, fmt, false, x, n, ws, grid, scale, qat::SrCtx{}, y, codes,
                                mask, flags, s, false);
}
