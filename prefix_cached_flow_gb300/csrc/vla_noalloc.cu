// Allocation-free variant of the W2A8 scaled ternary product entry point.
//
// vla_w2a8_ternary_gemm takes its fp32 partial-sum scratch from the stream's
// memory pool on every call.  Some callers cannot allocate device memory
// while they run: a robot control loop with a hard period, where a device
// allocation may synchronise the device or take an unbounded time, or a
// host program whose device memory is reserved up front by another runtime's
// pool and must not grow.  vla_w2a8_ternary_gemm_noalloc runs the same two
// kernels with the scratch in a fixed array that is part of the loaded
// library, so a call allocates nothing.
//
// The array is VLA_NOALLOC_MAX_ELEMS fp32 values (4 MiB).  Every GPU that
// loads the library holds its own copy until the process exits.  All calls
// share it: calls that overlap on the GPU (different streams, or different
// host threads, without ordering between them) race on it and must not be
// issued.  Nothing in it has to start at zero: the product kernel writes every
// one of the M x N slots that the scaling kernel then reads, on one stream.
#include <mutex>

#include "vla_common.cuh"

namespace {

static __device__ __align__(256) float g_noalloc_scratch[VLA_NOALLOC_MAX_ELEMS];

// Device address of g_noalloc_scratch per device ordinal.  In host code the
// array's name is only a host-side stand-in, never a device address, so the
// address is looked up once per device with that device current.  The cached
// address belongs to the device context that was current at the lookup: a
// caller that resets the device (cudaDeviceReset) must not call this entry
// point on that device again in the same process.
constexpr int kMaxDevices = 64;
float* g_scratch_dev[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = (float*)p;
  }
  *out = g_scratch_dev[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" vla_status vla_w2a8_ternary_gemm_noalloc(const int8_t* a, const float* alpha, const uint8_t* q,
                                                    float beta, int M, int N, int K, uint16_t* y, int32_t* acc,
                                                    void* stream) {
  // Same contract as vla_w2a8_ternary_gemm, plus: the product kernel reads the
  // codes as 32-bit words, so `a` must be 4-byte aligned.
  if (!a || !alpha || !q || !y || M < 1 || N < 1 || K < 64 || K % 64 || K > 65536 || N % 4 ||
      ((uintptr_t)a & 3u))
    return VLA_ERR_INVALID_ARG;
  if ((size_t)M * (size_t)N > (size_t)VLA_NOALLOC_MAX_ELEMS) return VLA_ERR_UNSUPPORTED;
  float* part = nullptr;
  cudaError_t e = noalloc_scratch(&part);
  if (e != cudaSuccess) {
    vla_set_last_error("cudaGetSymbolAddress(g_noalloc_scratch)", e);
    return VLA_ERR_CUDA;
  }
  cudaStream_t st = (cudaStream_t)stream;
  e = launch_ternary_simt(a, K, q, M, N, K, 1, part, 0, N, st);
  if (e == cudaSuccess) e = launch_ternary_finish(part, M, N, alpha, beta, y, acc, st);
  if (e != cudaSuccess) {
    vla_set_last_error("vla_w2a8_ternary_gemm_noalloc", e);
    return VLA_ERR_CUDA;
  }
  return VLA_OK;
}
