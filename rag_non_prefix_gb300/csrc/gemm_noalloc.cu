// cb_gemm_noalloc: the projection GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a host application that must not grow
// its device footprint after start-up (a fixed memory budget), code running inside
// another framework that owns every allocation, or a plugin handed raw pointers only.
// For them this entry point needs nothing but the operands: the stream-K scratch of the
// tcgen05 GEMM (its flags and partial tiles) lives in the file-scope array below, which
// every GPU that loads this library holds until the process exits.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[CB_GEMM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.  In
// host code the array's name is only a host-side stand-in, so kernels get this address.
cudaError_t noalloc_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}

thread_local char g_noalloc_msg[256];

}  // namespace

extern "C" cb_status cb_gemm_noalloc(const void* A, const void* B, const void* B2, void* C, int M, int N, int K,
                                     int ldc, int epilogue, cb_dtype dtype, void* stream) {
  if (!A || !B || !C || (epilogue == 2 && !B2)) return CB_ERR_INVALID_ARG;
  if (epilogue < 0 || epilogue > 2) return CB_ERR_INVALID_ARG;
  if (M < 0 || N < 1 || K < 1) return CB_ERR_SHAPE;
  if (dtype == CB_BF16) {
    if (K % 64 || N % 128 || (reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        (B2 && (reinterpret_cast<uintptr_t>(B2) & 15)) || ldc % 8 || (reinterpret_cast<uintptr_t>(C) & 15))
      return CB_ERR_SHAPE;
  } else if (dtype != CB_F32) {
    return CB_ERR_DTYPE;
  }
  if (epilogue == 2 ? ldc < N / 2 : ldc < N) return CB_ERR_SHAPE;
  // The schedule cb_gemm would pick with unlimited scratch; refuse what does not fit.
  const size_t need = cb::gemm_scratch_needed(N, M, K, dtype);
  if (need > CB_GEMM_STATIC_SCRATCH_BYTES) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg),
             "cb_gemm_noalloc: this shape's stream-K split needs %zu bytes of scratch, the built-in array holds %zu; "
             "use cb_gemm with caller scratch",
             need, static_cast<size_t>(CB_GEMM_STATIC_SCRATCH_BYTES));
    return CB_ERR_WORKSPACE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if (need > 0) {
    if (noalloc_scratch_address(&scratch) != cudaSuccess) return CB_ERR_CUDA;
    // the flags must start at zero; a previous call that gave up may have left some set
    if (cudaMemsetAsync(scratch, 0, 1024, s) != cudaSuccess) return CB_ERR_CUDA;
  }
  cudaError_t e = cb::launch_gemm(A, B, epilogue == 2 ? B2 : nullptr, nullptr, N, N, C, M, N, K, ldc, epilogue, dtype,
                                  nullptr, scratch, need > 0 ? CB_GEMM_STATIC_SCRATCH_BYTES : 0, s);
  return e == cudaSuccess ? CB_OK : CB_ERR_CUDA;
}

extern "C" const char* cb_gemm_noalloc_error(void) { return g_noalloc_msg; }
