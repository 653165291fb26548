// cb_gemm_noalloc: the projection GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a host application that must not grow
// its device footprint after start-up (a fixed memory budget), code running inside
// another framework that owns every allocation, or a plugin handed raw pointers only.
// For them this entry point needs nothing but the operands: the stream-K scratch of the
// tcgen05 GEMM (its flags and partial tiles) lives in the file-scope array below, which
// every GPU that loads this library holds until the process exits.
//
// This file also holds the status word of the standalone GEMM calls (cb_gemm and
// cb_gemm_noalloc): a stream-K wait that gives up records itself there, and
// cb_gemm_get_status reads and clears it.
#include <chrono>
#include <cstdio>
#include <mutex>
#include <thread>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[CB_GEMM_STATIC_SCRATCH_BYTES];
static __device__ int32_t g_gemm_status;  // zero at load; ST_* bits

constexpr int kMaxDevices = 64;
std::mutex g_symbols_mu;
void* g_scratch_addr[kMaxDevices] = {};
void* g_status_addr[kMaxDevices] = {};

// Device addresses of the file's device arrays on the current device, looked up once per
// device.  In host code an array's name is only a host-side stand-in, so kernels get
// these addresses.
cudaError_t symbol_addresses(void** scratch, void** status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_symbols_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    void* q = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(&q, g_gemm_status);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
    g_status_addr[dev] = q;
  }
  if (scratch) *scratch = g_scratch_addr[dev];
  if (status) *status = g_status_addr[dev];
  return cudaSuccess;
}

thread_local char g_noalloc_msg[256];

cb_status noalloc_fail(cb_status st, const char* msg) {
  snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "cb_gemm_noalloc: %s", msg);
  return st;
}

cb_status noalloc_cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "cb_gemm_noalloc: %s: %s", where, cudaGetErrorString(e));
  return CB_ERR_CUDA;
}

}  // namespace

namespace cb {

cudaError_t standalone_gemm_status(int32_t** out) {
  void* p = nullptr;
  cudaError_t e = symbol_addresses(nullptr, &p);
  *out = static_cast<int32_t*>(p);
  return e;
}

}  // namespace cb

extern "C" cb_status cb_gemm_noalloc(const void* A, const void* B, const void* B2, void* C, int M, int N, int K,
                                     int ldc, int epilogue, cb_dtype dtype, void* stream) {
  if (!A || !B || !C || (epilogue == 2 && !B2)) return noalloc_fail(CB_ERR_INVALID_ARG, "null pointer");
  if (epilogue < 0 || epilogue > 2) return noalloc_fail(CB_ERR_INVALID_ARG, "epilogue must be 0, 1 or 2");
  if (M < 0 || N < 1 || K < 1) return noalloc_fail(CB_ERR_SHAPE, "need M >= 0, N >= 1, K >= 1");
  if (dtype == CB_BF16) {
    if (K % 64 || N % 128 || (reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        (B2 && (reinterpret_cast<uintptr_t>(B2) & 15)))
      return noalloc_fail(CB_ERR_SHAPE, "bf16 needs K % 64 == 0, N % 128 == 0 and 16-byte aligned operands");
    if (ldc % 8 || (reinterpret_cast<uintptr_t>(C) & 15))
      return noalloc_fail(CB_ERR_SHAPE, "bf16 needs ldc % 8 == 0 and a 16-byte aligned C");
  } else if (dtype != CB_F32) {
    return noalloc_fail(CB_ERR_DTYPE, "unknown dtype");
  }
  if (epilogue == 2 ? ldc < N / 2 : ldc < N) return noalloc_fail(CB_ERR_SHAPE, "ldc smaller than the output row");
  // The schedule narrows its stream-K split to the partial slots the built-in array holds,
  // exactly as cb_gemm does with a small caller scratch, so every shape cb_gemm accepts
  // runs here.  A schedule that asked for more than the array would be refused.
  const void* B1 = epilogue == 2 ? B2 : nullptr;
  const size_t need = cb::gemm_scratch_used(A, B, B1, nullptr, N, N, M, N, K, epilogue, dtype, CB_GEMM_STATIC_SCRATCH_BYTES);
  if (need > CB_GEMM_STATIC_SCRATCH_BYTES) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg),
             "cb_gemm_noalloc: the schedule needs %zu bytes of scratch, the built-in array holds %zu", need,
             static_cast<size_t>(CB_GEMM_STATIC_SCRATCH_BYTES));
    return CB_ERR_WORKSPACE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  void* status = nullptr;
  cudaError_t e = symbol_addresses(&scratch, &status);
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "cudaGetSymbolAddress");
  if (need > 0) {
    // the flags must start at zero; a previous call that gave up may have left some set
    e = cudaMemsetAsync(scratch, 0, 1024, s);
    if (e != cudaSuccess) return noalloc_cuda_fail(e, "cudaMemsetAsync");
  }
  e = cb::launch_gemm(A, B, B1, nullptr, N, N, C, M, N, K, ldc, epilogue, dtype, static_cast<int32_t*>(status),
                      need > 0 ? scratch : nullptr, need > 0 ? CB_GEMM_STATIC_SCRATCH_BYTES : 0, s);
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "launch");
  g_noalloc_msg[0] = '\0';
  return CB_OK;
}

extern "C" const char* cb_gemm_noalloc_error(void) { return g_noalloc_msg; }

extern "C" size_t cb_gemm_noalloc_scratch_used(int M, int N, int K, int epilogue, cb_dtype dtype) {
  if (M <= 0 || N < 1 || K < 1 || epilogue < 0 || epilogue > 2) return 0;
  // aligned stand-ins for the operands: the schedule looks only at their alignment
  const void* op = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  return cb::gemm_scratch_used(op, op, epilogue == 2 ? op : nullptr, nullptr, N, N, M, N, K, epilogue, dtype,
                               CB_GEMM_STATIC_SCRATCH_BYTES);
}

extern "C" cb_status cb_gemm_get_status(void* stream, int timeout_ms) {
  void* status = nullptr;
  cudaError_t e = symbol_addresses(nullptr, &status);
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "cudaGetSymbolAddress");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t ev = nullptr;
  e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "cudaEventCreate");
  e = cudaEventRecord(ev, s);
  const auto t0 = std::chrono::steady_clock::now();
  while (e == cudaSuccess) {  // bounded wait for the stream's earlier work
    e = cudaEventQuery(ev);
    if (e != cudaErrorNotReady) break;  // done (cudaSuccess) or a real error
    e = cudaSuccess;
    if (timeout_ms >= 0 &&
        std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms)) {
      cudaEventDestroy(ev);
      snprintf(g_noalloc_msg, sizeof(g_noalloc_msg), "cb_gemm_get_status: stream not done within %d ms", timeout_ms);
      return CB_ERR_TIMEOUT;
    }
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  cudaEventDestroy(ev);
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "cudaEventQuery");
  int32_t v = 0;
  e = cudaMemcpyAsync(&v, status, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "reading the status word");
  if (v) {
    snprintf(g_noalloc_msg, sizeof(g_noalloc_msg),
             "cb_gemm_get_status: device status word %d (%s): outputs of the standalone GEMMs since the last check are "
             "not valid",
             static_cast<int>(v), (v & ST_WAIT_TIMEOUT) ? "a stream-K wait gave up" : "index out of range");
    return CB_ERR_DEVICE;
  }
  g_noalloc_msg[0] = '\0';
  return CB_OK;
}
