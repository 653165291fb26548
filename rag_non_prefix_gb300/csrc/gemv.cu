// Projections of a few token rows (M <= GEMV_MAX_ROWS: decoding): C = A . B^T streamed straight
// from the weights.  With so few rows every weight is used M times only, so the product is
// bound by reading the weights once from HBM; a tensor-core tile would be 1/16 to 1/128 full,
// and measured on GB300 the tiles stream the weights slower than this kernel for one or two
// rows (faster from three or four on, where the GEMM takes over).  A CTA owns four
// weight rows (SwiGLU: the gate and up rows of two features) and its 256 threads split the
// k range in 16-byte pieces (two pieces of each row in flight per thread), so that even
// 4096 output features give a thousand CTAs and every SM keeps enough loads in flight to
// cover DRAM latency.  The M activation rows are read from L1/L2; partial sums are reduced
// across the warps in shared memory and the epilogue (store, residual add, SiLU(gate) * up)
// writes each output once.
#include "common.cuh"
#include "internal.h"

namespace cb {

namespace {

constexpr int GV_THREADS = 256;
constexpr int GV_RC = 4;      // weight rows per CTA
constexpr int GV_UNROLL = 2;  // pieces per row in flight per thread

__device__ __forceinline__ void unpack16(const uint4& u, float* f, bf16*) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void unpack16(const uint4& u, float* f, float*) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

__device__ __forceinline__ float gv_silu(float x) { return x / (1.0f + __expf(-x)); }

// mode 0: C fp32 [m][ldc] = acc;  1: C fp32 += acc;  2: C (T) [m][ldc] = SiLU(acc_gate) * acc_up.
// n_out: output features (N, or the SwiGLU feature count).  B rows of [0, split0) come from B0,
// [split0, split1) from B1, the rest from B2 (SwiGLU: B0 gate, B1 up).
template <typename T, typename TA, int MM>
__global__ void __launch_bounds__(GV_THREADS) gemv_kernel(const TA* __restrict__ A, int M, int K,
                                                          const T* __restrict__ B0, const T* __restrict__ B1,
                                                          const T* __restrict__ B2, int split0, int split1, int n_out,
                                                          void* __restrict__ C, int ldc, int mode) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte piece
  __shared__ float red[GV_THREADS / 32][GV_RC * MM];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const T* wr[GV_RC];
  int n0;
  if (mode == 2) {  // rows: gate f, up f, gate f + 1, up f + 1
    n0 = blockIdx.x * (GV_RC / 2);
#pragma unroll
    for (int r = 0; r < GV_RC; ++r) {
      const int f = min(n0 + r / 2, n_out - 1);
      wr[r] = ((r & 1) ? B1 : B0) + static_cast<size_t>(f) * K;
    }
  } else {
    n0 = blockIdx.x * GV_RC;
#pragma unroll
    for (int r = 0; r < GV_RC; ++r) {
      const int n = min(n0 + r, n_out - 1);
      wr[r] = n < split0 ? B0 + static_cast<size_t>(n) * K
                         : (n < split1 ? B1 + static_cast<size_t>(n - split0) * K
                                       : B2 + static_cast<size_t>(n - split1) * K);
    }
  }
  float acc[GV_RC][MM];
#pragma unroll
  for (int r = 0; r < GV_RC; ++r)
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[r][m] = 0.f;
  const int pieces = K / V;
  for (int p0 = tid; p0 < pieces; p0 += GV_THREADS * GV_UNROLL) {
    uint4 wv[GV_UNROLL][GV_RC];
#pragma unroll
    for (int u = 0; u < GV_UNROLL; ++u) {
      const int pc = p0 + u * GV_THREADS;
#pragma unroll
      for (int r = 0; r < GV_RC; ++r)
        wv[u][r] = pc < pieces ? __ldg(reinterpret_cast<const uint4*>(wr[r]) + pc) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < GV_UNROLL; ++u) {
      const int pc = p0 + u * GV_THREADS;
      if (pc >= pieces) break;
      float wf[GV_RC][V];
#pragma unroll
      for (int r = 0; r < GV_RC; ++r) unpack16(wv[u][r], wf[r], static_cast<T*>(nullptr));
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        if (m < M) {
          float af[V];
          const TA* ar = A + static_cast<size_t>(m) * K + static_cast<size_t>(pc) * V;
          if (sizeof(TA) == sizeof(T)) {
            unpack16(__ldg(reinterpret_cast<const uint4*>(ar)), af, static_cast<TA*>(nullptr));
          } else {  // fp32 activations against bf16 weights: two 16-byte pieces per weight piece
            unpack16(__ldg(reinterpret_cast<const uint4*>(ar)), af, static_cast<float*>(nullptr));
            unpack16(__ldg(reinterpret_cast<const uint4*>(ar) + 1), af + 4, static_cast<float*>(nullptr));
          }
#pragma unroll
          for (int r = 0; r < GV_RC; ++r)
#pragma unroll
            for (int e = 0; e < V; ++e) acc[r][m] = fmaf(af[e], wf[r][e], acc[r][m]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < GV_RC; ++r)
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      const float v = warp_sum(acc[r][m]);
      if (lane == 0) red[w][r * MM + m] = v;
    }
  __syncthreads();
  if (mode == 2) {
    if (tid < (GV_RC / 2) * MM) {
      const int fi = tid / MM, m = tid - fi * MM;
      if (m < M && n0 + fi < n_out) {
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int ww = 0; ww < GV_THREADS / 32; ++ww) {
          g += red[ww][(2 * fi) * MM + m];
          u += red[ww][(2 * fi + 1) * MM + m];
        }
        static_cast<T*>(C)[static_cast<size_t>(m) * ldc + n0 + fi] = from_f<T>(gv_silu(g) * u);
      }
    }
  } else if (tid < GV_RC * MM) {
    const int r = tid / MM, m = tid - r * MM;
    if (m < M && n0 + r < n_out) {
      float v = 0.f;
#pragma unroll
      for (int ww = 0; ww < GV_THREADS / 32; ++ww) v += red[ww][r * MM + m];
      float* out = static_cast<float*>(C) + static_cast<size_t>(m) * ldc + n0 + r;
      *out = mode == 1 ? *out + v : v;
    }
  }
}

template <typename T, int MM, typename TA = T>
cudaError_t launch_gv(const void* A, int M, int K, const void* B0, const void* B1, const void* B2, int split0,
                      int split1, int n_out, void* C, int ldc, int mode, cudaStream_t s) {
  const int per = mode == 2 ? GV_RC / 2 : GV_RC;
  const int blocks = (n_out + per - 1) / per;
  launch_chain(gemv_kernel<T, TA, MM>, dim3(blocks), dim3(GV_THREADS), 0, s, static_cast<const TA*>(A), M, K,
               static_cast<const T*>(B0), static_cast<const T*>(B1), static_cast<const T*>(B2), split0, split1, n_out,
               C, ldc, mode);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_gv_t(const void* A, int M, int K, const void* B0, const void* B1, const void* B2, int split0,
                        int split1, int n_out, void* C, int ldc, int mode, cudaStream_t s) {
  if (M == 1) return launch_gv<T, 1>(A, M, K, B0, B1, B2, split0, split1, n_out, C, ldc, mode, s);
  return launch_gv<T, GEMV_MAX_ROWS>(A, M, K, B0, B1, B2, split0, split1, n_out, C, ldc, mode, s);
}

}  // namespace

bool gemv_applies(int M, int K, cb_dtype dt, const void* A, const void* B0, const void* B1, const void* B2) {
  const int v = dt == CB_BF16 ? 8 : 4;
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return M >= 1 && M <= GEMV_MAX_ROWS && K % v == 0 && al(A) && al(B0) && al(B1) && al(B2);
}

cudaError_t launch_gemv(const void* A, const void* B0, const void* B1, const void* B2, int split0, int split1, void* C,
                        int M, int N, int K, int ldc, int mode, cb_dtype dt, cudaStream_t s) {
  const int n_out = mode == 2 ? N / 2 : N;
  if (mode == 2) {
    split0 = split1 = n_out;
  }
  if (dt == CB_BF16) return launch_gv_t<bf16>(A, M, K, B0, B1, B2, split0, split1, n_out, C, ldc, mode, s);
  return launch_gv_t<float>(A, M, K, B0, B1, B2, split0, split1, n_out, C, ldc, mode, s);
}

// LM head of a few rows: logits fp32 [M][vocab] = x (fp32 [M][d]) . W^T, W [vocab][d] of dt.
cudaError_t launch_gemv_f32a(const float* x, const void* W, int M, int vocab, int d, float* logits, cb_dtype dt,
                             cudaStream_t s) {
  if (dt == CB_BF16) {
    if (M == 1) return launch_gv<bf16, 1, float>(x, M, d, W, W, W, vocab, vocab, vocab, logits, vocab, 0, s);
    return launch_gv<bf16, GEMV_MAX_ROWS, float>(x, M, d, W, W, W, vocab, vocab, vocab, logits, vocab, 0, s);
  }
  if (M == 1) return launch_gv<float, 1>(x, M, d, W, W, W, vocab, vocab, vocab, logits, vocab, 0, s);
  return launch_gv<float, GEMV_MAX_ROWS>(x, M, d, W, W, W, vocab, vocab, vocab, logits, vocab, 0, s);
}

}  // namespace cb
