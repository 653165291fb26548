// Decode attention: one new query token per sequence over its fused cache rows 0..p (p = the
// token's position, whose K/V row was just written), split along the keys so that a handful
// of sequences still fill the GPU ("split-KV"): each CTA owns one (sequence, KV head, range of
// at most 128 keys) and all G = H / Hkv query heads of that KV head, so every K/V row is read
// once.  A CTA of head_dim threads:
//   1. copies its K and V rows into shared memory with asynchronous 16-byte copies (every
//      copy of the range in flight at once; rows padded by 16 bytes so that the score pass
//      reads shared memory without bank conflicts);
//   2. scores: thread t takes keys t, t + head_dim, ... against every head (q pre-scaled by
//      log2(e) / sqrt(head_dim): base-2 logits);
//   3. softmax of the range per head (warp w takes heads w, w + nwarps, ...);
//   4. values: thread t owns output channel t of every head.
// With one range the CTA normalises and writes the output; otherwise it writes (o, max, sum)
// of its range to the partial buffers and a second kernel merges the ranges.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace cb {

namespace {


template <int DH>
constexpr int dec_row_bytes() { return DH * 2 + 16; }  // one padded bf16 row (fp32 rows: 4 DH + 16)

// G: query heads per KV head, a compile-time constant so that the per-head loops unroll to
// exactly G (a runtime bound left 16 predicated copies of every head loop).
template <typename T, int DH, int G>
__global__ void __launch_bounds__(DH) decode_attn_kernel(const T* __restrict__ q, const int32_t* __restrict__ pos,
                                                         const ReqDev* __restrict__ reqs, int layer, int H, int Hkv,
                                                         int n_splits, float scale_log2, float* __restrict__ part_o,
                                                         float2* __restrict__ part_ml, T* __restrict__ out,
                                                         int32_t* status) {
  pdl_trigger();
  pdl_wait();
  constexpr int NW = DH / 32;
  constexpr int VEC = 16 / static_cast<int>(sizeof(T));            // elements per 16-byte piece
  constexpr int ROW = (DH * static_cast<int>(sizeof(T)) + 16) / 16;  // padded row in 16-byte pieces
  extern __shared__ uint4 dsm[];
  uint4* ks = dsm;                              // [DECODE_KEYS][ROW]
  uint4* vs = dsm + DECODE_KEYS * ROW;          // [DECODE_KEYS][ROW]
  __shared__ __align__(16) float qs[G][DH];
  __shared__ float sc[G][DECODE_KEYS];
  __shared__ float ml[G][2];
  const int seq = blockIdx.x / Hkv, kvh = blockIdx.x - seq * Hkv;
  const int split = blockIdx.y;
  const int t = threadIdx.x, w = t >> 5, lane = t & 31;
  const int p = pos[seq];
  const ReqDev rq = reqs[seq];
  if (p < 0 || p >= rq.n_tokens || G * Hkv != H) {
    if (t == 0 && split == 0) set_status(status, ST_RANGE);
    return;
  }
  const int k0 = split * DECODE_KEYS, nk = max(0, min(p + 1, k0 + DECODE_KEYS) - k0);
  const size_t kvw = static_cast<size_t>(Hkv) * DH;
  const T* kbase = static_cast<const T*>(rq.k) + static_cast<size_t>(layer) * rq.layer_stride + kvh * DH;
  const T* vbase = static_cast<const T*>(rq.v) + static_cast<size_t>(layer) * rq.layer_stride + kvh * DH;
  // 1. the range's K and V rows -> shared memory: asynchronous 16-byte copies, all issued
  //    before the first wait
  constexpr int PIECES = DH / VEC;  // 16-byte pieces per row
  const uint32_t ks_u = smem_u32(ks), vs_u = smem_u32(vs);
  for (int i = t; i < nk * PIECES; i += DH) {
    const int j = i / PIECES, c = i - j * PIECES;
    const size_t g = static_cast<size_t>(k0 + j) * kvw + c * VEC;
    const uint32_t o = static_cast<uint32_t>((j * ROW + c) * 16);
    cp_async16(ks_u + o, kbase + g, 16);
    cp_async16(vs_u + o, vbase + g, 16);
  }
  cp_async_commit();
  for (int g = 0; g < G; ++g) qs[g][t] = to_f(q[(static_cast<size_t>(seq) * H + kvh * G + g) * DH + t]) * scale_log2;
  cp_async_wait<0>();
  __syncthreads();
  // 2. scores: thread t takes keys t, t + head_dim, ...
  for (int j = t; j < nk; j += DH) {
    const uint4* kr = ks + j * ROW;
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll 4
    for (int c = 0; c < PIECES; ++c) {
      const uint4 u = kr[c];
      float f[8];
      if (sizeof(T) == 2) {
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(h2[e]);
          f[2 * e] = x.x;
          f[2 * e + 1] = x.y;
        }
      } else {
        const float* x = reinterpret_cast<const float*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) f[e] = x[e];
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int e4 = 0; e4 < VEC; e4 += 4) {
          const float4 qv = *reinterpret_cast<const float4*>(&qs[g][c * VEC + e4]);
          acc[g] = fmaf(qv.x, f[e4], acc[g]);
          acc[g] = fmaf(qv.y, f[e4 + 1], acc[g]);
          acc[g] = fmaf(qv.z, f[e4 + 2], acc[g]);
          acc[g] = fmaf(qv.w, f[e4 + 3], acc[g]);
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) sc[g][j] = acc[g];
  }
  __syncthreads();
  // 3. softmax of the range, one warp per head
  for (int g = w; g < G; g += NW) {
    float mx = -INFINITY;
    for (int j = lane; j < nk; j += 32) mx = fmaxf(mx, sc[g][j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float sum = 0.f;
    for (int j = lane; j < nk; j += 32) {
      const float e = exp2f(sc[g][j] - mx);
      sc[g][j] = e;
      sum += e;
    }
    sum = warp_sum(sum);
    if (lane == 0) {
      ml[g][0] = mx;
      ml[g][1] = sum;
    }
  }
  __syncthreads();
  // 4. values: thread t owns channel t
  float o[G];
#pragma unroll
  for (int g = 0; g < G; ++g) o[g] = 0.f;
  const T* vsm = reinterpret_cast<const T*>(vs);
  constexpr int ROW_T = ROW * VEC;  // padded row in elements
#pragma unroll 4
  for (int j = 0; j < nk; ++j) {
    const float v = to_f(vsm[j * ROW_T + t]);
#pragma unroll
    for (int g = 0; g < G; ++g) o[g] = fmaf(sc[g][j], v, o[g]);
  }
  if (n_splits == 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) out[(static_cast<size_t>(seq) * H + kvh * G + g) * DH + t] = from_f<T>(o[g] / ml[g][1]);
    return;
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const size_t slot = (static_cast<size_t>(seq) * H + kvh * G + g) * n_splits + split;
    part_o[slot * DH + t] = o[g];
    if (t == 0) part_ml[slot] = nk > 0 ? make_float2(ml[g][0], ml[g][1]) : make_float2(-INFINITY, 0.f);
  }
}

// Merges the key ranges of one (sequence, head): weights 2^(m_s - M) on each range's sums.
// The (max, sum) pairs are read into shared memory by all threads at once (one load each),
// so the loops below run on shared memory instead of chaining global-load latencies.
template <typename T, int DH>
__global__ void __launch_bounds__(DH) decode_merge_kernel(const float* __restrict__ part_o,
                                                          const float2* __restrict__ part_ml, int n_splits,
                                                          T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float2 mls[];  // [n_splits] (max, sum), then [n_splits] weights
  float* wts = reinterpret_cast<float*>(mls + n_splits);
  __shared__ float inv_l;
  const size_t row = blockIdx.x;   // seq * H + head
  for (int s = threadIdx.x; s < n_splits; s += DH) mls[s] = part_ml[row * n_splits + s];
  __syncthreads();
  // one warp: the largest max, each range's weight 2^(m_s - M) and the total sum, once per row
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int s = threadIdx.x; s < n_splits; s += 32) M = fmaxf(M, mls[s].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int s = threadIdx.x; s < n_splits; s += 32) {
      const float2 ml = mls[s];
      const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
      wts[s] = w;
      L = fmaf(ml.y, w, L);
    }
    L = warp_sum(L);
    if (threadIdx.x == 0) inv_l = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  // each thread: one output element, the ranges' partial values loaded eight at a time
  const float* po = part_o + row * n_splits * DH + threadIdx.x;
  float acc = 0.f;
  int s = 0;
  for (; s + 8 <= n_splits; s += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = po[static_cast<size_t>(s + u) * DH];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc = fmaf(v[u], wts[s + u], acc);
  }
  for (; s < n_splits; ++s) acc = fmaf(po[static_cast<size_t>(s) * DH], wts[s], acc);
  out[row * DH + threadIdx.x] = from_f<T>(acc * inv_l);
}

template <typename T, int DH, int G>
cudaError_t launch_dec(const void* q, const int32_t* pos, const ReqDev* reqs, int n_seq, int layer, int H, int Hkv,
                       int n_splits, float* part_o, float2* part_ml, void* out, int32_t* status, cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(DH));
  const int smem = 2 * DECODE_KEYS * (DH * static_cast<int>(sizeof(T)) + 16);
  static DeviceOnce configured;
  cudaError_t e = max_dynamic_smem_once(reinterpret_cast<const void*>(decode_attn_kernel<T, DH, G>), smem, configured);
  if (e != cudaSuccess) return e;
  launch_chain(decode_attn_kernel<T, DH, G>, dim3(n_seq * Hkv, n_splits), dim3(DH), smem, s, static_cast<const T*>(q),
               pos, reqs, layer, H, Hkv, n_splits, scale_log2, part_o, part_ml, static_cast<T*>(out), status);
  if (n_splits > 1)
    launch_chain(decode_merge_kernel<T, DH>, dim3(n_seq * H), dim3(DH), n_splits * (sizeof(float2) + sizeof(float)), s,
                 static_cast<const float*>(part_o), static_cast<const float2*>(part_ml), n_splits, static_cast<T*>(out));
  return cudaGetLastError();
}

// Query heads per KV head that have a kernel: the grouped-query shapes of the workloads.
template <typename T, int DH>
cudaError_t launch_dec_g(const void* q, const int32_t* pos, const ReqDev* reqs, int n_seq, int layer, int H, int Hkv,
                         int n_splits, float* part_o, float2* part_ml, void* out, int32_t* status, cudaStream_t s) {
  switch (H / Hkv) {
    case 1: return launch_dec<T, DH, 1>(q, pos, reqs, n_seq, layer, H, Hkv, n_splits, part_o, part_ml, out, status, s);
    case 2: return launch_dec<T, DH, 2>(q, pos, reqs, n_seq, layer, H, Hkv, n_splits, part_o, part_ml, out, status, s);
    case 4: return launch_dec<T, DH, 4>(q, pos, reqs, n_seq, layer, H, Hkv, n_splits, part_o, part_ml, out, status, s);
    case 7: return launch_dec<T, DH, 7>(q, pos, reqs, n_seq, layer, H, Hkv, n_splits, part_o, part_ml, out, status, s);
    case 8: return launch_dec<T, DH, 8>(q, pos, reqs, n_seq, layer, H, Hkv, n_splits, part_o, part_ml, out, status, s);
    case 16: return launch_dec<T, DH, 16>(q, pos, reqs, n_seq, layer, H, Hkv, n_splits, part_o, part_ml, out, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_splits(int max_keys) { return std::max(1, (max_keys + DECODE_KEYS - 1) / DECODE_KEYS); }

cudaError_t launch_decode_attention(const void* q, const int32_t* pos, const ReqDev* reqs, int n_seq, int layer,
                                    int n_heads, int n_kv_heads, int head_dim, int n_splits, float* part_o,
                                    float2* part_ml, void* out, cb_dtype dt, int32_t* status, cudaStream_t s) {
  if (n_seq <= 0) return cudaSuccess;
  if (dt == CB_BF16) {
    if (head_dim == 128)
      return launch_dec_g<bf16, 128>(q, pos, reqs, n_seq, layer, n_heads, n_kv_heads, n_splits, part_o,
                                   part_ml, out, status, s);
    if (head_dim == 64)
      return launch_dec_g<bf16, 64>(q, pos, reqs, n_seq, layer, n_heads, n_kv_heads, n_splits, part_o,
                                  part_ml, out, status, s);
  } else {
    if (head_dim == 128)
      return launch_dec_g<float, 128>(q, pos, reqs, n_seq, layer, n_heads, n_kv_heads, n_splits, part_o,
                                    part_ml, out, status, s);
    if (head_dim == 64)
      return launch_dec_g<float, 64>(q, pos, reqs, n_seq, layer, n_heads, n_kv_heads, n_splits, part_o,
                                   part_ml, out, status, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace cb
