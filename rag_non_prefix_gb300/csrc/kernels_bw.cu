// Bandwidth-bound kernels of the blended prefill: embedding gather, RoPE re-rotation
// of cached keys, RMSNorm, RoPE of fresh q/k, KV deviation, compaction + KV scatter,
// LM head and argmax.  All use 16-byte vector accesses; rows are independent.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace cb {

static inline int grid_for(long long work, int per_block, int cap = 152 * 16) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return static_cast<int>(g);
}

// ----------------------------------------------------------------------------- embedding
template <typename T>
__global__ void embed_kernel(const T* __restrict__ E, const int32_t* __restrict__ ids, int d, int vocab,
                             float* __restrict__ h, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x;
  int id = ids[row];
  if (id < 0 || id >= vocab) {  // out-of-range token id: flag it and read row 0 instead
    if (threadIdx.x == 0) set_status(status, ST_RANGE);
    id = 0;
  }
  const T* src = E + static_cast<size_t>(id) * d;
  float* dst = h + static_cast<size_t>(row) * d;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float f[8];
    load8(src + c, f);
    store8(dst + c, f);
  }
}

cudaError_t launch_embed(const void* embed, const int32_t* ids, int n_rows, int d, int vocab, cb_dtype dt, float* h,
                         int32_t* status, cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  if (dt == CB_BF16)
    launch_chain(embed_kernel<bf16>, dim3(n_rows), dim3(128), 0, s, static_cast<const bf16*>(embed), ids, d, vocab, h, status);
  else
    launch_chain(embed_kernel<float>, dim3(n_rows), dim3(128), 0, s, static_cast<const float*>(embed), ids, d, vocab, h, status);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- re-rotation
// K rows: pairs (i, i + dh/2) of each head rotated by the angle delta * inv_freq_i,
// whose (cos, sin) come from cs[i].  V rows are copied.  One thread owns 8 pairs of
// K (two 16-byte vectors of a row) or one 16-byte vector of V.
template <typename T>
__device__ __forceinline__ void rerotate_item(const T* __restrict__ ks, T* __restrict__ kd, const T* __restrict__ vs,
                                              T* __restrict__ vd, long long t, int kvw, int head_dim,
                                              const float2* __restrict__ cs) {
  const int half = head_dim / 2;
  const int kthreads = kvw / 16;
  const int vthreads = vs ? kvw / 8 : 0;
  const int per_row = kthreads + vthreads;
  const long long row = t / per_row;
  const int w = static_cast<int>(t - row * per_row);
  if (w < kthreads) {
    const int cpr = half / 8;  // 8-pair chunks per head
    const int head = w / cpr, c = w - head * cpr;
    const size_t base = static_cast<size_t>(row) * kvw + static_cast<size_t>(head) * head_dim + c * 8;
    float a[8], b[8], na[8], nb[8];
    load8(ks + base, a);
    load8(ks + base + half, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 r = cs[c * 8 + j];
      na[j] = a[j] * r.x - b[j] * r.y;
      nb[j] = b[j] * r.x + a[j] * r.y;
    }
    store8(kd + base, na);
    store8(kd + base + half, nb);
  } else {
    const size_t base = static_cast<size_t>(row) * kvw + (w - kthreads) * 8;
    float f[8];
    load8(vs + base, f);
    store8(vd + base, f);
  }
}

template <typename T>
__global__ void rerotate_batched_kernel(const RerotSeg* __restrict__ segs, int n_kv_heads, int head_dim,
                                        const float2* __restrict__ table, int max_pos, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const RerotSeg sg = segs[blockIdx.y];
  const int kvw = n_kv_heads * head_dim;
  if (sg.delta < 0 || sg.delta >= max_pos) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, ST_RANGE);
    return;
  }
  const float2* cs = table + static_cast<size_t>(sg.delta) * (head_dim / 2);
  const int per_row = kvw / 16 + (sg.v_src ? kvw / 8 : 0);
  const long long total = static_cast<long long>(sg.n_rows) * per_row;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x)
    rerotate_item<T>(static_cast<const T*>(sg.k_src), static_cast<T*>(sg.k_dst), static_cast<const T*>(sg.v_src),
                     static_cast<T*>(sg.v_dst), t, kvw, head_dim, cs);
}

struct CosSin {
  float2 v[64];
};

template <typename T>
__global__ void rerotate_single_kernel(const T* __restrict__ ks, T* __restrict__ kd, const T* __restrict__ vs,
                                       T* __restrict__ vd, int n_rows, int kvw, int head_dim, CosSin cs) {
  const int per_row = kvw / 16 + (vs ? kvw / 8 : 0);
  const long long total = static_cast<long long>(n_rows) * per_row;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x)
    rerotate_item<T>(ks, kd, vs, vd, t, kvw, head_dim, cs.v);
}

cudaError_t launch_rerotate(const RerotSeg* segs, int n_segs, int max_rows, int n_kv_heads, int head_dim,
                            const float2* rope_table, int max_pos, cb_dtype dt, int32_t* status, cudaStream_t s) {
  if (n_segs <= 0 || max_rows <= 0) return cudaSuccess;
  const int kvw = n_kv_heads * head_dim;
  const long long work = static_cast<long long>(max_rows) * (kvw / 16 + kvw / 8);
  // About 32 CTAs per SM over all segments (the stand-alone launch's size), each striding
  // over its segment: one CTA per 256 items of every segment made hundreds of thousands of
  // short CTAs for the 960 chunk-layers of a 60-layer batch (measured on GB300: 4.03 GB in
  // 0.90 ms, 66 % of the copy bandwidth, against 92 % for the stand-alone launch).
  const int per_seg = std::max(1, (152 * 32 + n_segs - 1) / n_segs);
  const int gx = grid_for(work, 256, per_seg);
  dim3 grid(gx, n_segs);
  if (dt == CB_BF16)
    launch_chain(rerotate_batched_kernel<bf16>, dim3(grid), dim3(256), 0, s, segs, n_kv_heads, head_dim, rope_table, max_pos, status);
  else
    launch_chain(rerotate_batched_kernel<float>, dim3(grid), dim3(256), 0, s, segs, n_kv_heads, head_dim, rope_table, max_pos, status);
  return cudaGetLastError();
}

cudaError_t launch_rerotate_single(const void* k_src, void* k_dst, const void* v_src, void* v_dst, int n_rows,
                                   int n_kv_heads, int head_dim, const float* cs_host, cb_dtype dt, cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  CosSin cs;
  for (int i = 0; i < head_dim / 2; ++i) cs.v[i] = make_float2(cs_host[2 * i], cs_host[2 * i + 1]);
  const int kvw = n_kv_heads * head_dim;
  const long long work = static_cast<long long>(n_rows) * (kvw / 16 + (v_src ? kvw / 8 : 0));
  const int g = grid_for(work, 256, 152 * 32);
  if (dt == CB_BF16)
    rerotate_single_kernel<bf16><<<g, 256, 0, s>>>(static_cast<const bf16*>(k_src), static_cast<bf16*>(k_dst),
                                                   static_cast<const bf16*>(v_src), static_cast<bf16*>(v_dst), n_rows,
                                                   kvw, head_dim, cs);
  else
    rerotate_single_kernel<float><<<g, 256, 0, s>>>(static_cast<const float*>(k_src), static_cast<float*>(k_dst),
                                                    static_cast<const float*>(v_src), static_cast<float*>(v_dst),
                                                    n_rows, kvw, head_dim, cs);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- RMSNorm
__device__ __forceinline__ float block_sum_256(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = (l < (blockDim.x >> 5)) ? red[l] : 0.f;
  t = warp_sum(t);
  __syncthreads();
  return t;
}

// One CTA of 256 threads per row.  Rows of up to 8192 (= 256 x 8 x CH) elements stay in
// registers between the sum of squares and the scaled write (one read of h); longer rows
// are read twice.  Thread t always owns chunks t, t + 256, ... of 8 elements.
template <typename T, bool IN_REGS>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ h, int d, float eps, T* __restrict__ x) {
  pdl_trigger();
  pdl_wait();
  constexpr int CH = 4;
  __shared__ float red[32];
  const size_t row = blockIdx.x;
  const float* src = h + row * d;
  T* dst = x + row * d;
  float ss = 0.f;
  if (IN_REGS) {
    float f[CH][8];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int c = (threadIdx.x + k * 256) * 8;
      if (c < d) {
        load8(src + c, f[k]);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss += f[k][j] * f[k][j];
      }
    }
    ss = block_sum_256(ss, red);
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int c = (threadIdx.x + k * 256) * 8;
      if (c < d) {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[k][j] *= inv;
        store8(dst + c, f[k]);
      }
    }
  } else {
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
      float f[8];
      load8(src + c, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) ss += f[j] * f[j];
    }
    ss = block_sum_256(ss, red);
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
      float f[8];
      load8(src + c, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] *= inv;
      store8(dst + c, f);
    }
  }
}

cudaError_t launch_rmsnorm(const float* h, int n_rows, int d, float eps, void* x, cb_dtype dt, cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  const bool regs = d <= 256 * 8 * 4;
  if (dt == CB_BF16) {
    if (regs)
      launch_chain(rmsnorm_kernel<bf16, true>, dim3(n_rows), dim3(256), 0, s, h, d, eps, static_cast<bf16*>(x));
    else
      launch_chain(rmsnorm_kernel<bf16, false>, dim3(n_rows), dim3(256), 0, s, h, d, eps, static_cast<bf16*>(x));
  } else {
    if (regs)
      launch_chain(rmsnorm_kernel<float, true>, dim3(n_rows), dim3(256), 0, s, h, d, eps, static_cast<float*>(x));
    else
      launch_chain(rmsnorm_kernel<float, false>, dim3(n_rows), dim3(256), 0, s, h, d, eps, static_cast<float*>(x));
  }
  return cudaGetLastError();
}

// final norm of selected rows into fp32 (LM-head input)
__global__ void last_rows_norm_kernel(const float* __restrict__ h, const int32_t* __restrict__ rows, int d, float eps,
                                      float* __restrict__ x) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const float* src = h + static_cast<size_t>(rows[blockIdx.x]) * d;
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float f[8];
    load8(src + c, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += f[j] * f[j];
  }
  ss = block_sum_256(ss, red);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  float* dst = x + static_cast<size_t>(blockIdx.x) * d;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float f[8];
    load8(src + c, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] *= inv;
    store8(dst + c, f);
  }
}

cudaError_t launch_last_rows_norm(const float* h, const int32_t* rows, int n, int d, float eps, float* x_out,
                                  cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  launch_chain(last_rows_norm_kernel, dim3(n), dim3(256), 0, s, h, rows, d, eps, x_out);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- RoPE of fresh q and k
// Rotate-half RoPE of one head: elements j..j+7 (a) and j+dh/2..j+dh/2+7 (b) turn by the
// angles of pairs j..j+7 at the row's position (cs = the table row of that position).
// Applied where the fresh q and k are consumed (deviation, scatter), so the projection
// output is read once.
__device__ __forceinline__ void rope8(const float* a, const float* b, const float2* cs, float* ra, float* rb) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float2 r = cs[e];
    ra[e] = a[e] * r.x - b[e] * r.y;
    rb[e] = b[e] * r.x + a[e] * r.y;
  }
}

// ----------------------------------------------------------------------------- KV deviation
// mode 0: squared L2 of [k; v]_fresh - [k; v]_fused;  1: K part only;  2: V part only;
// 3: 1 - cos([k; v]_fresh, [k; v]_fused) (zero against zero: 0, zero against non-zero: 1).
// Sums run in fp32: `acc` holds the squared difference (modes 0-2) or the dot product (3),
// `aa` and `bb` the squared norms of the two rows (mode 3).
struct DevAcc {
  float acc = 0.f, aa = 0.f, bb = 0.f;
  __device__ __forceinline__ void add(float a, float b, bool cosine) {
    if (cosine) {
      acc = fmaf(a, b, acc);
      aa = fmaf(a, a, aa);
      bb = fmaf(b, b, bb);
    } else {
      const float e = a - b;
      acc = fmaf(e, e, acc);
    }
  }
  // warp-reduced result, valid in every lane
  __device__ __forceinline__ float finish(bool cosine) {
    const float s = warp_sum(acc);
    if (!cosine) return s;
    const float na = warp_sum(aa), nb = warp_sum(bb);
    if (na == 0.f && nb == 0.f) return 0.f;
    if (na == 0.f || nb == 0.f) return 1.f;
    return 1.f - s / (sqrtf(na) * sqrtf(nb));
  }
};

template <typename T>
__device__ __forceinline__ float dev_row(const float* __restrict__ kn, const float* __restrict__ vn,
                                         const T* __restrict__ kf, const T* __restrict__ vf, int kvw, int mode) {
  const bool cosine = mode == 3;
  DevAcc d;
  for (int c = (threadIdx.x & 31) * 8; c < kvw; c += 256) {
    float a[8], b[8];
    if (mode != 2) {
      load8(kn + c, a);
      load8(kf + c, b);
#pragma unroll
      for (int j = 0; j < 8; ++j) d.add(a[j], b[j], cosine);
    }
    if (mode != 1) {
      load8(vn + c, a);
      load8(vf + c, b);
#pragma unroll
      for (int j = 0; j < 8; ++j) d.add(a[j], b[j], cosine);
    }
  }
  return d.finish(cosine);
}

// One warp per row of R; only cached rows (position < Nc of their request) are candidates.
// The fresh k of the projection output is rotated to the row's position here (RoPE), then
// compared with the fused cache, whose cached rows were re-rotated to the same position.
template <typename T>
__global__ void deviation_rows_kernel(const float* __restrict__ qkv, int n_rows, const int32_t* __restrict__ pos,
                                      const int32_t* __restrict__ req, const ReqDev* __restrict__ reqs, int layer,
                                      int q_width, int kvw, int head_dim, int mode, const float2* __restrict__ table,
                                      int max_pos, float* __restrict__ dev, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int warps = blockDim.x >> 5;
  const int row = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  const int p = pos[row];
  const ReqDev rq = reqs[req[row]];
  if (p >= rq.n_cached) {
    if (lane == 0) dev[row] = 0.f;
    return;
  }
  if (p < 0 || p >= max_pos) {
    if (lane == 0) set_status(status, ST_RANGE);
    return;
  }
  const size_t width = static_cast<size_t>(q_width) + 2 * kvw;
  const float* kn = qkv + static_cast<size_t>(row) * width + q_width;
  const float* vn = kn + kvw;
  const size_t off = static_cast<size_t>(layer) * rq.layer_stride + static_cast<size_t>(p) * kvw;
  const T* kf = static_cast<const T*>(rq.k) + off;
  const T* vf = static_cast<const T*>(rq.v) + off;
  const int half = head_dim / 2, cpr = half / 8;
  const float2* cs = table + static_cast<size_t>(p) * half;
  const bool cosine = mode == 3;
  DevAcc acc;
  if (mode != 2) {
    for (int w = lane; w < kvw / 16; w += 32) {  // 8 rotation pairs per step
      const int head = w / cpr, j = (w - head * cpr) * 8;
      const int o = head * head_dim + j;
      float a[8], b[8], ra[8], rb[8], fa[8], fb[8];
      load8(kn + o, a);
      load8(kn + o + half, b);
      rope8(a, b, cs + j, ra, rb);
      load8(kf + o, fa);
      load8(kf + o + half, fb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc.add(ra[e], fa[e], cosine);
        acc.add(rb[e], fb[e], cosine);
      }
    }
  }
  if (mode != 1) {
    for (int c = lane * 8; c < kvw; c += 256) {
      float a[8], b[8];
      load8(vn + c, a);
      load8(vf + c, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc.add(a[e], b[e], cosine);
    }
  }
  const float r = acc.finish(cosine);
  if (lane == 0) dev[row] = r;
}

cudaError_t launch_deviation_rows(const float* qkv, int n_rows, const int32_t* pos, const int32_t* req,
                                  const ReqDev* reqs, int layer, int n_heads, int n_kv_heads, int head_dim, int mode,
                                  const float2* rope_table, int max_pos, cb_dtype dt, float* dev, int32_t* status,
                                  cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  const int blocks = (n_rows + 7) / 8;
  if (dt == CB_BF16)
    launch_chain(deviation_rows_kernel<bf16>, dim3(blocks), dim3(256), 0, s, qkv, n_rows, pos, req, reqs, layer, n_heads * head_dim,
                                                       n_kv_heads * head_dim, head_dim, mode, rope_table, max_pos,
                                                       dev, status);
  else
    launch_chain(deviation_rows_kernel<float>, dim3(blocks), dim3(256), 0, s, qkv, n_rows, pos, req, reqs, layer, n_heads * head_dim,
                                                        n_kv_heads * head_dim, head_dim, mode, rope_table, max_pos,
                                                        dev, status);
  return cudaGetLastError();
}

template <typename T>
__global__ void deviation_plain_kernel(const float* __restrict__ kn, const float* __restrict__ vn,
                                       const T* __restrict__ kf, const T* __restrict__ vf,
                                       const int32_t* __restrict__ idx, int n, int kvw, int mode,
                                       float* __restrict__ dev) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= n) return;
  const size_t f = static_cast<size_t>(idx ? idx[row] : row) * kvw;
  const size_t r = static_cast<size_t>(row) * kvw;
  const float d = dev_row<T>(kn + r, vn + r, kf + f, vf + f, kvw, mode);
  if ((threadIdx.x & 31) == 0) dev[row] = d;
}

cudaError_t launch_deviation_plain(const float* k_new, const float* v_new, const void* k_fus, const void* v_fus,
                                   const int32_t* idx, int n, int kv_width, int mode, cb_dtype dt, float* dev,
                                   cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int blocks = (n + 7) / 8;
  if (dt == CB_BF16)
    deviation_plain_kernel<bf16><<<blocks, 256, 0, s>>>(k_new, v_new, static_cast<const bf16*>(k_fus),
                                                        static_cast<const bf16*>(v_fus), idx, n, kv_width, mode, dev);
  else
    deviation_plain_kernel<float><<<blocks, 256, 0, s>>>(k_new, v_new, static_cast<const float*>(k_fus),
                                                         static_cast<const float*>(v_fus), idx, n, kv_width, mode,
                                                         dev);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- compaction + KV scatter
// For every row t of S: q and k of its source row rotated at the row's position (RoPE),
// q -> q_out[t] (model dtype), k and v -> the fused cache row at that position; hidden
// state h_in[src] -> h_out[t] when the set shrank (h_out != h_in).
template <typename T>
__global__ void post_qkv_kernel(const float* __restrict__ qkv, const int32_t* __restrict__ s_src,
                                const int32_t* __restrict__ s_pos, const int32_t* __restrict__ s_req,
                                const ReqDev* __restrict__ reqs, int layer, int q_width, int kvw, int head_dim,
                                const float2* __restrict__ table, int max_pos, T* __restrict__ q_out,
                                const float* __restrict__ h_in, float* __restrict__ h_out, int d, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int src = s_src ? s_src[t] : t;
  const int p = s_pos[t];
  const ReqDev rq = reqs[s_req[t]];
  if (p < 0 || p >= rq.n_tokens || p >= max_pos) {
    if (threadIdx.x == 0) set_status(status, ST_RANGE);
    return;
  }
  const size_t width = static_cast<size_t>(q_width) + 2 * kvw;
  const float* row = qkv + static_cast<size_t>(src) * width;
  const size_t off = static_cast<size_t>(layer) * rq.layer_stride + static_cast<size_t>(p) * kvw;
  T* kd = static_cast<T*>(rq.k) + off;
  T* vd = static_cast<T*>(rq.v) + off;
  T* qd = q_out + static_cast<size_t>(t) * q_width;
  const int half = head_dim / 2, cpr = half / 8;
  const float2* cs = table + static_cast<size_t>(p) * half;
  const int qsteps = q_width / 16, steps = qsteps + kvw / 16;
  for (int w = threadIdx.x; w < steps; w += blockDim.x) {  // 8 rotation pairs of q or k per step
    const bool is_k = w >= qsteps;
    const int ww = is_k ? w - qsteps : w;
    const int head = ww / cpr, j = (ww - head * cpr) * 8;
    const int o = head * head_dim + j;
    const float* a = row + (is_k ? q_width : 0) + o;
    float fa[8], fb[8], ra[8], rb[8];
    load8(a, fa);
    load8(a + half, fb);
    rope8(fa, fb, cs + j, ra, rb);
    T* dst = (is_k ? kd : qd) + o;
    store8(dst, ra);
    store8(dst + half, rb);
  }
  for (int c = threadIdx.x * 8; c < kvw; c += blockDim.x * 8) {
    float f[8];
    load8(row + q_width + kvw + c, f);
    store8(vd + c, f);
  }
  if (h_out != h_in) {
    const float* hs = h_in + static_cast<size_t>(src) * d;
    float* hd = h_out + static_cast<size_t>(t) * d;
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
      float f[8];
      load8(hs + c, f);
      store8(hd + c, f);
    }
  }
}

cudaError_t launch_post_qkv(const float* qkv, int n_s_rows, const int32_t* s_src, const int32_t* s_pos,
                            const int32_t* s_req, const ReqDev* reqs, int layer, int n_heads, int n_kv_heads,
                            int head_dim, const float2* rope_table, int max_pos, cb_dtype dt, void* q_out,
                            const float* h_in, float* h_out, int d, int32_t* status, cudaStream_t s) {
  if (n_s_rows <= 0) return cudaSuccess;
  if (dt == CB_BF16)
    launch_chain(post_qkv_kernel<bf16>, dim3(n_s_rows), dim3(256), 0, s, qkv, s_src, s_pos, s_req, reqs, layer, n_heads * head_dim,
                                                   n_kv_heads * head_dim, head_dim, rope_table, max_pos,
                                                   static_cast<bf16*>(q_out), h_in, h_out, d, status);
  else
    launch_chain(post_qkv_kernel<float>, dim3(n_s_rows), dim3(256), 0, s, qkv, s_src, s_pos, s_req, reqs, layer, n_heads * head_dim,
                                                    n_kv_heads * head_dim, head_dim, rope_table, max_pos,
                                                    static_cast<float*>(q_out), h_in, h_out, d, status);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- outputs
__global__ void write_hidden_kernel(const float* __restrict__ h, const int32_t* __restrict__ s_pos, int row0, int d,
                                    float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int t = row0 + blockIdx.x;
  const float* src = h + static_cast<size_t>(t) * d;
  float* dst = out + static_cast<size_t>(s_pos[t]) * d;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float f[8];
    load8(src + c, f);
    store8(dst + c, f);
  }
}

cudaError_t launch_write_hidden(const float* h, const int32_t* s_pos, int row0, int n, int d, float* out,
                                cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  launch_chain(write_hidden_kernel, dim3(n), dim3(256), 0, s, h, s_pos, row0, d, out);
  return cudaGetLastError();
}

constexpr int LM_MAX_REQ = 16;

// logits[r][v] = <x[r], W[v]>: one warp per vocabulary row, every request at once.
template <typename T>
__global__ void lm_head_kernel(const float* __restrict__ x, int n_req, int d, const T* __restrict__ w, int vocab,
                               float* __restrict__ logits) {
  pdl_trigger();
  pdl_wait();
  const int v = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (v >= vocab) return;
  const int lane = threadIdx.x & 31;
  float acc[LM_MAX_REQ];
#pragma unroll
  for (int r = 0; r < LM_MAX_REQ; ++r) acc[r] = 0.f;
  const T* wr = w + static_cast<size_t>(v) * d;
  for (int c = lane * 8; c < d; c += 256) {
    float wf[8];
    load8(wr + c, wf);
#pragma unroll
    for (int r = 0; r < LM_MAX_REQ; ++r) {
      if (r < n_req) {
        float xf[8];
        load8(x + static_cast<size_t>(r) * d + c, xf);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r] += wf[j] * xf[j];
      }
    }
  }
#pragma unroll
  for (int r = 0; r < LM_MAX_REQ; ++r) {
    if (r < n_req) {
      const float t = warp_sum(acc[r]);
      if (lane == 0) logits[static_cast<size_t>(r) * vocab + v] = t;
    }
  }
}

cudaError_t launch_lm_head(const float* x, int n_req, int d, const void* w, int vocab, cb_dtype dt, float* logits,
                           cudaStream_t s) {
  if (n_req <= 0) return cudaSuccess;
  // a row or two (the decode step, a single blended request): the weight-streaming GEMV
  if (n_req <= GEMV_MAX_ROWS && d % 8 == 0 && (reinterpret_cast<uintptr_t>(w) & 15u) == 0 &&
      (reinterpret_cast<uintptr_t>(x) & 15u) == 0)
    return launch_gemv_f32a(x, w, n_req, vocab, d, logits, dt, s);
  for (int r0 = 0; r0 < n_req; r0 += LM_MAX_REQ) {
    const int nr = n_req - r0 < LM_MAX_REQ ? n_req - r0 : LM_MAX_REQ;
    const int blocks = (vocab + 7) / 8;
    if (dt == CB_BF16)
      launch_chain(lm_head_kernel<bf16>, dim3(blocks), dim3(256), 0, s, x + static_cast<size_t>(r0) * d, nr, d, static_cast<const bf16*>(w),
                                                  vocab, logits + static_cast<size_t>(r0) * vocab);
    else
      launch_chain(lm_head_kernel<float>, dim3(blocks), dim3(256), 0, s, x + static_cast<size_t>(r0) * d, nr, d,
                                                   static_cast<const float*>(w), vocab,
                                                   logits + static_cast<size_t>(r0) * vocab);
  }
  return cudaGetLastError();
}

// argmax per request; ties go to the lowest token id; NaN logits never win.
__global__ void argmax_kernel(const float* __restrict__ logits, int vocab, int32_t* const* outs,
                              int32_t* __restrict__ out_dev) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sv[32];
  __shared__ int si[32];
  const float* l = logits + static_cast<size_t>(blockIdx.x) * vocab;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int v = threadIdx.x; v < vocab; v += blockDim.x) {
    const float x = l[v];
    if (x > best || (x == best && v < bi)) {
      best = x;
      bi = v;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ob > best || (ob == best && oi < bi)) {
      best = ob;
      bi = oi;
    }
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[w] = best;
    si[w] = bi;
  }
  __syncthreads();
  if (w == 0) {
    best = lane < (blockDim.x >> 5) ? sv[lane] : -INFINITY;
    bi = lane < (blockDim.x >> 5) ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    if (lane == 0) {
      if (bi == 0x7fffffff) bi = 0;
      if (out_dev) out_dev[blockIdx.x] = bi;
      if (outs && outs[blockIdx.x]) *outs[blockIdx.x] = bi;
    }
  }
}

cudaError_t launch_argmax(const float* logits, int n_req, int vocab, int32_t* const* outs, int32_t* out_dev,
                          cudaStream_t s) {
  if (n_req <= 0) return cudaSuccess;
  launch_chain(argmax_kernel, dim3(n_req), dim3(1024), 0, s, logits, vocab, outs, out_dev);
  return cudaGetLastError();
}

}  // namespace cb
