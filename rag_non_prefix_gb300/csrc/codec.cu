// KIVI-style KV codec of cached chunks ([P2] KV量子化とメモリ管理 / 非対称量子化: keys are
// quantised per channel, values per token, to int8 or int4) and the decoder that turns a
// chunk's codes back into re-rotated K and V rows of the fused cache in one pass.
//
// A group is quantised asymmetrically by its minimum and maximum: scale = (max - min) /
// (2^b - 1), code = clamp(rint((x - min) / scale), 0, 2^b - 1) (code 0 when scale is 0), and
// decoded as min + code * scale.  A key group is one channel of one KV head of one layer over
// all the chunk's tokens; a value group is one token's head_dim channels of one KV head.
// The codes are decided with single IEEE float32 operations (__fsub_rn, __fdiv_rn, rintf),
// so they do not depend on contraction or on the order of operations.
#include "common.cuh"
#include "internal.h"

namespace cb {

namespace {

template <int BITS>
__device__ __forceinline__ int quantise(float x, float mn, float scale) {
  if (!(scale > 0.f)) return 0;
  const float q = rintf(__fdiv_rn(__fsub_rn(x, mn), scale));
  return static_cast<int>(fminf(fmaxf(q, 0.f), static_cast<float>((1 << BITS) - 1)));
}

// ----------------------------------------------------------------------------- encode: keys
// One block per (layer, KV head), one thread per channel: min / max down the channel over
// the n tokens, then the codes.  Reads are coalesced along the channels of a token row.
template <typename T, int BITS>
__global__ void encode_k_kernel(const T* __restrict__ k, int n, int n_kv_heads, int head_dim, uint8_t* __restrict__ blob) {
  const int layer = blockIdx.x / n_kv_heads, h = blockIdx.x - layer * n_kv_heads;
  const int c = threadIdx.x;
  const CodecLayout lay = codec_layout(n, n_kv_heads, head_dim, BITS);
  uint8_t* blk = blob + static_cast<size_t>(layer) * lay.bytes;
  const size_t kvw = static_cast<size_t>(n_kv_heads) * head_dim;
  const T* src = k + static_cast<size_t>(layer) * n * kvw + static_cast<size_t>(h) * head_dim + c;
  float mn = INFINITY, mx = -INFINITY;
  for (int t = 0; t < n; ++t) {
    const float x = to_f(src[static_cast<size_t>(t) * kvw]);
    mn = fminf(mn, x);
    mx = fmaxf(mx, x);
  }
  const float scale = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>((1 << BITS) - 1));
  reinterpret_cast<float*>(blk + lay.ks)[h * head_dim + c] = scale;
  reinterpret_cast<float*>(blk + lay.kz)[h * head_dim + c] = mn;
  uint8_t* codes = blk + lay.kc;
  for (int t = 0; t < n; ++t) {
    const int q = quantise<BITS>(to_f(src[static_cast<size_t>(t) * kvw]), mn, scale);
    const size_t e = (static_cast<size_t>(t) * n_kv_heads + h) * head_dim + c;  // element index of the row
    if (BITS == 8) {
      codes[e] = static_cast<uint8_t>(q);
    } else {
      const int hi = __shfl_down_sync(0xffffffffu, q, 1);  // the odd channel's code
      if ((c & 1) == 0) codes[e >> 1] = static_cast<uint8_t>(q | (hi << 4));
    }
  }
}

// ----------------------------------------------------------------------------- encode: values
// One warp per (layer, token, KV head) row of head_dim channels; lane owns head_dim/32
// consecutive channels.
template <typename T, int BITS>
__global__ void encode_v_kernel(const T* __restrict__ v, int L, int n, int n_kv_heads, int head_dim,
                                uint8_t* __restrict__ blob) {
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long rows_per_layer = static_cast<long long>(n) * n_kv_heads;
  if (row >= L * rows_per_layer) return;
  const int layer = static_cast<int>(row / rows_per_layer);
  const long long r = row - layer * rows_per_layer;  // t * Hkv + h within the layer
  const CodecLayout lay = codec_layout(n, n_kv_heads, head_dim, BITS);
  uint8_t* blk = blob + static_cast<size_t>(layer) * lay.bytes;
  const int per = head_dim / 32;  // 2 or 4 channels per lane
  const T* src = v + (static_cast<size_t>(layer) * rows_per_layer + r) * head_dim + lane * per;
  float x[4];
  float mn = INFINITY, mx = -INFINITY;
  for (int j = 0; j < per; ++j) {
    x[j] = to_f(src[j]);
    mn = fminf(mn, x[j]);
    mx = fmaxf(mx, x[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const float scale = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>((1 << BITS) - 1));
  if (lane == 0) {
    reinterpret_cast<float*>(blk + lay.vs)[r] = scale;
    reinterpret_cast<float*>(blk + lay.vz)[r] = mn;
  }
  uint8_t* codes = blk + lay.vc + static_cast<size_t>(r) * head_dim * BITS / 8;
  for (int j = 0; j < per; j += (BITS == 8 ? 1 : 2)) {
    const int q0 = quantise<BITS>(x[j], mn, scale);
    if (BITS == 8) {
      codes[lane * per + j] = static_cast<uint8_t>(q0);
    } else {
      const int q1 = quantise<BITS>(x[j + 1], mn, scale);
      codes[(lane * per + j) >> 1] = static_cast<uint8_t>(q0 | (q1 << 4));
    }
  }
}

// ----------------------------------------------------------------------------- decode + re-rotation
// 8 codes starting at channel c of a row (c a multiple of 8) as floats.
template <int BITS>
__device__ __forceinline__ void load_codes8(const uint8_t* row, int c, float* f) {
  if (BITS == 8) {
    const uint2 u = *reinterpret_cast<const uint2*>(row + c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[j] = static_cast<float>((u.x >> (8 * j)) & 255u);
      f[4 + j] = static_cast<float>((u.y >> (8 * j)) & 255u);
    }
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(row + c / 2);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = static_cast<float>((u >> (4 * j)) & 15u);
  }
}

// One (token, KV head) row of one chunk-layer block: head_dim/16 threads, thread m owning
// channels [8m, 8m + 8) and their rotation partners [dh/2 + 8m, dh/2 + 8m + 8).  K is
// dequantised and turned by R(delta) (cs = the rotary (cos, sin) row of delta), V dequantised.
template <typename T, int BITS>
__device__ __forceinline__ void decode_row(const uint8_t* __restrict__ blk, const CodecLayout& lay, int n_kv_heads,
                                           int head_dim, long long r, int m, T* __restrict__ kd,
                                           T* __restrict__ vd, const float2* __restrict__ cs) {
  const int h = static_cast<int>(r % n_kv_heads);
  const int half = head_dim / 2, a0 = 8 * m, b0 = half + 8 * m;
  const size_t row_bytes = static_cast<size_t>(head_dim) * BITS / 8;
  const float* ks = reinterpret_cast<const float*>(blk + lay.ks) + h * head_dim;
  const float* kz = reinterpret_cast<const float*>(blk + lay.kz) + h * head_dim;
  float ca[8], cb_[8], sa[8], sb[8], za[8], zb[8], a[8], b[8];
  const uint8_t* krow = blk + lay.kc + static_cast<size_t>(r) * row_bytes;
  load_codes8<BITS>(krow, a0, ca);
  load_codes8<BITS>(krow, b0, cb_);
  load8(ks + a0, sa);
  load8(ks + b0, sb);
  load8(kz + a0, za);
  load8(kz + b0, zb);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float x = fmaf(ca[j], sa[j], za[j]), y = fmaf(cb_[j], sb[j], zb[j]);
    const float2 rot = cs[a0 + j];
    a[j] = x * rot.x - y * rot.y;
    b[j] = y * rot.x + x * rot.y;
  }
  T* kr = kd + static_cast<size_t>(r) * head_dim;
  store8(kr + a0, a);
  store8(kr + b0, b);
  const float vs = reinterpret_cast<const float*>(blk + lay.vs)[r];
  const float vz = reinterpret_cast<const float*>(blk + lay.vz)[r];
  const uint8_t* vrow = blk + lay.vc + static_cast<size_t>(r) * row_bytes;
  load_codes8<BITS>(vrow, a0, ca);
  load_codes8<BITS>(vrow, b0, cb_);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a[j] = fmaf(ca[j], vs, vz);
    b[j] = fmaf(cb_[j], vs, vz);
  }
  T* vr = vd + static_cast<size_t>(r) * head_dim;
  store8(vr + a0, a);
  store8(vr + b0, b);
}

// Batched: blockIdx.y = segment (one chunk-layer block into its fused-cache rows); the bit
// width is a property of the segment.
template <typename T, int BITS>
__device__ __forceinline__ void decode_seg(const CodecSeg& sg, int n_kv_heads, int head_dim, const float2* cs) {
  const CodecLayout lay = codec_layout(sg.n, n_kv_heads, head_dim, BITS);
  const int lpu = head_dim / 16;
  const long long units = static_cast<long long>(sg.n) * n_kv_heads;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < units * lpu;
       t += static_cast<long long>(gridDim.x) * blockDim.x)
    decode_row<T, BITS>(sg.block, lay, n_kv_heads, head_dim, t / lpu, static_cast<int>(t % lpu),
                        static_cast<T*>(sg.k_dst), static_cast<T*>(sg.v_dst), cs);
}

template <typename T>
__global__ void decode_batched_kernel(const CodecSeg* __restrict__ segs, int n_kv_heads, int head_dim,
                                      const float2* __restrict__ table, int max_pos, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const CodecSeg sg = segs[blockIdx.y];
  if (sg.delta < 0 || sg.delta >= max_pos || (sg.bits != 8 && sg.bits != 4)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, ST_RANGE);
    return;
  }
  const float2* cs = table + static_cast<size_t>(sg.delta) * (head_dim / 2);
  if (sg.bits == 8)
    decode_seg<T, 8>(sg, n_kv_heads, head_dim, cs);
  else
    decode_seg<T, 4>(sg, n_kv_heads, head_dim, cs);
}

struct CosSin64 {
  float2 v[64];
};

// Standalone: blockIdx.y = layer of one chunk blob, all rows turned by the same delta.
template <typename T, int BITS>
__global__ void decode_blob_kernel(const uint8_t* __restrict__ blob, int n, int n_kv_heads, int head_dim,
                                   T* __restrict__ k_out, T* __restrict__ v_out, CosSin64 cs) {
  const CodecLayout lay = codec_layout(n, n_kv_heads, head_dim, BITS);
  const int layer = blockIdx.y;
  const int lpu = head_dim / 16;
  const long long units = static_cast<long long>(n) * n_kv_heads;
  const size_t off = static_cast<size_t>(layer) * units * head_dim;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < units * lpu;
       t += static_cast<long long>(gridDim.x) * blockDim.x)
    decode_row<T, BITS>(blob + static_cast<size_t>(layer) * lay.bytes, lay, n_kv_heads, head_dim, t / lpu,
                        static_cast<int>(t % lpu), k_out + off, v_out + off, cs.v);
}

int decode_grid(long long units, int head_dim, int cap) {
  const long long threads = units * (head_dim / 16);
  long long g = (threads + 255) / 256;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_kv_encode(const void* k, const void* v, int L, int n, int n_kv_heads, int head_dim, int bits,
                             cb_dtype dt, void* blob, cudaStream_t s) {
  uint8_t* b = static_cast<uint8_t*>(blob);
  const long long vrows = static_cast<long long>(L) * n * n_kv_heads;
  const int vblocks = static_cast<int>((vrows + 7) / 8);
#define CB_ENC(T, B)                                                                                       \
  encode_k_kernel<T, B><<<L * n_kv_heads, head_dim, 0, s>>>(static_cast<const T*>(k), n, n_kv_heads, head_dim, b); \
  encode_v_kernel<T, B><<<vblocks, 256, 0, s>>>(static_cast<const T*>(v), L, n, n_kv_heads, head_dim, b)
  if (dt == CB_BF16) {
    if (bits == 8) { CB_ENC(bf16, 8); } else { CB_ENC(bf16, 4); }
  } else {
    if (bits == 8) { CB_ENC(float, 8); } else { CB_ENC(float, 4); }
  }
#undef CB_ENC
  return cudaGetLastError();
}

cudaError_t launch_codec_decode(const CodecSeg* segs, int n_segs, int max_n, int n_kv_heads, int head_dim,
                                const float2* rope_table, int max_pos, cb_dtype dt, int32_t* status, cudaStream_t s) {
  if (n_segs <= 0 || max_n <= 0) return cudaSuccess;
  const dim3 grid(decode_grid(static_cast<long long>(max_n) * n_kv_heads, head_dim, 1 << 16), n_segs);
  if (dt == CB_BF16)
    launch_chain(decode_batched_kernel<bf16>, grid, dim3(256), 0, s, segs, n_kv_heads, head_dim, rope_table, max_pos,
                 status);
  else
    launch_chain(decode_batched_kernel<float>, grid, dim3(256), 0, s, segs, n_kv_heads, head_dim, rope_table, max_pos,
                 status);
  return cudaGetLastError();
}

cudaError_t launch_codec_decode_blob(const void* blob, int L, int n, int n_kv_heads, int head_dim, int bits,
                                     const float* cs_host, cb_dtype dt, void* k_out, void* v_out, cudaStream_t s) {
  CosSin64 cs;
  for (int i = 0; i < head_dim / 2; ++i) cs.v[i] = make_float2(cs_host[2 * i], cs_host[2 * i + 1]);
  const dim3 grid(decode_grid(static_cast<long long>(n) * n_kv_heads, head_dim, 1 << 16), L);
  const uint8_t* b = static_cast<const uint8_t*>(blob);
#define CB_DECB(T, B) \
  decode_blob_kernel<T, B><<<grid, 256, 0, s>>>(b, n, n_kv_heads, head_dim, static_cast<T*>(k_out), static_cast<T*>(v_out), cs)
  if (dt == CB_BF16) {
    if (bits == 8) { CB_DECB(bf16, 8); } else { CB_DECB(bf16, 4); }
  } else {
    if (bits == 8) { CB_DECB(float, 8); } else { CB_DECB(float, 4); }
  }
#undef CB_DECB
  return cudaGetLastError();
}

}  // namespace cb
