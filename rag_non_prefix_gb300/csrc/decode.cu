// Decode attention: one new query token per sequence over its fused cache rows 0..p (p = the
// token's position, whose K/V row was just written), split along the keys so that a handful
// of sequences still fill the GPU ("split-KV"): each CTA owns one (sequence, KV head, key
// range) and all G = H / Hkv query heads of that KV head, so every K/V row is read once.
//
// Per CTA (head_dim threads, thread t owning output channel t of every head):
//   scores   warp w takes keys w, w + nwarps, ... of a 64-key block; lane l holds head_dim/32
//            channels of the key row (one coalesced row read per key) and the G dot products
//            are warp-reduced; q is pre-scaled by log2(e) / sqrt(head_dim) so scores are in
//            base-2 logits;
//   softmax  warp w updates heads w, w + nwarps, ...: block max, running max, rescale factor,
//            probabilities written back over the scores, running sum;
//   values   thread t: o[g] = o[g] * alpha[g] + sum_j p[g][j] * V[j][t].
// With one split the CTA normalises and writes the output; otherwise it writes (o, max, sum)
// of its range to the partial buffers and a second kernel merges the ranges.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace cb {

namespace {

constexpr int DEC_BK = 64;     // keys per block
constexpr int DEC_GMAX = 16;   // query heads per KV head

template <typename T, int DH>
__global__ void __launch_bounds__(DH) decode_attn_kernel(const T* __restrict__ q, const int32_t* __restrict__ pos,
                                                         const ReqDev* __restrict__ reqs, int layer, int H, int Hkv,
                                                         int split_len, int n_splits, float scale_log2,
                                                         float* __restrict__ part_o, float2* __restrict__ part_ml,
                                                         T* __restrict__ out, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  constexpr int E = DH / 32;  // channels per lane in the score pass
  constexpr int NW = DH / 32;
  __shared__ float qs[DEC_GMAX][DH];
  __shared__ float sc[DEC_GMAX][DEC_BK];
  __shared__ float m_run[DEC_GMAX], l_run[DEC_GMAX], alpha[DEC_GMAX];
  const int G = H / Hkv;
  const int seq = blockIdx.x / Hkv, kvh = blockIdx.x - seq * Hkv;
  const int split = blockIdx.y;
  const int t = threadIdx.x, w = t >> 5, lane = t & 31;
  const int p = pos[seq];
  const ReqDev rq = reqs[seq];
  if (p < 0 || p >= rq.n_tokens || G > DEC_GMAX) {
    if (t == 0 && split == 0) set_status(status, ST_RANGE);
    return;
  }
  const int k0 = split * split_len, k1 = min(p + 1, k0 + split_len);
  const size_t kvw = static_cast<size_t>(Hkv) * DH;
  const T* kbase = static_cast<const T*>(rq.k) + static_cast<size_t>(layer) * rq.layer_stride + kvh * DH;
  const T* vbase = static_cast<const T*>(rq.v) + static_cast<size_t>(layer) * rq.layer_stride + kvh * DH;
  for (int g = 0; g < G; ++g) qs[g][t] = to_f(q[(static_cast<size_t>(seq) * H + kvh * G + g) * DH + t]) * scale_log2;
  if (t < G) {
    m_run[t] = -INFINITY;
    l_run[t] = 0.f;
  }
  float o[DEC_GMAX];
#pragma unroll
  for (int g = 0; g < DEC_GMAX; ++g) o[g] = 0.f;
  __syncthreads();
  for (int kb = k0; kb < k1; kb += DEC_BK) {
    const int nb = min(DEC_BK, k1 - kb);
    for (int j = w; j < nb; j += NW) {
      const T* kr = kbase + static_cast<size_t>(kb + j) * kvw + lane * E;
      float kk[E];
#pragma unroll
      for (int e = 0; e < E; ++e) kk[e] = to_f(kr[e]);
#pragma unroll
      for (int g = 0; g < DEC_GMAX; ++g) {
        if (g < G) {
          float part = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) part = fmaf(qs[g][lane * E + e], kk[e], part);
          part = warp_sum(part);
          if (lane == 0) sc[g][j] = part;
        }
      }
    }
    __syncthreads();
    for (int g = w; g < G; g += NW) {
      const float s0 = lane < nb ? sc[g][lane] : -INFINITY;
      const float s1 = lane + 32 < nb ? sc[g][lane + 32] : -INFINITY;
      float bmax = fmaxf(s0, s1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
      const float m_old = m_run[g];
      const float m_new = fmaxf(m_old, bmax);
      const float p0 = lane < nb ? exp2f(s0 - m_new) : 0.f;
      const float p1 = lane + 32 < nb ? exp2f(s1 - m_new) : 0.f;
      if (lane < nb) sc[g][lane] = p0;
      if (lane + 32 < nb) sc[g][lane + 32] = p1;
      const float bsum = warp_sum(p0 + p1);
      if (lane == 0) {
        const float a = m_old == -INFINITY ? 0.f : exp2f(m_old - m_new);
        alpha[g] = a;
        l_run[g] = l_run[g] * a + bsum;
        m_run[g] = m_new;
      }
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < DEC_GMAX; ++g)
      if (g < G) o[g] *= alpha[g];
    for (int j = 0; j < nb; ++j) {
      const float v = to_f(vbase[static_cast<size_t>(kb + j) * kvw + t]);
#pragma unroll
      for (int g = 0; g < DEC_GMAX; ++g)
        if (g < G) o[g] = fmaf(sc[g][j], v, o[g]);
    }
    __syncthreads();
  }
  if (n_splits == 1) {
#pragma unroll
    for (int g = 0; g < DEC_GMAX; ++g)
      if (g < G) out[(static_cast<size_t>(seq) * H + kvh * G + g) * DH + t] = from_f<T>(o[g] / l_run[g]);
    return;
  }
#pragma unroll
  for (int g = 0; g < DEC_GMAX; ++g) {
    if (g < G) {
      const size_t slot = (static_cast<size_t>(seq) * H + kvh * G + g) * n_splits + split;
      part_o[slot * DH + t] = o[g];
      if (t == 0) part_ml[slot] = make_float2(m_run[g], l_run[g]);  // (-inf, 0) for an empty range
    }
  }
}

// Merges the key ranges of one (sequence, head): weights 2^(m_s - M) on each range's sums.
template <typename T, int DH>
__global__ void __launch_bounds__(DH) decode_merge_kernel(const float* __restrict__ part_o,
                                                          const float2* __restrict__ part_ml, int n_splits,
                                                          T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const size_t row = blockIdx.x;  // seq * H + head
  const float2* ml = part_ml + row * n_splits;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, ml[s].x);
  float L = 0.f, acc = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    if (ml[s].x == -INFINITY) continue;
    const float wgt = exp2f(ml[s].x - M);
    L = fmaf(ml[s].y, wgt, L);
    acc = fmaf(part_o[(row * n_splits + s) * DH + threadIdx.x], wgt, acc);
  }
  out[row * DH + threadIdx.x] = from_f<T>(acc / L);
}

template <typename T, int DH>
cudaError_t launch_dec(const void* q, const int32_t* pos, const ReqDev* reqs, int n_seq, int layer, int H, int Hkv,
                       int split_len, int n_splits, float* part_o, float2* part_ml, void* out, int32_t* status,
                       cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(DH));
  launch_chain(decode_attn_kernel<T, DH>, dim3(n_seq * Hkv, n_splits), dim3(DH), 0, s, static_cast<const T*>(q), pos,
               reqs, layer, H, Hkv, split_len, n_splits, scale_log2, part_o, part_ml, static_cast<T*>(out), status);
  if (n_splits > 1)
    launch_chain(decode_merge_kernel<T, DH>, dim3(n_seq * H), dim3(DH), 0, s, static_cast<const float*>(part_o),
                 static_cast<const float2*>(part_ml), n_splits, static_cast<T*>(out));
  return cudaGetLastError();
}

}  // namespace

void decode_split_plan(int n_seq, int n_kv_heads, int max_keys, int* split_len, int* n_splits) {
  // about two CTAs per SM over all (sequence, KV head) pairs, each range a whole number of
  // 64-key blocks, at most DECODE_MAX_SPLITS ranges
  const int want = (2 * 152 + n_seq * n_kv_heads - 1) / (n_seq * n_kv_heads);
  const int blocks = (max_keys + DEC_BK - 1) / DEC_BK;
  int splits = std::max(1, std::min({want, blocks, DECODE_MAX_SPLITS}));
  const int per = (blocks + splits - 1) / splits;
  *split_len = per * DEC_BK;
  *n_splits = (blocks + per - 1) / per;
}

cudaError_t launch_decode_attention(const void* q, const int32_t* pos, const ReqDev* reqs, int n_seq, int layer,
                                    int n_heads, int n_kv_heads, int head_dim, int split_len, int n_splits,
                                    float* part_o, float2* part_ml, void* out, cb_dtype dt, int32_t* status,
                                    cudaStream_t s) {
  if (n_seq <= 0) return cudaSuccess;
  if (n_heads / n_kv_heads > DEC_GMAX) return cudaErrorInvalidValue;
  if (dt == CB_BF16) {
    if (head_dim == 128)
      return launch_dec<bf16, 128>(q, pos, reqs, n_seq, layer, n_heads, n_kv_heads, split_len, n_splits, part_o,
                                   part_ml, out, status, s);
    if (head_dim == 64)
      return launch_dec<bf16, 64>(q, pos, reqs, n_seq, layer, n_heads, n_kv_heads, split_len, n_splits, part_o,
                                  part_ml, out, status, s);
  } else {
    if (head_dim == 128)
      return launch_dec<float, 128>(q, pos, reqs, n_seq, layer, n_heads, n_kv_heads, split_len, n_splits, part_o,
                                    part_ml, out, status, s);
    if (head_dim == 64)
      return launch_dec<float, 64>(q, pos, reqs, n_seq, layer, n_heads, n_kv_heads, split_len, n_splits, part_o,
                                   part_ml, out, status, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace cb
