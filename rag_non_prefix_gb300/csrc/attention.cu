// Causal attention of sparse (selected) queries over a fused KV cache.
//
// bf16, head_dim 128: flash-attention style.  A tile packs QT queries x G heads of one
// KV group into 64 rows (G = n_heads / n_kv_heads, QT = 64 / G), so the group's K/V
// blocks are read once for all its heads.  Four warps, 16 rows each; S = Q K^T and
// O += P V on mma.sync m16n8k16 (bf16 in, fp32 accumulate); 64-key K/V blocks are
// double-buffered in shared memory with cp.async (16-byte chunks, XOR-swizzled rows);
// online softmax in fp32 with exp2f.  The mask is per row: key j is visible to the row
// iff j <= the row's token position.  Tiles run longest-first (reverse launch order).
//
// fp32 (any head_dim multiple of 32 up to 128): one warp per (query, head); lanes split
// 32 keys at a time for the scores and head_dim for the output; expf softmax.
#include "common.cuh"
#include "internal.h"

namespace cb {

constexpr int AT_ROWS = 64;
constexpr int AT_KB = 64;
constexpr int AT_DH = 128;
constexpr int AT_THREADS = 128;
constexpr int AT_SMEM = (AT_ROWS * AT_DH + 4 * AT_KB * AT_DH) * 2;  // Q + 2 x (K, V)

struct AttnArgs {
  const bf16* q;
  const int32_t* s_pos;
  const int32_t* s_req;
  const ReqDev* reqs;
  const AttnTile* tiles;
  // direct mode (reqs == nullptr): one cache, tiles implied by m
  const bf16* k_direct;
  const bf16* v_direct;
  int n_kv_direct;
  int m_direct;
  int layer, H, Hkv, G, QT;
  bf16* out;
  float scale_log2;
};

// element offset of 16-byte chunk `ch` of row `r` in a [rows][128] bf16 tile, swizzled
__device__ __forceinline__ int swz(int r, int ch) { return r * AT_DH + ((ch ^ (r & 7)) << 3); }

__global__ void __launch_bounds__(AT_THREADS) attn_bf16_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t at_smem[];
  bf16* Qs = reinterpret_cast<bf16*>(at_smem);
  bf16* Ks = Qs + AT_ROWS * AT_DH;
  bf16* Vs = Ks + 2 * AT_KB * AT_DH;
  __shared__ int rowpos[AT_ROWS];
  __shared__ int s_maxpos;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y;
  AttnTile t;
  const bf16* Kc;
  const bf16* Vc;
  int n_kv;
  if (a.reqs) {
    t = a.tiles[gridDim.x - 1 - blockIdx.x];
    const ReqDev rq = a.reqs[t.req];
    const size_t off = static_cast<size_t>(a.layer) * rq.layer_stride;
    Kc = static_cast<const bf16*>(rq.k) + off;
    Vc = static_cast<const bf16*>(rq.v) + off;
    n_kv = rq.n_tokens;
  } else {
    const int b = gridDim.x - 1 - blockIdx.x;
    t.req = 0;
    t.row0 = b * a.QT;
    t.count = min(a.QT, a.m_direct - t.row0);
    Kc = a.k_direct;
    Vc = a.v_direct;
    n_kv = a.n_kv_direct;
  }
  const int G = a.G, QT = a.QT, H = a.H, Hkv = a.Hkv;

  if (tid < AT_ROWS) {
    const int qi = tid / G;
    int p = -1;
    if (qi < t.count && tid < QT * G) {
      p = a.s_pos[t.row0 + qi];
      if (p >= n_kv) p = n_kv - 1;  // positions are < n_kv by construction; clamp defensively
    }
    rowpos[tid] = p;
  }
  // Q tile: 64 rows x 16 chunks
  for (int c = tid; c < AT_ROWS * 16; c += AT_THREADS) {
    const int r = c >> 4, ch = c & 15;
    const int qi = r / G, g = r - qi * G;
    const bool valid = qi < t.count && r < QT * G;
    const bf16* src = valid ? a.q + (static_cast<size_t>(t.row0 + qi) * H + kvh * G + g) * AT_DH + ch * 8 : a.q;
    cp_async16(smem_u32(Qs + swz(r, ch)), src, valid ? 16 : 0);
  }
  cp_async_commit();
  __syncthreads();
  if (tid == 0) {
    int mp = -1;
    for (int r = 0; r < AT_ROWS; ++r) mp = max(mp, rowpos[r]);
    s_maxpos = mp;
  }
  __syncthreads();
  const int maxpos = s_maxpos;
  const int n_kb = maxpos < 0 ? 0 : maxpos / AT_KB + 1;

  auto load_kv = [&](int kb, int buf) {
    bf16* kd = Ks + buf * AT_KB * AT_DH;
    bf16* vd = Vs + buf * AT_KB * AT_DH;
    for (int c = tid; c < AT_KB * 16; c += AT_THREADS) {
      const int r = c >> 4, ch = c & 15;
      const int key = kb * AT_KB + r;
      const bool valid = key < n_kv;
      const size_t off = (static_cast<size_t>(valid ? key : 0) * Hkv + kvh) * AT_DH + ch * 8;
      cp_async16(smem_u32(kd + swz(r, ch)), Kc + off, valid ? 16 : 0);
      cp_async16(smem_u32(vd + swz(r, ch)), Vc + off, valid ? 16 : 0);
    }
  };
  if (n_kb > 0) load_kv(0, 0);
  cp_async_commit();
  cp_async_wait<1>();  // Q has landed
  __syncthreads();

  // Q fragments of this warp's 16 rows: 8 k-steps of 16 over head_dim
  uint32_t qf[8][4];
  {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int ch = ks * 2 + (lane >> 4);
      ldsm_x4(smem_u32(Qs + swz(r, ch)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  }
  const int r_lo = warp * 16 + (lane >> 2), r_hi = r_lo + 8;
  const int pos_lo = rowpos[r_lo], pos_hi = rowpos[r_hi];
  float m_lo = -1e30f, m_hi = -1e30f, l_lo = 0.f, l_hi = 0.f;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int kb = 0; kb < n_kb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < n_kb) load_kv(kb + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const bf16* kt = Ks + buf * AT_KB * AT_DH;
    const bf16* vt = Vs + buf * AT_KB * AT_DH;
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int nb2 = 0; nb2 < 4; ++nb2) {
        const int key = nb2 * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(kt + swz(key, ch)), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * nb2], qf[ks], b0, b1);
        mma_bf16_16816(s[2 * nb2 + 1], qf[ks], b2, b3);
      }
    }
    // mask, scale, online softmax
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kb * AT_KB + nb * 8 + 2 * (lane & 3) + (e & 1);
        const int pos = e < 2 ? pos_lo : pos_hi;
        float v = s[nb][e] * a.scale_log2;
        if (key > pos) v = -INFINITY;
        s[nb][e] = v;
        if (e < 2)
          mx_lo = fmaxf(mx_lo, v);
        else
          mx_hi = fmaxf(mx_hi, v);
      }
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float al_lo = exp2f(m_lo - mn_lo), al_hi = exp2f(m_hi - mn_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      s[nb][0] = exp2f(s[nb][0] - mn_lo);
      s[nb][1] = exp2f(s[nb][1] - mn_lo);
      s[nb][2] = exp2f(s[nb][2] - mn_hi);
      s[nb][3] = exp2f(s[nb][3] - mn_hi);
      ps_lo += s[nb][0] + s[nb][1];
      ps_hi += s[nb][2] + s[nb][3];
    }
    l_lo = l_lo * al_lo + ps_lo;
    l_hi = l_hi * al_hi + ps_hi;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= al_lo;
      o[i][1] *= al_lo;
      o[i][2] *= al_hi;
      o[i][3] *= al_hi;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dn2 = 0; dn2 < 8; ++dn2) {
        const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int ch = dn2 * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(vt + swz(key, ch)), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dn2], pa, b0, b1);
        mma_bf16_16816(o[2 * dn2 + 1], pa, b2, b3);
      }
    }
    __syncthreads();  // this buffer is refilled by the next iteration's prefetch
  }
  cp_async_wait<0>();

  // finalize: full row sums across the quad, normalise, store bf16
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
  const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? r_hi : r_lo;
    const int qi = r / G, g = r - qi * G;
    if (qi >= t.count || r >= QT * G) continue;
    const float inv = half ? inv_hi : inv_lo;
    bf16* dst = a.out + (static_cast<size_t>(t.row0 + qi) * H + kvh * G + g) * AT_DH;
#pragma unroll
    for (int nb = 0; nb < 16; ++nb) {
      const int col = nb * 8 + 2 * (lane & 3);
      *reinterpret_cast<__nv_bfloat162*>(dst + col) =
          __floats2bfloat162_rn(o[nb][2 * half] * inv, o[nb][2 * half + 1] * inv);
    }
  }
}

// ----------------------------------------------------------------------------- fp32
struct AttnArgsF32 {
  const float* q;
  const int32_t* s_pos;
  const int32_t* s_req;
  const ReqDev* reqs;
  const float* k_direct;
  const float* v_direct;
  int n_kv_direct;
  int n_rows;
  int layer, H, Hkv, dh;
  float* out;
  float scale;
};

__global__ void __launch_bounds__(256) attn_f32_kernel(AttnArgsF32 a) {
  __shared__ float qs[8][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (item >= static_cast<long long>(a.n_rows) * a.H) return;
  const int row = static_cast<int>(item / a.H), h = static_cast<int>(item % a.H);
  const int dh = a.dh, Hkv = a.Hkv;
  const int kvh = h / (a.H / Hkv);
  const float* Kc;
  const float* Vc;
  int n_kv;
  if (a.reqs) {
    const ReqDev rq = a.reqs[a.s_req[row]];
    const size_t off = static_cast<size_t>(a.layer) * rq.layer_stride;
    Kc = static_cast<const float*>(rq.k) + off;
    Vc = static_cast<const float*>(rq.v) + off;
    n_kv = rq.n_tokens;
  } else {
    Kc = a.k_direct;
    Vc = a.v_direct;
    n_kv = a.n_kv_direct;
  }
  int pos = a.s_pos[row];
  if (pos >= n_kv) pos = n_kv - 1;
  const float* q = a.q + (static_cast<size_t>(row) * a.H + h) * dh;
  for (int e = lane; e < dh; e += 32) qs[warp][e] = q[e];
  __syncwarp();
  const int per = dh / 32;  // output elements per lane (dh <= 128)
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  float m = -INFINITY, l = 0.f;
  for (int k0 = 0; k0 <= pos; k0 += 32) {
    const int key = k0 + lane;
    float sc = -INFINITY;
    if (key <= pos) {
      const float* kr = Kc + (static_cast<size_t>(key) * Hkv + kvh) * dh;
      float acc = 0.f;
      for (int e = 0; e < dh; ++e) acc = fmaf(qs[warp][e], kr[e], acc);
      sc = acc * a.scale;
    }
    float mx = sc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float mn = fmaxf(m, mx);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - mn);
    const float p = (key <= pos) ? expf(sc - mn) : 0.f;
    float ps = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
    m = mn;
    for (int i = 0; i < per; ++i) o[i] *= alpha;
    const int nk = min(32, pos - k0 + 1);
    for (int j = 0; j < nk; ++j) {
      const float w = __shfl_sync(0xffffffffu, p, j);
      const float* vr = Vc + (static_cast<size_t>(k0 + j) * Hkv + kvh) * dh;
      for (int i = 0; i < per; ++i) o[i] = fmaf(w, vr[lane + 32 * i], o[i]);
    }
  }
  float* dst = a.out + (static_cast<size_t>(row) * a.H + h) * dh;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  for (int i = 0; i < per; ++i) dst[lane + 32 * i] = o[i] * inv;
}

// ----------------------------------------------------------------------------- launchers
int attention_tile_rows(int n_heads, int n_kv_heads, cb_dtype dt) {
  if (dt == CB_F32) return 1;
  const int G = n_heads / n_kv_heads;
  return G >= AT_ROWS ? 1 : AT_ROWS / G;
}

static cudaError_t attn_bf16_launch(const AttnArgs& args, int n_tiles, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(n_tiles, args.Hkv);
  attn_bf16_kernel<<<grid, AT_THREADS, AT_SMEM, s>>>(args);
  return cudaGetLastError();
}

// Batched: tiles (bf16) or all rows (fp32, n_tiles = number of S rows) of one layer.
cudaError_t launch_attention(const void* q, const int32_t* s_pos, const int32_t* s_req, const ReqDev* reqs,
                             const AttnTile* tiles, int n_tiles, int layer, int n_heads, int n_kv_heads, int head_dim,
                             void* out, cb_dtype dt, cudaStream_t s) {
  if (n_tiles <= 0) return cudaSuccess;
  if (dt == CB_BF16) {
    AttnArgs a{};
    a.q = static_cast<const bf16*>(q);
    a.s_pos = s_pos;
    a.s_req = s_req;
    a.reqs = reqs;
    a.tiles = tiles;
    a.layer = layer;
    a.H = n_heads;
    a.Hkv = n_kv_heads;
    a.G = n_heads / n_kv_heads;
    a.QT = attention_tile_rows(n_heads, n_kv_heads, dt);
    a.out = static_cast<bf16*>(out);
    a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(head_dim));
    return attn_bf16_launch(a, n_tiles, s);
  }
  AttnArgsF32 a{};
  a.q = static_cast<const float*>(q);
  a.s_pos = s_pos;
  a.s_req = s_req;
  a.reqs = reqs;
  a.n_rows = n_tiles;
  a.layer = layer;
  a.H = n_heads;
  a.Hkv = n_kv_heads;
  a.dh = head_dim;
  a.out = static_cast<float*>(out);
  a.scale = 1.0f / sqrtf(static_cast<float>(head_dim));
  const long long items = static_cast<long long>(n_tiles) * n_heads;
  attn_f32_kernel<<<static_cast<unsigned>((items + 7) / 8), 256, 0, s>>>(a);
  return cudaGetLastError();
}

// Standalone (one cache, no workspace): used by cb_attention.
cudaError_t launch_attention_direct(const void* q, const int32_t* q_pos, int m, const void* k, const void* v,
                                   int n_kv, int n_heads, int n_kv_heads, int head_dim, void* out, cb_dtype dt,
                                   cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  if (dt == CB_BF16) {
    AttnArgs a{};
    a.q = static_cast<const bf16*>(q);
    a.s_pos = q_pos;
    a.k_direct = static_cast<const bf16*>(k);
    a.v_direct = static_cast<const bf16*>(v);
    a.n_kv_direct = n_kv;
    a.m_direct = m;
    a.H = n_heads;
    a.Hkv = n_kv_heads;
    a.G = n_heads / n_kv_heads;
    a.QT = attention_tile_rows(n_heads, n_kv_heads, dt);
    a.out = static_cast<bf16*>(out);
    a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(head_dim));
    return attn_bf16_launch(a, (m + a.QT - 1) / a.QT, s);
  }
  AttnArgsF32 a{};
  a.q = static_cast<const float*>(q);
  a.s_pos = q_pos;
  a.k_direct = static_cast<const float*>(k);
  a.v_direct = static_cast<const float*>(v);
  a.n_kv_direct = n_kv;
  a.n_rows = m;
  a.H = n_heads;
  a.Hkv = n_kv_heads;
  a.dh = head_dim;
  a.out = static_cast<float*>(out);
  a.scale = 1.0f / sqrtf(static_cast<float>(head_dim));
  const long long items = static_cast<long long>(m) * n_heads;
  attn_f32_kernel<<<static_cast<unsigned>((items + 7) / 8), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace cb
