// Causal attention of sparse (selected) queries over a fused KV cache.
//
// bf16, head_dim 128, on the tcgen05 tensor cores.  One CTA per (tile, KV head): a tile
// packs QT queries x G heads of one KV group into the 128 rows of the MMA (G = n_heads /
// n_kv_heads, QT = 128 / G), so each K/V block is read once for all heads of the group.
//   warp 0: TMA producers (lane 0: K, lane 1: V) -- 4-D tensor maps over the fused cache
//           [L][N][Hkv][dh] bring 128-key K and V blocks (128-byte swizzle) into two-slot rings
//   warp 1: TMEM owner + MMA issuer -- S_j = Q K_j^T into one of two TMEM buffers, then
//           O += P_{j-1} V_{j-1} (V as an MN-major operand) accumulated in TMEM
//   warps 2-5: one query row per thread -- read S_j from TMEM, apply the causal mask (key
//           j is visible iff j <= the row's token position) and the online softmax in fp32
//           (ex2.approx), and write P_j (bf16) to one of two shared-memory buffers.  P is taken
//           relative to a reference max that moves only when a row's max grows by more
//           than 2^8; then the row of O in TMEM is rescaled (rarely).  Finally O / l -> bf16.
// The grid is one-dimensional, KV head fastest and the longest tiles first.  When a layer's
// (tile, head) units leave SMs idle, its longest tiles get a second CTA: a tile of at least
// ATTN_SPLIT_MIN_BLOCKS key blocks then splits its key range in two, each CTA writes its
// unnormalised O and per-row (max, sum) to a partial slot, and the CTA that finishes second
// (an atomic ticket) combines the two halves in a fixed order and writes the rows.
// Every mbarrier wait is bounded: on timeout the CTA records ST_WAIT_TIMEOUT and leaves.
//
// fp32 (any head_dim multiple of 32 up to 128): one warp per (query, head); lanes split
// 32 keys at a time for the scores and head_dim for the output; expf softmax.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace cb {

namespace ta {

constexpr int ROWS = 128;    // MMA M: (query, head) rows of a tile
constexpr int BKV = 128;     // keys per block (MMA N of S, K of PV)
constexpr int DH = 128;
constexpr int THREADS = 320;   // producer, MMA, two softmax warpgroups
constexpr int MAXREQ = 16;   // requests (tensor-map pairs) per launch
constexpr int ATOM = ROWS * 64 * 2;          // one [128][64] bf16 swizzle-atom column: 16 KiB
constexpr int OFF_Q = 0;                     // Q: 2 atom columns (head_dim 0-63, 64-127)
constexpr int OFF_P = OFF_Q + 2 * ATOM;      // P[2]: 2 atom columns each (keys 0-63, 64-127)
constexpr int OFF_KV = OFF_P + 4 * ATOM;     // stages of K (2 columns) then V (2 columns)
constexpr int STAGE = 4 * ATOM;              // 64 KiB
constexpr int STAGES = 2;
constexpr int OFF_BAR = OFF_KV + STAGES * STAGE;
constexpr int SMEM = OFF_BAR + 3072;         // barriers, row positions, max exchange: the 227 KiB limit
// The operand tiles fill shared memory, leaving no slack to realign the base: the kernel
// relies on the dynamic shared memory starting 1024-byte aligned (it checks, and reports
// ST_RANGE instead of computing when it is not).
constexpr uint32_t TMEM_COLS = 512;          // S[2] at columns 0 and 128, O at 256
constexpr uint32_t O_COL = 256;
constexpr float RESCALE_LOG2 = 8.0f;         // O is rescaled only when a row max grows by > 2^8

// 2^x with the PTX ex2.approx.ftz.f32 instruction (relative error ~2^-22; results below
// 2^-126 flush to 0, which for a softmax numerator next to a row sum >= 1 is below the
// bf16 rounding of P).  The library exp2f adds range fix-ups around the same instruction
// that this kernel does not need, and they made the softmax twice as slow.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100 family): one instruction for two lanes of fp32 arithmetic, each
// rounded as its scalar counterpart.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

struct Args {
  CUtensorMap kmap[MAXREQ];
  CUtensorMap vmap[MAXREQ];
  int n_kv[MAXREQ];
  int layer_coord[MAXREQ];  // 4th coordinate of the maps (0 for a one-layer cache)
  const bf16* q;
  const int32_t* s_pos;
  const AttnTile* tiles;    // null: direct mode (one request, tiles of QT rows over m queries)
  int req_base;
  int n_tiles;
  int direct_m;
  int H, Hkv, G, QT;
  bf16* out;
  float scale_log2;
  int32_t* status;
  // key-range splits: the n_paired longest tiles get two CTAs (unit = tile * Hkv + head, tile in
  // longest-first order), the others one (n_paired 0 or part_o null: one CTA per tile)
  float* part_o;       // [unit][2 ranges] x float4 [2 halves][16][128 rows]: unnormalised O
  float2* part_ml;     // [unit][2][128] (reference max, row sum)
  int* part_cnt;       // [unit] CTAs of the unit done (reset to 0 by the second)
  int n_paired;
  // two query tiles per CTA (attn_tc2_kernel): request r's tiles are tiles[tile_off[r] ..
  // tile_off[r + 1]) of this launch and its tile pairs pair_off[r] .. pair_off[r + 1]
  int tile_off[MAXREQ + 1];
  int pair_off[MAXREQ + 1];
  int n_pairs;
};

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {  // K-major, 128-byte swizzle
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}
// MN-major, 128-byte swizzle: 64-element column blocks lbo bytes apart, 8-row groups 1 KiB apart
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr, uint32_t lbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// kind::f16, bf16 inputs, fp32 accumulator, M = 128, N = 128; B MN-major when b_mn
__host__ __device__ constexpr uint32_t idesc(bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
}

// Key-range split epilogue of attn_tc_kernel, run by its 256 softmax threads (named
// barrier 5; thread 64 is the first of them): this range's unnormalised O (ov, one row half at
// the reference max m) and (m, row sum of both halves) go to its partial slot; the unit's CTA that
// finishes second combines range 0 and range 1 in that order (whichever finished first),
// normalises and stores.  Partials are float4 [slot][half][16][128 rows]: one warp instruction
// stores or loads 512 contiguous bytes.  The release of the partials is the CTA barrier followed
// by one thread's device-scope fence before its ticket; the merging CTA fences after its ticket.
__device__ __forceinline__ void split_epilogue(const Args& a, int unit, int part, int half, int r, bool valid,
                                               const uint32_t* ov, float m, float l_all, bf16* dst,
                                               volatile int* merge_flag) {
  const size_t mine = static_cast<size_t>(unit) * 2 + part, other = static_cast<size_t>(unit) * 2 + (part ^ 1);
  float4* po = reinterpret_cast<float4*>(a.part_o) + (mine * 2 + half) * 16 * ROWS + r;
#pragma unroll
  for (int c = 0; c < 16; ++c)
    po[c * ROWS] = make_float4(__uint_as_float(ov[4 * c]), __uint_as_float(ov[4 * c + 1]),
                               __uint_as_float(ov[4 * c + 2]), __uint_as_float(ov[4 * c + 3]));
  if (half == 0) a.part_ml[mine * ROWS + r] = make_float2(m, l_all);
  asm volatile("bar.sync 5, 256;" ::: "memory");
  if (threadIdx.x == 64) {
    __threadfence();
    *merge_flag = atomicAdd(&a.part_cnt[unit], 1) == 1;
    __threadfence();
  }
  asm volatile("bar.sync 5, 256;" ::: "memory");
  if (!*merge_flag) return;
  const float2 oml = __ldcg(&a.part_ml[other * ROWS + r]);
  const float m0 = part == 0 ? m : oml.x, m1 = part == 0 ? oml.x : m;
  const float l0 = part == 0 ? l_all : oml.y, l1 = part == 0 ? oml.y : l_all;
  const float mm = fmaxf(m0, m1);
  const float w0 = ex2(m0 - mm), w1 = ex2(m1 - mm);
  const float ls = __fmaf_rn(l1, w1, __fmul_rn(l0, w0));
  const float inv = ls > 0.f ? 1.f / ls : 0.f;
  const float4* qo = reinterpret_cast<const float4*>(a.part_o) + (other * 2 + half) * 16 * ROWS + r;
  if (valid) {
#pragma unroll
    for (int c0 = 0; c0 < 16; c0 += 8) {  // eight loads in flight before their sums
      float4 x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = __ldcg(qo + (c0 + u) * ROWS);
#pragma unroll
      for (int u = 0; u < 8; u += 2) {
        const float xo[8] = {x[u].x, x[u].y, x[u].z, x[u].w, x[u + 1].x, x[u + 1].y, x[u + 1].z, x[u + 1].w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float mine_v = __uint_as_float(ov[(c0 + u) * 4 + e]);
          const float o0 = part == 0 ? mine_v : xo[e];
          const float o1 = part == 0 ? xo[e] : mine_v;
          f[e] = __fmul_rn(__fmaf_rn(o1, w1, __fmul_rn(o0, w0)), inv);
        }
        store8(dst + (c0 + u) * 4, f);
      }
    }
  }
  if (threadIdx.x == 64) a.part_cnt[unit] = 0;  // for the next launch
}

// Barriers (phase of use u of a two-slot barrier b[x & 1] is (x >> 1) & 1):
//   q_full            softmax warps stored Q                       (4 arrivals)
//   k_full[2]         K_j landed                                   (TMA bytes)
//   k_empty[2]        S_j done: K slot free                        (MMA commit)
//   v_full[2]         V_j landed                                   (TMA bytes)
//   v_empty[2]        PV_j done: V slot free                       (MMA commit)
//   s_full[2]         S_j in TMEM                                  (MMA commit)
//   s_empty[2]        S_j read into registers                      (4 arrivals)
//   p_full[2]         P_j in shared memory (and O rescaled)        (4 arrivals)
//   pv_done[2]        PV_j accumulated into O                      (MMA commit)
__global__ void __launch_bounds__(THREADS, 1) attn_tc_kernel(const __grid_constant__ Args a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  pdl_trigger();
  pdl_wait();
  if (smem_u32(smem_raw) & 1023u) {  // uniform across the block
    if (threadIdx.x == 0) set_status(a.status, ST_RANGE);
    return;
  }
  uint8_t* smem = smem_raw;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bar;
  uint64_t* k_full = bar + 1;
  uint64_t* k_empty = bar + 3;
  uint64_t* s_full = bar + 5;
  uint64_t* s_empty = bar + 7;
  uint64_t* p_full = bar + 9;
  uint64_t* pv_done = bar + 11;
  uint64_t* drain = bar + 13;
  uint64_t* v_full = bar + 14;
  uint64_t* v_empty = bar + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* rowpos = reinterpret_cast<int*>(bar + 20);  // [128] (bar + 18: slot, abort flag)
  float* xmax = reinterpret_cast<float*>(rowpos + ROWS);  // [2][2][128]: per block parity, per half

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // One-dimensional grid, KV head fastest, then the two key ranges of a paired tile, then the
  // tiles, longest first: CTAs start in that order, so the longest work of every head goes
  // first and the shorter tiles fill the SMs that free up.
  const int n_paired = a.part_o != nullptr ? a.n_paired : 0;
  const int kvh = static_cast<int>(blockIdx.x % a.Hkv);
  const int rest = static_cast<int>(blockIdx.x / a.Hkv);
  const bool paired = rest < 2 * n_paired;
  const int tix = paired ? (rest >> 1) : rest - n_paired;
  const int part = paired ? (rest & 1) : 0;
  AttnTile t;
  if (a.tiles) {
    t = a.tiles[a.n_tiles - 1 - tix];  // longest tiles first
    t.req -= a.req_base;
  } else {
    const int b = a.n_tiles - 1 - tix;
    t.req = 0;
    t.row0 = b * a.QT;
    t.count = min(a.QT, a.direct_m - t.row0);
  }
  const int G = a.G, QT = a.QT, H = a.H;
  const int n_kv = a.n_kv[t.req];

  if (threadIdx.x == 0) {
    mbar_init(q_full, 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 8);
      mbar_init(&p_full[i], 8);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  int* wmaxpos = reinterpret_cast<int*>(smem + OFF_BAR + 2720);  // [4] per-warp maxima of rowpos
  if (threadIdx.x >= 64 && threadIdx.x < 64 + ROWS) {  // row positions (-1: no query in this row)
    const int r = threadIdx.x - 64;
    const int qi = r / G;
    int p = -1;
    if (qi < t.count && r < QT * G) p = min(a.s_pos[t.row0 + qi], n_kv - 1);
    rowpos[r] = p;
    const int wm = __reduce_max_sync(0xffffffffu, p);
    if ((r & 31) == 0) wmaxpos[r >> 5] = wm;
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int maxpos = max(max(wmaxpos[0], wmaxpos[1]), max(wmaxpos[2], wmaxpos[3]));
  const int n_blk = maxpos < 0 ? 0 : maxpos / BKV + 1;
  // Key blocks [b0, b1) of this CTA: a long paired tile's two CTAs take one half each; the
  // second CTA of a short one has nothing to do.
  const bool split = paired && n_blk >= ATTN_SPLIT_MIN_BLOCKS;
  if (paired && !split && part == 1) {  // uniform across the block
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, TMEM_COLS);
    }
    return;
  }
  const int b_half = (n_blk + 1) / 2;
  const int b0 = (split && part == 1) ? b_half : 0;
  const int nb = split ? (part == 0 ? b_half : n_blk - b_half) : n_blk;  // blocks of this CTA
  const int unit = tix * a.Hkv + kvh;  // (paired tiles only: tix < n_paired)

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // Lane 0 streams K, lane 1 streams V, each at the pace its own slots free up (K_j
    // once S_{j-2} is done with its slot, V_j once PV_{j-2} is), so that a K load never
    // queues behind a V slot that the previous PV still holds.
    if (lane < 2) {
      const bool is_v = lane == 1;
      const CUtensorMap* map = is_v ? &a.vmap[t.req] : &a.kmap[t.req];
      uint64_t* empty = is_v ? v_empty : k_empty;
      uint64_t* full = is_v ? v_full : k_full;
      const int lc = a.layer_coord[t.req];
      int issued = 0;
      for (int j = 0; j < nb; ++j) {  // local block j = key block b0 + j
        const int st = j & 1;
        const uint32_t ph = ((j >> 1) & 1) ^ 1;
        uint8_t* dst = smem + OFF_KV + st * STAGE + (is_v ? 2 * ATOM : 0);
        if (!mbar_wait_bounded(&empty[st], ph, abort_flag)) break;
        mbar_arrive_expect_tx(&full[st], 2 * ATOM);
        tma_load_4d(dst, map, &full[st], 0, kvh, (b0 + j) * BKV, lc);
        tma_load_4d(dst + ATOM, map, &full[st], 64, kvh, (b0 + j) * BKV, lc);
        issued = j + 1;
      }
      if (issued < nb && !*abort_flag) {
        *abort_flag = 1;
        set_status(a.status, ST_WAIT_TIMEOUT);
      }
      // copies issued into slots that nobody consumed must land before the block exits
      for (int j = max(0, issued - 2); j < issued; ++j) mbar_wait_bounded(&full[j & 1], (j >> 1) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    const uint32_t sq = smem_u32(smem + OFF_Q);
    bool ok = true;
    auto wait = [&](uint64_t* b, uint32_t ph) {
      if (ok && lane == 0) ok = mbar_wait_bounded(b, ph, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      return ok;
    };
    auto issue_pv = [&](int i) {  // O (+)= P_i V_i
      const int st = i & 1;
      if (!wait(&p_full[st], (i >> 1) & 1) || !wait(&v_full[st], (i >> 1) & 1)) return;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sp = smem_u32(smem + OFF_P + st * 2 * ATOM);
        const uint32_t sv = smem_u32(smem + OFF_KV + st * STAGE + 2 * ATOM);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {  // 16 keys per step: P columns, V rows
          const uint64_t da = desc_kmajor(sp + (kk >> 2) * ATOM) + 2 * (kk & 3);
          const uint64_t db = desc_mnmajor(sv + kk * 16 * 128, ATOM);
          tc_mma_f16(tmem + O_COL, da, db, idesc(true), (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[st]);
        tc_commit(&v_empty[st]);
      }
      __syncwarp();
    };
    wait(q_full, 0);
    for (int j = 0; ok && j < nb; ++j) {
      const int st = j & 1;
      if (!wait(&k_full[st], (j >> 1) & 1) || !wait(&s_empty[st], ((j >> 1) & 1) ^ 1)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sk = smem_u32(smem + OFF_KV + st * STAGE);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {  // 16 head-dim elements per step
          const uint64_t da = desc_kmajor(sq + (kk >> 2) * ATOM) + 2 * (kk & 3);
          const uint64_t db = desc_kmajor(sk + (kk >> 2) * ATOM) + 2 * (kk & 3);
          tc_mma_f16(tmem + st * 128, da, db, idesc(false), kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[st]);
        tc_commit(&k_empty[st]);
      }
      __syncwarp();
      if (j >= 1) issue_pv(j - 1);
    }
    if (ok && nb > 0) issue_pv(nb - 1);
    if (!ok && lane == 0) {
      *abort_flag = 1;
      set_status(a.status, ST_WAIT_TIMEOUT);
    }
    if (lane == 0) {  // no MMA may run when the tensor memory is released
      tc_commit(drain);
      mbar_wait_bounded(drain, 0u, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax / output (warps 2..9)
    // Two warpgroups: half h handles columns 64h..64h+63 of every row of S, P and O.
    const int sw = warp - 2;           // 0..7
    const int half = sw >> 2;
    const int quarter = warp & 3;      // TMEM lanes 32*quarter .. +31 belong to this warp
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(half * 64);
    const int qi = r / G, g = r - qi * G;
    const bool valid = qi < t.count && r < QT * G;
    // Q: half h stores head_dim atom h of its rows
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + (static_cast<size_t>(t.row0 + (valid ? qi : 0)) * H + kvh * G + g) * DH + half * 64);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = valid ? src[c] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + OFF_Q + half * ATOM + r * 128 + ((c ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    const int pos = rowpos[r];
    float m = -1e30f, l = 0.f;  // reference max of P (log2 units, scaled); this half's row sum
    // A failed (bounded) wait clears ok and skips the work that depends on it, but never the
    // named barriers: both halves run the same barriers in the same order, and every later
    // wait returns at once (ok stays false), so the loop still ends.
    bool ok = true;
    auto wait = [&](uint64_t* b, uint32_t ph) {
      if (ok && lane == 0) ok = mbar_wait_bounded(b, ph, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
    };
    // The two warps that hold the same 32 rows (one per column half) exchange row maxima and
    // sums through shared memory: a named barrier per such pair (ids 1-4, 64 threads), so a
    // warp never waits for the other six.
    const uint32_t pair_bar = 1u + static_cast<uint32_t>(quarter);
    auto sm_bar = [pair_bar]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    for (int j = 0; j < nb; ++j) {  // local block j = key block b0 + j
      const int st = j & 1;
      wait(&s_full[st], (j >> 1) & 1);
      uint32_t sv[64];
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 64; c += 16) tmem_ld16_nowait(tmem + st * 128 + col0 + lane_off + c, sv + c);
        tmem_wait_ld();
        tc_fence_before();
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[e] = 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[st]);
      const int k0 = (b0 + j) * BKV + half * 64;
      // the unmasked path only when every row of the warp sees the whole block (a warp-uniform
      // branch: rows of sparse tiles sit at scattered positions)
      const bool full = __all_sync(0xffffffffu, k0 + 63 <= pos);
      // row max of this half: eight independent chains, then a tree
      float pm[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
      if (full) {  // three-input max: 32 instructions for the 64 columns
#pragma unroll
        for (int e = 0; e < 64; e += 16)
#pragma unroll
          for (int u = 0; u < 8; ++u) pm[u] = max3(pm[u], __uint_as_float(sv[e + u]), __uint_as_float(sv[e + 8 + u]));
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (k0 + e <= pos) pm[e & 7] = fmaxf(pm[e & 7], __uint_as_float(sv[e]));
      }
      float mx = max3(max3(pm[0], pm[1], pm[2]), max3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
      mx *= a.scale_log2;  // scale > 0: the max commutes with it
      // row max over both halves (slots by block parity: a slot is rewritten two blocks later,
      // after the barrier of the next block, so the partner has read it)
      xmax[(st * 2 + half) * ROWS + r] = mx;
      sm_bar();
      mx = fmaxf(mx, xmax[(st * 2 + (half ^ 1)) * ROWS + r]);
      // lazy rescale: move the reference max only when this block exceeds it by > 2^8
      const bool need = mx > m + RESCALE_LOG2;
      const float m_new = need ? mx : m;
      const float alpha = ex2(m - m_new);
      // O needs the rescale only in rows that already hold mass: a row that saw no key yet
      // (the second key range of a split tile starts past some rows' positions) has O = 0
      if (__any_sync(0xffffffffu, need && m > -1e29f) && j > 0) {  // same rows, same decision in both halves
        // O holds PV_0..PV_{j-1}: wait for the last of them, then scale this warp's part
        wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            uint32_t ov[16];
            tmem_ld16_nowait(tmem + O_COL + col0 + lane_off + c, ov);
            tmem_wait_ld();
            float f[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(ov[e]) * alpha;
            tmem_st16(tmem + O_COL + col0 + lane_off + c, f);
          }
          tmem_wait_st();
        }
      }
      l *= alpha;
      m = m_new;
      // P_j (this half's 64 keys = one swizzle atom) -> its buffer, free once PV_{j-2} is done
      if (j >= 2) wait(&pv_done[st], ((j - 2) >> 1) & 1);
      if (ok) {
        uint8_t* pb = smem + OFF_P + st * 2 * ATOM + half * ATOM;
        if (full) {
          // every key visible: (s * scale - m) for two columns per packed FMA, the row sum in
          // two packed accumulators
          const uint64_t sc2 = f2(a.scale_log2, a.scale_log2), nm2 = f2(-m, -m);
          uint64_t acc0 = f2(0.f, 0.f), acc1 = acc0;
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              float t0, t1;
              f2_split(fma2(f2(__uint_as_float(sv[c + e]), __uint_as_float(sv[c + e + 1])), sc2, nm2), t0, t1);
              const float p0 = ex2(t0), p1 = ex2(t1);
              if (e & 2)
                acc1 = add2(acc1, f2(p0, p1));
              else
                acc0 = add2(acc0, f2(p0, p1));
              pk[e >> 1] = pack_bf16x2(p0, p1);
            }
            *reinterpret_cast<uint4*>(pb + r * 128 + (((c >> 3) ^ (r & 7)) << 4)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          float a0, a1, b0, b1;
          f2_split(acc0, a0, a1);
          f2_split(acc1, b0, b1);
          l += (a0 + a1) + (b0 + b1);
        } else {
          float ls[4] = {0.f, 0.f, 0.f, 0.f};  // four independent partial row sums
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const int x = c + e;
              const float p0 = k0 + x <= pos ? ex2(fmaf(__uint_as_float(sv[x]), a.scale_log2, -m)) : 0.f;
              const float p1 = k0 + x + 1 <= pos ? ex2(fmaf(__uint_as_float(sv[x + 1]), a.scale_log2, -m)) : 0.f;
              ls[e >> 1] += p0 + p1;
              pk[e >> 1] = pack_bf16x2(p0, p1);
            }
            *reinterpret_cast<uint4*>(pb + r * 128 + (((c >> 3) ^ (r & 7)) << 4)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[st]);
    }
    // O = PV_0 + ... + PV_{n-1} (at the reference max) / (row sum of both halves); the sums go
    // to the exchange slots of parity nb, last read before the previous block's barrier
    float* xsum = xmax + (nb & 1) * 2 * ROWS;
    xsum[half * ROWS + r] = l;
    if (nb > 0) wait(&pv_done[(nb - 1) & 1], ((nb - 1) >> 1) & 1);
    sm_bar();
    const float l_all = xsum[r] + xsum[ROWS + r];  // same order in both halves
    bf16* dst = a.out + (static_cast<size_t>(t.row0 + (valid ? qi : 0)) * H + kvh * G + g) * DH + half * 64;
    if (split) {
      // This CTA's key range: O unnormalised (at the reference max m) and (m, row sum) of every
      // row go to its partial slot; the CTA of the tile that finishes second adds the two
      // ranges (each scaled to the larger max), normalises and stores.
      uint32_t ov[64];
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 64; c += 16) tmem_ld16_nowait(tmem + O_COL + col0 + lane_off + c, ov + c);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) ov[e] = 0u;
      }
      split_epilogue(a, unit, part, half, r, valid, ov, m, l_all, dst, reinterpret_cast<volatile int*>(wmaxpos + 4));
    } else if (ok && nb > 0) {
      tc_fence_after();
      const float inv = l_all > 0.f ? 1.f / l_all : 0.f;
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        uint32_t ov[16];
        tmem_ld16_nowait(tmem + O_COL + col0 + lane_off + c, ov);
        tmem_wait_ld();
        if (valid) {
          float f[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(ov[e]) * inv;
          store8(dst + c, f);
          store8(dst + c + 8, f + 8);
        }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      set_status(a.status, ST_WAIT_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace ta

// ----------------------------------------------------------------------------- two tiles per CTA
// attn_tc2_kernel: the same attention with two query tiles of one KV head per CTA, so that
// the tensor core works for one tile while the other tile's softmax runs, and every K/V
// block is loaded once for both.  Per tile, S is single-buffered in tensor memory: the
// softmax reads S_j into registers and releases it at once, so S_{j+1} is computed while
// the softmax of block j still runs; P is single-buffered in shared memory and written
// (and O rescaled) only after PV_{j-1} is done, the P values waiting in registers.  K and V
// blocks share a three-slot ring loaded in the order K0, K1, V0, K2, V1, ..., K_{n-1},
// V_{n-2}, V_{n-1}, the order the MMA issuer consumes them (S_{j+1} before PV_j): each K
// block arrives two iterations ahead of its use, each V block one.
//   warp 0: TMA producer (lane 0)            warp 1: TMEM owner + MMA issuer (lane 0)
//   warps 2-9: softmax of tile 0             warps 10-17: softmax of tile 1
// (in each group, as in attn_tc_kernel: two column halves x four lane quarters).
// Tiles are paired within a request (tiles 2i and 2i + 1); pairs run longest first.  No
// key-range split here: the launcher takes this kernel when the pairs fill the SMs.
namespace tp {

using namespace ta;
constexpr int THREADS2 = 18 * 32;
constexpr int OFF_Q2 = 0;                       // Q[2 tiles]: 2 atom columns each
constexpr int OFF_P2 = OFF_Q2 + 4 * ATOM;       // P[2 tiles]: 2 atom columns each
constexpr int OFF_RING = OFF_P2 + 4 * ATOM;     // 3 slots of one K or V block (2 atom columns)
constexpr int SLOTS = 3;
constexpr int SLOT = 2 * ATOM;
constexpr int OFF_BAR2 = OFF_RING + SLOTS * SLOT;
constexpr int SMEM2 = OFF_BAR2 + 3072;          // the 227 KiB limit, as attn_tc_kernel
constexpr uint32_t S_COL = 0;                   // S of tile t at column 128 t
constexpr uint32_t O_COL2 = 256;                // O of tile t at column 256 + 128 t

// Non-blocking test of an mbarrier phase (the MMA issuer polls several barriers in turn).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Position of K_j / V_j in the load order K0, K1, V0, K2, V1, ..., K_{n-1}, V_{n-2}, V_{n-1}
__device__ __forceinline__ int k_item(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_item(int j, int nb) { return min(2 * j + 2, 2 * nb - 1); }

struct PairTiles {
  AttnTile t[2];
  int n;  // tiles in the pair: 1 or 2
};

__device__ __forceinline__ PairTiles pair_of(const Args& a, int p) {
  PairTiles pt;
  if (a.tiles) {
    int r = 0;
    while (r + 1 < MAXREQ && p >= a.pair_off[r + 1]) ++r;
    const int i0 = a.tile_off[r] + 2 * (p - a.pair_off[r]);
    pt.n = i0 + 1 < a.tile_off[r + 1] ? 2 : 1;
    for (int u = 0; u < 2; ++u) {
      if (u < pt.n) {
        pt.t[u] = a.tiles[i0 + u];
        pt.t[u].req -= a.req_base;
      } else {
        pt.t[u] = AttnTile{pt.t[0].req, 0, 0, 0};
      }
    }
  } else {
    for (int u = 0; u < 2; ++u) {
      const int row0 = (2 * p + u) * a.QT;
      pt.t[u] = AttnTile{0, row0, max(0, min(a.QT, a.direct_m - row0)), 0};
    }
    pt.n = pt.t[1].count > 0 ? 2 : 1;
  }
  return pt;
}

// Barriers (per tile t, phase of block j is j & 1):
//   q_full[t]   softmax warps of tile t stored Q_t      (8 arrivals)
//   s_full[t]   S_t(j) in TMEM                          (MMA commit)
//   s_empty[t]  S_t(j) read into registers              (8 arrivals)
//   p_full[t]   P_t(j) in shared memory, O_t rescaled   (8 arrivals)
//   pv_done[t]  PV_t(j) accumulated into O_t            (MMA commit)
//   full[3]     ring slot loaded (TMA bytes); empty[3] ring slot consumed (MMA commit)
__global__ void __launch_bounds__(THREADS2, 1) attn_tc2_kernel(const __grid_constant__ Args a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  pdl_trigger();
  pdl_wait();
  if (smem_u32(smem_raw) & 1023u) {  // uniform across the block
    if (threadIdx.x == 0) set_status(a.status, ST_RANGE);
    return;
  }
  uint8_t* smem = smem_raw;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR2);
  uint64_t* q_full = bar;        // [2]
  uint64_t* s_full = bar + 2;    // [2]
  uint64_t* s_empty = bar + 4;   // [2]
  uint64_t* p_full = bar + 6;    // [2]
  uint64_t* pv_done = bar + 8;   // [2]
  uint64_t* full = bar + 10;     // [3]
  uint64_t* empty = bar + 13;    // [3]
  uint64_t* drain = bar + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR2 + 144);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR2 + 148);
  int* wmaxpos = reinterpret_cast<int*>(smem + OFF_BAR2 + 152);     // [2 tiles][4 quarters]
  float* xch = reinterpret_cast<float*>(smem + OFF_BAR2 + 256);     // [2 tiles][2 halves][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = static_cast<int>(blockIdx.x % a.Hkv);
  const int pix = a.n_pairs - 1 - static_cast<int>(blockIdx.x / a.Hkv);  // longest pairs first
  const PairTiles pt = pair_of(a, pix);
  const int G = a.G, QT = a.QT, H = a.H;
  const int n_kv = a.n_kv[pt.t[0].req];

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 8);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 8);
      mbar_init(&p_full[i], 8);
      mbar_init(&pv_done[i], 1);
    }
    for (int i = 0; i < SLOTS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // softmax thread: tile, column half, TMEM lane quarter, row
  const int sw = warp - 2;
  const int tl = sw >> 3;
  const int half = (sw >> 2) & 1;
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;
  const int qi = r / G, g = r - qi * G;
  const AttnTile mt = tl == 1 ? pt.t[1] : pt.t[0];
  const bool valid = warp >= 2 && qi < mt.count && r < QT * G;
  const int pos = valid ? min(a.s_pos[mt.row0 + qi], n_kv - 1) : -1;
  if (warp >= 2 && half == 0) {
    const int wm = __reduce_max_sync(0xffffffffu, pos);
    if (lane == 0) wmaxpos[tl * 4 + quarter] = wm;
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int nbt[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int mp = max(max(wmaxpos[u * 4], wmaxpos[u * 4 + 1]), max(wmaxpos[u * 4 + 2], wmaxpos[u * 4 + 3]));
    nbt[u] = mp < 0 ? 0 : mp / BKV + 1;
  }
  const int nb = max(nbt[0], nbt[1]);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const CUtensorMap* kmap = &a.kmap[pt.t[0].req];
      const CUtensorMap* vmap = &a.vmap[pt.t[0].req];
      const int lc = a.layer_coord[pt.t[0].req];
      int issued = 0;
      for (int x = 0; x < 2 * nb; ++x) {
        const bool is_v = x == 2 * nb - 1 || (x > 0 && (x & 1) == 0);
        const int j = x == 2 * nb - 1 ? nb - 1 : (x & 1) ? (x + 1) >> 1 : is_v ? (x - 2) >> 1 : 0;
        const int st = x % SLOTS;
        if (!mbar_wait_bounded(&empty[st], ((x / SLOTS) & 1) ^ 1, abort_flag)) break;
        uint8_t* dst = smem + OFF_RING + st * SLOT;
        mbar_arrive_expect_tx(&full[st], 2 * ATOM);
        tma_load_4d(dst, is_v ? vmap : kmap, &full[st], 0, kvh, j * BKV, lc);
        tma_load_4d(dst + ATOM, is_v ? vmap : kmap, &full[st], 64, kvh, j * BKV, lc);
        issued = x + 1;
      }
      if (issued < 2 * nb && !*abort_flag) {
        *abort_flag = 1;
        set_status(a.status, ST_WAIT_TIMEOUT);
      }
      // copies issued into slots that nobody consumed must land before the block exits
      for (int x = max(0, issued - SLOTS); x < issued; ++x) mbar_wait_bounded(&full[x % SLOTS], (x / SLOTS) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Lane 0 polls the two tiles' barriers and issues whatever is ready: S_t(j) once the
    // softmax of tile t has read S_t(j-1) and K_j has landed, PV_t(j) once P_t(j) is stored
    // and V_j has landed.  A fixed order would make a tile whose MMA is ready wait behind the
    // other tile's softmax.  A ring slot is released once both tiles are past its block.
    bool ok = true;
    if (lane == 0) {
      for (int u = 0; u < 2; ++u)
        if (nbt[u] > 0 && ok) ok = mbar_wait_bounded(&q_full[u], 0, abort_flag);
      int sn[2] = {0, 0}, pn[2] = {0, 0};  // next S / PV block of each tile
      int k_rel = 0, v_rel = 0;            // next K / V block whose ring slot is still held
      uint64_t t_last = global_ns();
      while (ok && (pn[0] < nbt[0] || pn[1] < nbt[1])) {
        bool progress = false;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int js = sn[u];
          const int xk = k_item(js);
          if (js < nbt[u] && (js == 0 || mbar_test(&s_empty[u], (js - 1) & 1)) &&
              mbar_test(&full[xk % SLOTS], (xk / SLOTS) & 1)) {  // S_u = Q_u K_js^T
            tc_fence_after();
            const uint32_t sq = smem_u32(smem + OFF_Q2 + u * 2 * ATOM);
            const uint32_t sk = smem_u32(smem + OFF_RING + (xk % SLOTS) * SLOT);
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
              const uint64_t da = desc_kmajor(sq + (kk >> 2) * ATOM) + 2 * (kk & 3);
              const uint64_t db = desc_kmajor(sk + (kk >> 2) * ATOM) + 2 * (kk & 3);
              tc_mma_f16(tmem + S_COL + u * 128, da, db, idesc(false), kk > 0 ? 1u : 0u);
            }
            tc_commit(&s_full[u]);
            sn[u] = js + 1;
            progress = true;
          }
          const int jp = pn[u];
          const int xv = v_item(jp, nb);
          if (jp < sn[u] && mbar_test(&p_full[u], jp & 1) && mbar_test(&full[xv % SLOTS], (xv / SLOTS) & 1)) {
            tc_fence_after();  // O_u (+)= P_u V_jp
            const uint32_t sp = smem_u32(smem + OFF_P2 + u * 2 * ATOM);
            const uint32_t sv = smem_u32(smem + OFF_RING + (xv % SLOTS) * SLOT);
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk) {
              const uint64_t da = desc_kmajor(sp + (kk >> 2) * ATOM) + 2 * (kk & 3);
              const uint64_t db = desc_mnmajor(sv + kk * 16 * 128, ATOM);
              tc_mma_f16(tmem + O_COL2 + u * 128, da, db, idesc(true), (jp > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&pv_done[u]);
            pn[u] = jp + 1;
            progress = true;
          }
        }
        // release, in load order per slot, the blocks both tiles have consumed
        while (k_rel < nb && (sn[0] > k_rel || k_rel >= nbt[0]) && (sn[1] > k_rel || k_rel >= nbt[1])) {
          tc_commit(&empty[k_item(k_rel) % SLOTS]);
          ++k_rel;
        }
        while (v_rel < nb && (pn[0] > v_rel || v_rel >= nbt[0]) && (pn[1] > v_rel || v_rel >= nbt[1])) {
          tc_commit(&empty[v_item(v_rel, nb) % SLOTS]);
          ++v_rel;
        }
        if (progress) {
          t_last = global_ns();
        } else if (*abort_flag || global_ns() - t_last > 2000000000ull) {
          ok = false;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, ST_WAIT_TIMEOUT);
      }
      // no MMA may run when the tensor memory is released
      tc_commit(drain);
      mbar_wait_bounded(drain, 0u, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax / output (warps 2..17)
    const int nbu = tl == 1 ? nbt[1] : nbt[0];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(half * 64);
    const uint32_t s_base = tmem + S_COL + tl * 128 + col0 + lane_off;
    const uint32_t o_base = tmem + O_COL2 + tl * 128 + col0 + lane_off;
    float* xs = xch + tl * 2 * ROWS;
    bool ok = true;
    auto wait = [&](uint64_t* b, uint32_t ph) {  // every lane polls: no divergent branch
      if (ok) ok = mbar_wait_bounded(b, ph, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    };
    const uint32_t pair_bar = 1u + static_cast<uint32_t>(tl * 4 + quarter);
    auto sm_bar = [pair_bar]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    if (nbu > 0) {
      {  // Q_tl: half h stores head_dim atom h of its rows
        const uint4* src = reinterpret_cast<const uint4*>(
            a.q + (static_cast<size_t>(mt.row0 + (valid ? qi : 0)) * H + kvh * G + g) * DH + half * 64);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = valid ? src[c] : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(smem + OFF_Q2 + tl * 2 * ATOM + half * ATOM + r * 128 + ((c ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[tl]);
      }
      float m = -1e30f, l = 0.f;
      for (int j = 0; j < nbu; ++j) {
        wait(&s_full[tl], j & 1);
        uint32_t sv[64];
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 64; c += 16) tmem_ld16_nowait(s_base + c, sv + c);
          tmem_wait_ld();
          tc_fence_before();
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) sv[e] = 0u;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[tl]);  // S_{j+1} may now overwrite S_j
        const int k0 = j * BKV + half * 64;
        const bool fullblk = __all_sync(0xffffffffu, k0 + 63 <= pos);
        float pm[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
        if (fullblk) {
#pragma unroll
          for (int e = 0; e < 64; e += 16)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              pm[u] = max3(pm[u], __uint_as_float(sv[e + u]), __uint_as_float(sv[e + 8 + u]));
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (k0 + e <= pos) pm[e & 7] = fmaxf(pm[e & 7], __uint_as_float(sv[e]));
        }
        float mx = max3(max3(pm[0], pm[1], pm[2]), max3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
        mx *= a.scale_log2;
        // row max over both halves through one slot per (tile, half, row): the second barrier
        // keeps either thread from rewriting its slot before the partner has read it
        xs[half * ROWS + r] = mx;
        sm_bar();
        mx = fmaxf(mx, xs[(half ^ 1) * ROWS + r]);
        sm_bar();
        const bool need = mx > m + RESCALE_LOG2;
        const float m_new = need ? mx : m;
        const float alpha = ex2(m - m_new);
        l *= alpha;
        m = m_new;
        // P_j in registers (bf16 pairs), then into this tile's buffer once PV_{j-1} is done
        uint32_t pk[32];
        if (fullblk) {
          const uint64_t sc2 = f2(a.scale_log2, a.scale_log2), nm2 = f2(-m, -m);
          uint64_t acc0 = f2(0.f, 0.f), acc1 = acc0;
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float t0, t1;
            f2_split(fma2(f2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nm2), t0, t1);
            const float p0 = ex2(t0), p1 = ex2(t1);
            if (e & 2)
              acc1 = add2(acc1, f2(p0, p1));
            else
              acc0 = add2(acc0, f2(p0, p1));
            pk[e >> 1] = pack_bf16x2(p0, p1);
          }
          float a0, a1, b0, b1;
          f2_split(acc0, a0, a1);
          f2_split(acc1, b0, b1);
          l += (a0 + a1) + (b0 + b1);
        } else {
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const float p0 = k0 + e <= pos ? ex2(fmaf(__uint_as_float(sv[e]), a.scale_log2, -m)) : 0.f;
            const float p1 = k0 + e + 1 <= pos ? ex2(fmaf(__uint_as_float(sv[e + 1]), a.scale_log2, -m)) : 0.f;
            ls[(e >> 1) & 3] += p0 + p1;
            pk[e >> 1] = pack_bf16x2(p0, p1);
          }
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        if (j > 0) wait(&pv_done[tl], (j - 1) & 1);  // PV_{j-1} read P and wrote O
        if (ok) {
          tc_fence_after();
          uint8_t* pb = smem + OFF_P2 + tl * 2 * ATOM + half * ATOM;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(pb + r * 128 + ((c ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          fence_proxy_async_smem();
        }
        if (__any_sync(0xffffffffu, need) && j > 0 && ok) {
          // lazy rescale, after P (the S values are no longer live): O_tl holds PV_0 ..
          // PV_{j-1}, complete (waited above); PV_j waits for this block's P
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            uint32_t ov[16];
            tmem_ld16_nowait(o_base + c, ov);
            tmem_wait_ld();
            float f[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(ov[e]) * alpha;
            tmem_st16(o_base + c, f);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[tl]);
      }
      // O / (row sum of both halves)
      sm_bar();
      xs[half * ROWS + r] = l;
      wait(&pv_done[tl], (nbu - 1) & 1);  // the last PV of this tile
      sm_bar();
      const float l_all = xs[r] + xs[ROWS + r];  // same order in both halves
      if (ok) {
        tc_fence_after();
        bf16* dst = a.out + (static_cast<size_t>(mt.row0 + (valid ? qi : 0)) * H + kvh * G + g) * DH + half * 64;
        const float inv = l_all > 0.f ? 1.f / l_all : 0.f;
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          uint32_t ov[16];
          tmem_ld16_nowait(o_base + c, ov);
          tmem_wait_ld();
          if (valid) {
            float f[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(ov[e]) * inv;
            store8(dst + c, f);
            store8(dst + c + 8, f + 8);
          }
        }
      }
      if (!ok && lane == 0) {
        *abort_flag = 1;
        set_status(a.status, ST_WAIT_TIMEOUT);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace tp

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
  return G >= ta::ROWS ? 1 : ta::ROWS / G;
}

typedef CUresult (*EncodeTiledFn4)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 4-D map over a KV cache [L][N][Hkv][128] (bf16): box {64, 1, 128 keys, 1}, 128-byte swizzle.
bool encode_kv_map(CUtensorMap* map, const void* base, int n_layers, int n_tokens, int n_kv_heads,
                   long long layer_stride_elems) {
  static EncodeTiledFn4 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn4>(p);
  }
  const uint64_t row = static_cast<uint64_t>(n_kv_heads) * ta::DH * 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(ta::DH), static_cast<cuuint64_t>(n_kv_heads),
                        static_cast<cuuint64_t>(n_tokens), static_cast<cuuint64_t>(layer_stride_elems ? n_layers : 1)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(ta::DH * 2), row,
                           layer_stride_elems ? static_cast<cuuint64_t>(layer_stride_elems) * 2 : row * n_tokens};
  cuuint32_t box[4] = {64, 1, ta::BKV, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tiles per CTA of the bf16 attention, process-wide: 0 chosen per launch (two when the
// tile pairs of a launch fill the SMs), 1 or 2 forced (tests, tuning).
static std::atomic<int> g_attn_tiles{0};

void attention_set_tiles(int tiles) { g_attn_tiles.store(tiles); }

// Two tiles per CTA when the waves of pair units finish sooner than the waves of single
// tiles: a pair unit takes ~1.5x a single tile's time (measured on GB300: full causal 8320
// tokens, 56/8 heads 1.359 -> 1.045 ms in 25 -> 13 waves; 1357 of 8320 queries 0.232 ->
// 0.183 ms; 3200 tokens, 32/8 heads 0.140 -> 0.119 ms), so the pairs win where they save a
// wave or more (884 of 8256 queries, 64/8 heads, 3 -> 2 waves: 0.167 ms either way).  With
// one head per KV head (MHA, 128 queries a tile) the two tiles of a sparse pair often differ
// in length: pairs only when single tiles take four waves or more (4128 causal, 32 heads:
// 0.216 -> 0.185 ms; 646 of 4128 queries, 2 waves: 0.067 ms alone, 0.093 paired).
static bool use_pairs(long long tiles, long long pairs, int n_heads, int n_kv_heads, int n_sm) {
  const int mode = g_attn_tiles.load();
  if (mode != 0) return mode == 2;
  const long long w1 = (tiles * n_kv_heads + n_sm - 1) / n_sm;
  const long long w2 = (pairs * n_kv_heads + n_sm - 1) / n_sm;
  if (n_heads == n_kv_heads && w1 < 4) return false;
  return 1.5 * static_cast<double>(w2) < 0.97 * static_cast<double>(w1);
}

static int sm_count_cached() {
  static int n_sm = 0;
  if (n_sm == 0) {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    n_sm = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0 ? v : 148;
  }
  return n_sm;
}

static cudaError_t tc2_launch(ta::Args& args, cudaStream_t s) {
  static DeviceOnce configured;
  cudaError_t e = max_dynamic_smem_once(reinterpret_cast<const void*>(tp::attn_tc2_kernel), tp::SMEM2, configured);
  if (e != cudaSuccess) return e;
  if (args.n_pairs <= 0) return cudaSuccess;
  launch_chain(tp::attn_tc2_kernel, dim3(args.n_pairs * args.Hkv), dim3(tp::THREADS2), tp::SMEM2, s, args);
  return cudaGetLastError();
}

static cudaError_t tc_launch(ta::Args& args, int n_tiles, cudaStream_t s) {
  static DeviceOnce configured;
  cudaError_t e = max_dynamic_smem_once(reinterpret_cast<const void*>(ta::attn_tc_kernel), ta::SMEM, configured);
  if (e != cudaSuccess) return e;
  if (n_tiles <= 0) return cudaSuccess;
  args.n_tiles = n_tiles;
  const int paired = args.part_o ? std::min(args.n_paired, n_tiles) : 0;
  args.n_paired = paired;
  dim3 grid((n_tiles + paired) * args.Hkv);
  launch_chain(ta::attn_tc_kernel, grid, dim3(ta::THREADS), ta::SMEM, s, args);
  return cudaGetLastError();
}

// Batched (bf16): one launch per group of at most MAXREQ requests; tiles of request r are
// tiles[tile_off[r] .. tile_off[r+1]).
cudaError_t launch_attention_bf16(const void* q, const int32_t* s_pos, const AttnTile* tiles, const int* tile_off,
                                  const CUtensorMap* kmaps, const CUtensorMap* vmaps, const int* n_kv,
                                  const int* one_layer, int n_req, int layer, int n_heads, int n_kv_heads, void* out,
                                  int32_t* status, float* part_o, float2* part_ml, int* part_cnt, cudaStream_t s) {
  ta::Args a;
  // Key-range splits: when one CTA per (tile, head) unit leaves SMs idle, the longest tiles get a
  // second CTA -- as many tiles as the idle SMs hold, plus two per KV head: the CTAs past one wave
  // are then the shortest tiles', which start as soon as the first short tiles finish.  One launch
  // per layer.  Measured on GB300 (535 selected rows of 3200, 136 units on 152 SMs), attention
  // phase per blend: no pairs 1.68 ms, the idle SMs' 2 tiles per head 1.63, 4 tiles 1.47, 6 tiles
  // 1.71, every tile 1.91 (the extra CTAs' fixed cost and a second wave); seam repair (176 rows,
  // 48 units, every tile paired) 7.38 -> 7.20 ms per blend.
  const int n_sm = sm_count_cached();
  long long pairs = 0;
  for (int r = 0; r < n_req; ++r) pairs += (tile_off[r + 1] - tile_off[r] + 1) / 2;
  const bool two = use_pairs(tile_off[n_req], pairs, n_heads, n_kv_heads, n_sm);
  const long long units = static_cast<long long>(tile_off[n_req]) * n_kv_heads;
  const int n_paired = (n_req <= ta::MAXREQ && units < n_sm)
                           ? static_cast<int>(std::min<long long>(tile_off[n_req], (n_sm - units) / n_kv_heads + 2))
                           : 0;
  const bool split = part_o && part_ml && part_cnt && n_paired > 0 &&
                     static_cast<long long>(n_paired) * n_kv_heads <= ATTN_SPLIT_UNITS;
  a.part_o = split ? part_o : nullptr;
  a.n_paired = split ? n_paired : 0;
  a.part_ml = part_ml;
  a.part_cnt = part_cnt;
  a.q = static_cast<const bf16*>(q);
  a.s_pos = s_pos;
  a.H = n_heads;
  a.Hkv = n_kv_heads;
  a.G = n_heads / n_kv_heads;
  a.QT = attention_tile_rows(n_heads, n_kv_heads, CB_BF16);
  a.out = static_cast<bf16*>(out);
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(ta::DH));
  a.status = status;
  a.direct_m = 0;
  for (int r0 = 0; r0 < n_req; r0 += ta::MAXREQ) {
    const int r1 = std::min(n_req, r0 + ta::MAXREQ);
    for (int r = r0; r < r1; ++r) {
      a.kmap[r - r0] = kmaps[r];
      a.vmap[r - r0] = vmaps[r];
      a.n_kv[r - r0] = n_kv[r];
      a.layer_coord[r - r0] = one_layer[r] ? 0 : layer;
    }
    a.req_base = r0;
    a.tiles = tiles + tile_off[r0];
    cudaError_t e;
    if (two) {
      int np = 0;
      for (int r = r0; r <= r0 + ta::MAXREQ - 1; ++r) {
        const int rr = std::min(r, r1);  // entries past the group repeat its end
        a.tile_off[r - r0] = tile_off[rr] - tile_off[r0];
        a.pair_off[r - r0] = np;
        if (r < r1) np += (tile_off[r + 1] - tile_off[r] + 1) / 2;
      }
      a.tile_off[ta::MAXREQ] = tile_off[r1] - tile_off[r0];
      a.pair_off[ta::MAXREQ] = np;
      a.n_pairs = np;
      e = tc2_launch(a, s);
    } else {
      e = tc_launch(a, tile_off[r1] - tile_off[r0], s);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// fp32 (all rows of S).
cudaError_t launch_attention(const void* q, const int32_t* s_pos, const int32_t* s_req, const ReqDev* reqs,
                             const AttnTile* tiles, int n_tiles, int layer, int n_heads, int n_kv_heads, int head_dim,
                             void* out, cb_dtype dt, cudaStream_t s) {
  (void)tiles;
  if (n_tiles <= 0) return cudaSuccess;
  if (dt != CB_F32) return cudaErrorInvalidValue;
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
    ta::Args a;
    if (!encode_kv_map(&a.kmap[0], k, 1, n_kv, n_kv_heads, 0) || !encode_kv_map(&a.vmap[0], v, 1, n_kv, n_kv_heads, 0))
      return cudaErrorInvalidValue;
    a.n_kv[0] = n_kv;
    a.layer_coord[0] = 0;
    a.q = static_cast<const bf16*>(q);
    a.s_pos = q_pos;
    a.tiles = nullptr;
    a.req_base = 0;
    a.n_paired = 0;
    a.part_o = nullptr;  // one CTA per tile
    a.part_ml = nullptr;
    a.part_cnt = nullptr;
    a.direct_m = m;
    a.H = n_heads;
    a.Hkv = n_kv_heads;
    a.G = n_heads / n_kv_heads;
    a.QT = attention_tile_rows(n_heads, n_kv_heads, CB_BF16);
    a.out = static_cast<bf16*>(out);
    a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(head_dim));
    a.status = nullptr;
    const int n_tiles = (m + a.QT - 1) / a.QT;
    if (use_pairs(n_tiles, (n_tiles + 1) / 2, n_heads, n_kv_heads, sm_count_cached())) {
      a.n_pairs = (n_tiles + 1) / 2;
      return tc2_launch(a, s);
    }
    return tc_launch(a, n_tiles, s);
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
