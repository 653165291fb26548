// Dense projections C = A . B^T of the blended prefill on CTA pairs.
//
// The weights sit on the tensor core's rows.  A cluster holds one CTA pair (2 CTAs) or two
// (4 CTAs), one CTA per SM.  A pair computes a tile of 256 weight rows (128 per CTA) by bt
// tokens, bt a multiple of 16 up to 256 (each CTA stages bt/2 of the tokens): the pair's even
// CTA issues one tcgen05.mma.cta_group::2 (M = 256, N = bt) per 16 elements of K into the
// tensor memory of both CTAs.  Per SM and 64-element k-block this stages 128 weight rows and
// bt/2 token rows, where a single-CTA 128 x 256 tile stages 384 rows: fewer bytes leave L2
// per tensor-core cycle, and L2 -> SM bandwidth is what bounds the single-CTA kernel (ncu on
// GB300 at 1357 tokens: ~18.5 TB/s of L2 -> SM reads, tensor pipe ~66 % busy).  In a cluster
// of two pairs both pairs take the same 256 weight rows for two token tiles, and each CTA
// loads half of its 128 weight rows and multicasts them to its counterpart in the other pair.
//   warp 0: TMA producer   warp 1: tensor-memory owner and, in even CTAs, the MMA issuer
//   warps 2-5: epilogue (tensor memory -> fp32 store, fp32 residual add, or SiLU(gate) * up)
// A ring stage holds ksub (1 or 2) 64-element atoms of K.  Measured on GB300, each barrier
// round of the issuing thread (wait for a stage, commit its release) costs about as much as
// issuing four of the MMAs, so two atoms per stage (eight MMAs per round) keep the tensor
// core busier even though fewer, larger stages fit.  Shared memory left over by the ring
// holds the epilogue's output slabs, as many as fit, so that the epilogue of one tile keeps
// several TMA stores in flight while the next tile's main loop runs.
// SwiGLU: each CTA's 128 rows are 64 gate rows and the 64 up rows of the same features (a
// pair covers 128 features); the output goes out as 16-token x 64-feature bf16 tiles.
// Every wait is bounded: on timeout the kernel records ST_WAIT_TIMEOUT, and the cluster
// still meets at its closing barrier before any CTA frees its tensor memory or leaves.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace cb {
namespace pr {

constexpr int THREADS = 192;
constexpr int ROWS = 128;                 // weight rows per CTA (the MMA's rows in this CTA)
constexpr int BK = 64;                    // elements of K per 128-byte swizzle atom
constexpr int A_ATOM = ROWS * BK * 2;     // 16 KiB: 128 weight rows x one atom of K
constexpr int MAX_STAGES = 12;
constexpr int OFF_RING = 1024;            // after the barriers
constexpr int SMEM_ALLOC = 232448;        // the per-block maximum (227 KiB), 1 KiB of it aligns the base
constexpr int SMEM_USE = SMEM_ALLOC - 1024;
constexpr int XCH_BYTES = 4608;           // SwiGLU exchange: 2 x 64 rows x 9 floats
// RoPE epilogue: the tile's positions and its K/V destination rows
constexpr int XCH_ROPE = 256 * 4 + 256 * 8;
constexpr int F32_SLAB = 8 * ROWS * 4;    // 8 tokens x 128 features fp32
constexpr int F32_SLAB_TOK = 8;
constexpr int BF_SLAB = 16 * 64 * 2;      // 16 tokens x 64 features bf16
constexpr uint32_t TMEM_COLS = 512;       // two accumulators of up to 256 columns
constexpr int ACC_STRIDE = 256;

// The epilogue's exchange area and output slab (a bf16 16-token tile of the RoPE epilogue is
// as large as an fp32 8-token slab), and the shared memory it needs at the least.
__host__ __device__ constexpr int epi_xch(int mode) {
  return mode == EPI_SWIGLU ? XCH_BYTES : mode == EPI_QKV_ROPE ? XCH_ROPE : 0;
}
__host__ __device__ constexpr int epi_slab(int mode) { return mode == EPI_SWIGLU ? BF_SLAB : F32_SLAB; }
__host__ __device__ constexpr int min_staging(int mode) { return epi_xch(mode) + 2 * epi_slab(mode); }

struct Params {
  int M, N, K, mode;
  void* out;
  int ldc;
  int split0, split1;  // non-SwiGLU weight rows [0,split0) from map 0, [split0,split1) map 1, rest map 2
  int32_t* status;
  int bt;              // tokens per pair tile
  int tok_tiles;       // ceil(M / bt)
  int tok_groups;      // token tiles per cluster unit: ceil(tok_tiles / pairs per cluster)
  int units;           // weight tiles x tok_groups
  int ksub;            // 64-element atoms of K per ring stage (1 or 2)
  int n_kb;            // ring stages per unit: K / (64 ksub)
  int stages;          // ring depth
  int stage_bytes;     // ksub x (16 KiB of weights + bt/2 x 128 B of tokens), per CTA
  int stg_off;         // epilogue staging: offset (after the ring)
  int slabs;           // output slabs in the staging area (2, 4, 8 or 16)
  QkvRope qr;          // EPI_QKV_ROPE only
};

// The idx-th unit of cluster cid, round-robin (false when there is none).
__device__ __forceinline__ bool get_unit(const Params& p, int cid, int NC, int idx, int& u) {
  u = cid + idx * NC;
  return u < p.units;
}


// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major, M = 256, N = n.
__host__ __device__ constexpr uint32_t idesc_pair(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Unit u of the persistent loop: weight tile u / tok_groups, token group u % tok_groups
// (consecutive clusters take the same weight rows, which then come from DRAM once).
// ROPE: the EPI_QKV_ROPE instantiation (its producer loads q and k rows interleaved, its
// epilogue rotates); the other epilogues run in the instantiation without it.
template <int CL, bool ROPE>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                     const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
                     const __grid_constant__ CUtensorMap tmC, Params p) {
  constexpr int PPC = CL / 2;  // pairs per cluster
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [stages], used in even CTAs
  uint64_t* empty = full + MAX_STAGES;                 // [stages]
  uint64_t* acc_full = empty + MAX_STAGES;             // [2]
  uint64_t* acc_empty = acc_full + 2;                  // [2], used in even CTAs
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort, [1..2] go

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int q = static_cast<int>(rank >> 1), h = static_cast<int>(rank & 1u);
  const bool even = h == 0;
  const int cid = static_cast<int>(cluster_id_x()), NC = static_cast<int>(n_clusters_x());
  const uint32_t stages = static_cast<uint32_t>(p.stages);
  uint8_t* ring = smem + OFF_RING;

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PPC);  // one commit from the MMA issuer of each pair
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // the four epilogue warps of both CTAs of the pair
    }
    mbar_init(drain, 1);
    abort_flag[0] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW0);
    prefetch_tmap(&tmW1);
    prefetch_tmap(&tmC);
    if (p.mode != EPI_SWIGLU) prefetch_tmap(&tmW2);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // every CTA's barriers are initialised before a copy, commit or arrive of another reaches them
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  const uint32_t lead = rank & ~1u;  // the even CTA of this CTA's pair
  const int half_rows = p.bt / 2;
  const uint32_t b_atom = static_cast<uint32_t>(half_rows) * 128u;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint16_t mc_mask = static_cast<uint16_t>((1u << h) | (1u << (2 + h)));  // (0,h) and (1,h)
      // this CTA's 128 weight rows of unit u: rows r_lo.. of map m_lo, then r_hi.. of map m_hi
      auto weight_rows = [&](int u, const CUtensorMap*& m_lo, const CUtensorMap*& m_hi, int& r_lo, int& r_hi,
                             bool& inter) {
        const int wt = u / p.tok_groups;
        m_lo = &tmW0;
        m_hi = &tmW1;
        inter = false;
        if (p.mode == EPI_SWIGLU) {
          r_lo = r_hi = wt * 128 + h * 64;  // 64 gate rows, then the up rows of the same features
        } else {
          const int f = wt * 256 + h * 128;
          const CUtensorMap* m = &tmW0;
          int r = f;
          if (f >= p.split1) {
            m = &tmW2;
            r = f - p.split1;
          } else if (f >= p.split0) {
            m = &tmW1;
            r = f - p.split0;
          }
          m_lo = m_hi = m;
          r_lo = r;
          r_hi = r + 64;
          inter = ROPE && f < p.split1;  // q or k head: r_lo / 128 is the head
        }
      };
      // weight atom j of stage s (k-block kb): to this CTA, and by multicast in clusters of two pairs
      auto load_weight_atom = [&](uint32_t s, int kb, int j, const CUtensorMap* m_lo, const CUtensorMap* m_hi, int r_lo,
                                  int r_hi, bool inter) {
        uint8_t* aj = ring + s * static_cast<uint32_t>(p.stage_bytes) + j * A_ATOM;
        const uint32_t bar = mapa_shared(smem_u32(&full[s]), lead);
        const int k0 = (kb * p.ksub + j) * BK;
        if (inter) {
          // rows (i, i + 64) of the head for i < 32, then for i >= 32: 64 rows per box
          const int head = r_lo / ROWS;
          if (PPC == 2) {
            tma_load_4d_pair_mc(aj + q * (A_ATOM / 2), m_lo, bar, k0, 0, q * 32, head, mc_mask);
          } else {
            tma_load_4d_pair(aj, m_lo, bar, k0, 0, 0, head);
            tma_load_4d_pair(aj + A_ATOM / 2, m_lo, bar, k0, 0, 32, head);
          }
        } else if (PPC == 2) {
          // half of the weight rows, to this CTA and to its counterpart in the other pair
          if (q == 0)
            tma_load_2d_pair_mc(aj, m_lo, bar, k0, r_lo, mc_mask);
          else
            tma_load_2d_pair_mc(aj + A_ATOM / 2, m_hi, bar, k0, r_hi, mc_mask);
        } else {
          tma_load_2d_pair(aj, m_lo, bar, k0, r_lo);
          tma_load_2d_pair(aj + A_ATOM / 2, m_hi, bar, k0, r_hi);
        }
      };
      int u = 0;
      uint32_t s = 0, ph = 0;
      bool ok = true;
      for (int idx = 0; ok && get_unit(p, cid, NC, idx, u); ++idx) {
        const int tt = (u % p.tok_groups) * PPC + q;
        const int trow = tt * p.bt + h * half_rows;  // first token this CTA stages
        const CUtensorMap *m_lo, *m_hi;
        int r_lo, r_hi;
        bool inter;
        weight_rows(u, m_lo, m_hi, r_lo, r_hi, inter);
        for (int kb = 0; kb < p.n_kb; ++kb) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = ring + s * static_cast<uint32_t>(p.stage_bytes) + p.ksub * A_ATOM;
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), lead);
          // (each atom's weights and tokens back to back: measured faster on GB300 than all
          // weight atoms first, e.g. the Yi-34B gate/up 482 -> 465 us)
          if (even) mbar_arrive_expect_tx(&full[s], 2u * static_cast<uint32_t>(p.stage_bytes));
          for (int j = 0; j < p.ksub; ++j) {
            load_weight_atom(s, kb, j, m_lo, m_hi, r_lo, r_hi, inter);
            tma_load_2d_pair(sb + j * b_atom, &tmX, bar, (kb * p.ksub + j) * BK, trow);
          }
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        abort_flag[0] = 1;
        set_status(p.status, ST_WAIT_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTAs)
    if (even && lane == 0) {
      const uint32_t idesc = idesc_pair(p.bt);
      const uint16_t all_mask = static_cast<uint16_t>((1u << CL) - 1u);
      const uint16_t pair_mask = static_cast<uint16_t>(3u << (2 * q));
      const uint32_t ring_u32 = smem_u32(ring);
      const uint32_t sbytes = static_cast<uint32_t>(p.stage_bytes);
      const uint32_t b_off = static_cast<uint32_t>(p.ksub * A_ATOM);
      const uint64_t a_step = A_ATOM >> 4, b_step = b_atom >> 4;  // descriptor steps per atom
      const int ksub = p.ksub;
      uint32_t s = 0, ph = 0, sa = ring_u32;
      bool ok = true;
      int u = 0;
      for (int i = 0; ok && get_unit(p, cid, NC, i, u); ++i) {
        const int b = i & 1;
        const uint32_t use = static_cast<uint32_t>(i >> 1);
        if (!mbar_wait_bounded(&acc_empty[b], (use & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tacc = tmem + static_cast<uint32_t>(b * ACC_STRIDE);
        uint32_t accum = 0u;  // the tile's first MMA overwrites the accumulator
        for (int kb = 0; kb < p.n_kb; ++kb) {
          if (!mbar_try_wait(&full[s], ph) && !mbar_wait_bounded(&full[s], ph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint64_t da = sw128_desc(sa), db = sw128_desc(sa + b_off);
          for (int j = 0; j < ksub; ++j) {  // +32 bytes along K per MMA (encoded >> 4)
            tc_mma_f16_pair(tacc, da, db, idesc, accum);
            tc_mma_f16_pair(tacc, da + 2, db + 2, idesc, 1u);
            tc_mma_f16_pair(tacc, da + 4, db + 4, idesc, 1u);
            tc_mma_f16_pair(tacc, da + 6, db + 6, idesc, 1u);
            accum = 1u;
            da += a_step;
            db += b_step;
          }
          tc_commit_pair_mc(&empty[s], all_mask);  // frees stage s in every CTA once read
          sa += sbytes;
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
            sa = ring_u32;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&acc_full[b], pair_mask);  // accumulator b complete in both CTAs
      }
      if (!ok) {
        abort_flag[0] = 1;
        set_status(p.status, ST_WAIT_TIMEOUT);
      }
      // no MMA may still be running when the cluster meets at its closing barrier
      tc_commit_pair_mc(drain, static_cast<uint16_t>(1u << rank));
      mbar_wait_bounded(drain, 0u, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;           // tensor-memory lanes 32 quarter .. +31
    const int r_loc = quarter * 32 + lane;  // this thread's weight row within the CTA
    const int et = threadIdx.x - 64;        // et == 0 issues the output stores
    volatile int* go = abort_flag + 1;
    const uint32_t acc_empty_lead = mapa_shared(smem_u32(acc_empty), lead);
    uint8_t* stg = smem + p.stg_off;
    const bool swig = p.mode == EPI_SWIGLU;
    float* xg = reinterpret_cast<float*>(stg);  // SwiGLU: gate of tokens 8-15 [64][9]
    float* xu = xg + 64 * 9;                     //         up of tokens 0-7 [64][9]
    int* upos = reinterpret_cast<int*>(stg);     // RoPE: the tile's positions [256]
    bf16** udst = reinterpret_cast<bf16**>(upos + 256);
    uint8_t* slab0 = stg + epi_xch(p.mode);
    const int slab_bytes = epi_slab(p.mode);
    const int keep = p.slabs - 1;  // stores that may still read their slab when one is refilled
    int slab = 0;                  // output slabs issued so far
    int u = 0, nx = 0;
    for (int i = 0; get_unit(p, cid, NC, i, u); ++i) {
      const int b = i & 1;
      // The last unit's stores are staged in the ring, which its accumulator's completion
      // leaves idle (every copy landed and was read): one fresh slab each, none waited for
      // (measured on GB300: 1-2 % per launch, the last unit's epilogue being the tail).
      const bool last = !get_unit(p, cid, NC, i + 1, nx) &&
                        (swig ? (p.bt / 16) * BF_SLAB
                              : (p.mode == EPI_QKV_ROPE ? p.bt / 16 : p.bt / F32_SLAB_TOK) * F32_SLAB) <=
                            p.stg_off - OFF_RING;
      int fresh = 0;  // ring slabs used by the last unit
      const uint32_t use = static_cast<uint32_t>(i >> 1);
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(&acc_full[b], use & 1u, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok && lane == 0) {
        abort_flag[0] = 1;
        set_status(p.status, ST_WAIT_TIMEOUT);
      }
      // one decision for the four warps, so that each named barrier below is met by all
      epi_bar();
      if (et == 0) go[b] = !abort_flag[0];
      epi_bar();
      if (!go[b]) break;
      tc_fence_after();
      const int tt = (u % p.tok_groups) * PPC + q, wt = u / p.tok_groups;
      const int t0 = tt * p.bt;
      const int nt = min(p.bt, p.M - t0);  // <= 0: a pad tile of the second pair, nothing to store
      const uint32_t tbase = tmem + static_cast<uint32_t>(b * ACC_STRIDE) + (static_cast<uint32_t>(quarter * 32) << 16);
      if (swig) {
        // lanes 0-63 hold the gate and lanes 64-127 the up projection of features
        // f0 .. f0 + 63; per 16 tokens the gate warps pass the gate of tokens 8-15 and the up
        // warps the up of tokens 0-7 through shared memory, then the gate warps write
        // SiLU(gate) * up of tokens 0-7 and the up warps of tokens 8-15 into a 16-token x
        // 64-feature bf16 tile, stored by one thread
        const int f0 = wt * 128 + h * 64;
        const int fr = r_loc & 63;
        const bool gate_row = quarter < 2;
#pragma unroll 1
        for (int c = 0; c < nt; c += 16, ++slab) {
          float v[16];
          tmem_ld16(tbase + c, v);
          bf16* tile = reinterpret_cast<bf16*>(last ? ring + (fresh++) * slab_bytes : slab0 + (slab % p.slabs) * slab_bytes);
          if (et == 0 && !last) bulk_wait_read_keep(keep);  // the store that last used this slab has read it
#pragma unroll
          for (int j = 0; j < 8; ++j) (gate_row ? xg : xu)[fr * 9 + j] = v[gate_row ? 8 + j : j];
          epi_bar();
          if (gate_row) {
#pragma unroll
            for (int j = 0; j < 8; ++j) tile[j * 64 + fr] = __float2bfloat16_rn(silu_f(v[j]) * xu[fr * 9 + j]);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) tile[(8 + j) * 64 + fr] = __float2bfloat16_rn(silu_f(xg[fr * 9 + j]) * v[8 + j]);
          }
          fence_proxy_async_smem();
          epi_bar();
          if (et == 0) {
            tma_store_2d(&tmC, tile, f0, t0 + c);
            bulk_commit();
          }
        }
      } else if (ROPE) {
        if (nt > 0) {  // (uniform) a pad tile stores nothing
          // This CTA's 128 rows are one head of q, k or v.  Per 16 tokens: q and k rotate at each
          // token's position (dimension i with i + 64) and round to bf16 into a 16-token x
          // 128-dimension tile; q's tile is one TMA store into q_out, k's and v's rows are copied
          // to the fused cache row of each token's position (256 contiguous bytes per token).
          const int f0 = wt * 256 + h * 128;
          const int kind = f0 < p.split0 ? 0 : f0 < p.split1 ? 1 : 2;  // q, k, v
          const int head = (kind == 0 ? f0 : kind == 1 ? f0 - p.split0 : f0 - p.split1) / ROWS;
          const int di = r_loc >> 1;  // q, k: this lane's rotation pair (rows interleaved)
          const QkvRope& qr = p.qr;
          // Once per tile: the tokens' positions (clamped for the table; out-of-range rows are not
          // stored) and, for k and v, each token's destination row in the fused cache (null when
          // the position is out of range).  (cos, sin) of a round's 16 tokens are loaded two
          // rounds ahead.
          for (int x = et; x < nt; x += 128) {
            const int pos = __ldg(qr.s_pos + t0 + x);
            upos[x] = min(max(pos, 0), qr.max_pos - 1);
            if (kind > 0) {
              const ReqDev rq = qr.reqs[__ldg(qr.s_req + t0 + x)];
              bf16* row = nullptr;
              if (pos >= 0 && pos < rq.n_tokens && pos < qr.max_pos) {
                row = static_cast<bf16*>(kind == 1 ? rq.k : rq.v) + static_cast<size_t>(qr.layer) * rq.layer_stride +
                      static_cast<size_t>(pos) * qr.kvw + head * ROWS;
              } else {
                set_status(p.status, ST_RANGE);
              }
              udst[x] = row;
            }
          }
          epi_bar();
          float2 cs1[16], cs2[16];
          if (kind < 2) {
  #pragma unroll
            for (int j = 0; j < 16; ++j) cs1[j] = __ldg(qr.rope + static_cast<size_t>(upos[min(j, nt - 1)]) * 64 + di);
  #pragma unroll
            for (int j = 0; j < 16; ++j) cs2[j] = __ldg(qr.rope + static_cast<size_t>(upos[min(16 + j, nt - 1)]) * 64 + di);
          }
  #pragma unroll 1
          for (int c = 0; c < nt; c += 16, ++slab) {
            float v[16];
            tmem_ld16(tbase + c, v);
            bf16* tile = reinterpret_cast<bf16*>(last ? ring + (fresh++) * slab_bytes : slab0 + (slab % p.slabs) * slab_bytes);
            if (et == 0 && !last && kind == 0) bulk_wait_read_keep(keep);  // the store that last used this slab has read it
            if (kind < 2) {
              // q and k rows are loaded interleaved: lane pairs (2i, 2i + 1) hold rows i and i + 64
              // of the head, which meet by a shuffle
              float2 cs[16];
  #pragma unroll
              for (int j = 0; j < 16; ++j) {
                cs[j] = cs1[j];
                cs1[j] = cs2[j];
              }
              if (c + 32 < nt) {
  #pragma unroll
                for (int j = 0; j < 16; ++j)
                  cs2[j] = __ldg(qr.rope + static_cast<size_t>(upos[min(c + 32 + j, nt - 1)]) * 64 + di);
              }
              const bool lo = (r_loc & 1) == 0;
              const int dim = (r_loc >> 1) + (lo ? 0 : 64);
  #pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float w = __shfl_xor_sync(0xffffffffu, v[j], 1);
                const float a = lo ? v[j] : w;
                const float b = lo ? w : v[j];
                const float o = lo ? a * cs[j].x - b * cs[j].y : b * cs[j].x + a * cs[j].y;
                tile[j * ROWS + dim] = __float2bfloat16_rn(o);
              }
            } else {
  #pragma unroll
              for (int j = 0; j < 16; ++j) tile[j * ROWS + r_loc] = __float2bfloat16_rn(v[j]);
            }
            fence_proxy_async_smem();
            epi_bar();
            if (kind == 0) {
              if (et == 0) {
                tma_store_2d(&tmC, tile, head * ROWS, t0 + c);
                bulk_commit();
              }
            } else {
              // two tokens per thread, 16 bytes of each
              const int ch = et & 15;
  #pragma unroll
              for (int pass = 0; pass < 2; ++pass) {
                const int j = (et >> 4) + pass * 8;
                if (c + j < nt) {
                  bf16* row = udst[c + j];
                  if (row) *reinterpret_cast<uint4*>(row + ch * 8) = *reinterpret_cast<const uint4*>(tile + j * ROWS + ch * 8);
                }
              }
            }
          }
        }
      } else {
        // 8-token x 128-feature fp32 slabs, one TMA store (or add-reduction) each; a
        // 16-column tensor-memory load feeds two of them
        const int f0 = wt * 256 + h * 128;
#pragma unroll 1
        for (int c = 0; c < nt; c += 16) {
          float v[16];
          tmem_ld16(tbase + c, v);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (c + half * F32_SLAB_TOK >= nt) break;  // (uniform)
            float* sbuf = reinterpret_cast<float*>(last ? ring + (fresh++) * slab_bytes : slab0 + (slab % p.slabs) * slab_bytes);
            ++slab;
            if (et == 0 && !last) bulk_wait_read_keep(keep);
            epi_bar();
#pragma unroll
            for (int j = 0; j < F32_SLAB_TOK; ++j) sbuf[j * ROWS + r_loc] = v[half * F32_SLAB_TOK + j];
            fence_proxy_async_smem();
            epi_bar();
            if (et == 0) {
              if (p.mode == EPI_ADD_F32)
                tma_reduce_add_2d(&tmC, sbuf, f0, t0 + c + half * F32_SLAB_TOK);
              else
                tma_store_2d(&tmC, sbuf, f0, t0 + c + half * F32_SLAB_TOK);
              bulk_commit();
            }
          }
        }
      }
      // accumulator b may be overwritten once every epilogue warp of both CTAs has read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_lead + static_cast<uint32_t>(b * 8));
    }
    if (et == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  // No CTA leaves, or frees the pair's tensor memory, while another may still reach its
  // barriers or shared memory: every issuer has drained its MMAs (whose completion follows
  // every copy they read), every producer and epilogue has finished.
  cluster_sync_all();
  // After a timeout anywhere in the cluster, copies issued for stages that were never
  // consumed may still be in flight: give them time to land before the memory is released.
  if (abort_flag[0] || (p.status != nullptr && (*reinterpret_cast<volatile int32_t*>(p.status) & ST_WAIT_TIMEOUT))) {
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 200000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// Ring stages and epilogue slabs of one configuration (0 stages: it does not fit).
struct Layout {
  int stage_bytes, stages, stg_off, slabs;
};
__host__ inline Layout layout(int bt, int ksub, int mode) {
  Layout l{};
  l.stage_bytes = ksub * (A_ATOM + bt * 64);
  l.stages = std::min(MAX_STAGES, (SMEM_USE - OFF_RING - min_staging(mode)) / l.stage_bytes);
  l.stg_off = OFF_RING + l.stages * l.stage_bytes;
  const int room = (SMEM_USE - l.stg_off - epi_xch(mode)) / epi_slab(mode);
  l.slabs = room >= 16 ? 16 : room >= 8 ? 8 : room >= 4 ? 4 : 2;  // the waits take 1, 3, 7 or 15 in flight
  return l;
}

}  // namespace pr

// ============================================================================= planner + launcher
// 0: time model; 1: never; 2: clusters of one pair; 4: clusters of two pairs.
static std::atomic<int> g_pairing{0};
void gemm_set_pairing(int m) { g_pairing.store(m); }
int gemm_pairing() { return g_pairing.load(); }

// Clusters of `cl` CTAs that are resident at once (one CTA per SM), per device.
static int max_clusters(int cl) {
  static std::atomic<int> cache[2][64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int ci = cl == 4 ? 1 : 0;
  if (dev >= 0 && dev < 64) {
    const int v = cache[ci][dev].load();
    if (v > 0) return v;
  }
  // (the RoPE instantiation has the same block and shared memory: one CTA per SM either way)
  const void* fn = cl == 4 ? reinterpret_cast<const void*>(pr::gemm_pair_kernel<4, false>)
                           : reinterpret_cast<const void*>(pr::gemm_pair_kernel<2, false>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, pr::SMEM_ALLOC) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t q = {};
  q.gridDim = dim3(cl * 64);
  q.blockDim = dim3(pr::THREADS);
  q.dynamicSmemBytes = pr::SMEM_ALLOC;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &q) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) cache[ci][dev].store(n);
  return n;
}

// Time model of the paired kernel (microseconds at the ~1.75 GHz these kernels run at).
// Measured on GB300 with clock64 counters in the issuing thread: a 64-element k-block costs
// about max(2 bt + 70, 460) cycles with two atoms per ring stage (the tensor core's 2 bt
// cycles at N = bt, or the issuing thread's eight MMAs plus one barrier round) and about
// max(2 bt + 90, 640) with one; a shallow ring adds the copy latency (~2200 cycles) spread
// over the k-blocks in flight.  The clusters take units round-robin; a unit's epilogue
// overlaps the next unit's main loop unless it is longer, and the first stage's arrival
// (~5000 cycles) and the last unit's epilogue are exposed.  The epilogue writes about 24
// bytes per cycle (fp32 slabs) or the SwiGLU tile at about 8 bytes of input per cycle.
static double pair_us(int M, int K, int w_tiles, int cl, int bt, int ksub, int clusters, int mode) {
  const bool swiglu = mode == EPI_SWIGLU;
  const pr::Layout l = pr::layout(bt, ksub, mode);
  const int ppc = cl / 2;
  const int tok_tiles = (M + bt - 1) / bt;
  const int groups = (tok_tiles + ppc - 1) / ppc;
  const long long units = static_cast<long long>(w_tiles) * groups;
  const double issue = ksub == 2 ? std::max(2.0 * bt + 70.0, 460.0) : std::max(2.0 * bt + 90.0, 640.0);
  const double lat = 2200.0 / ((l.stages - 1) * ksub);
  const double kb = std::max(issue, lat);
  const double main = (K / 64) * kb;
  const double epi = swiglu ? bt * 96.0 : bt * 50.0;  // per token (measured: 10.5 us / 192, 4.9 us / 176)
  const double unit = std::max(main, epi);
  return (((units + clusters - 1) / clusters) * unit + 5000.0 + epi) / 1750.0;
}

bool plan_gemm_pair(int M, int N, int K, int split0, int split1, int mode, int forced_bt, PairPlan* out) {
  const int pm = g_pairing.load();
  if (pm == 1 || M <= 0 || K % 64 != 0) return false;
  const bool swiglu = mode == EPI_SWIGLU;
  int w_tiles;
  if (swiglu) {
    if (N % 2 != 0 || (N / 2) % 128 != 0) return false;
    w_tiles = (N / 2) / 128;
  } else {
    if (N % 256 != 0 || split0 % 128 != 0 || split1 % 128 != 0) return false;
    w_tiles = N / 256;
  }
  PairPlan best{};
  best.us = 1e30;
  for (int cl = 2; cl <= 4; cl += 2) {
    if (pm >= 2 && cl != pm) continue;
    const int clusters = max_clusters(cl);
    if (clusters <= 0) continue;
    for (int bt = 16; bt <= 256; bt += 16) {
      if (forced_bt >= 16 && bt != forced_bt) continue;
      for (int ksub = 1; ksub <= 2; ++ksub) {
        if (K % (64 * ksub) != 0 || pr::layout(bt, ksub, mode).stages < 3) continue;
        const double us = pair_us(M, K, w_tiles, cl, bt, ksub, clusters, mode);
        if (us < best.us) {
          best.us = us;
          best.cl = cl;
          best.bt = bt;
          best.ksub = ksub;
          best.clusters = clusters;
          best.w_tiles = w_tiles;
        }
      }
    }
  }
  if (best.cl == 0) return false;
  *out = best;
  return true;
}

// 4-D map over a [heads x 128][K] bf16 weight whose box of 64 rows is rows (i, i + 64) of one
// head for 32 consecutive i: dims {K, 2, 64, heads}, strides 64 rows, 1 row, 128 rows.
static bool encode_rope_rows(CUtensorMap* map, const void* w, int K, int heads) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeFn>(f);
  }
  if (heads <= 0 || (reinterpret_cast<uintptr_t>(w) & 15u) != 0) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(K) * 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(K), 2, 64, static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[3] = {64 * row, row, 128 * row};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(pr::BK), 2, 32, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int CL, bool ROPE>
static cudaError_t launch_pair_cl(const CUtensorMap& x, const CUtensorMap& w0, const CUtensorMap& w1,
                                  const CUtensorMap& w2, const CUtensorMap& c, pr::Params p, int clusters,
                                  cudaStream_t s) {
  static DeviceOnce configured;
  cudaError_t e = max_dynamic_smem_once(reinterpret_cast<const void*>(pr::gemm_pair_kernel<CL, ROPE>),
                                        pr::SMEM_ALLOC, configured);
  if (e != cudaSuccess) return e;
  const int n = std::min(clusters, p.units);
  launch_chain(pr::gemm_pair_kernel<CL, ROPE>, dim3(CL * n), dim3(pr::THREADS), pr::SMEM_ALLOC, s, x, w0, w1, w2, c,
               p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_pair(const PairPlan& g, const void* A, const void* B0, const void* B1, const void* B2,
                             int split0, int split1, void* C, int M, int N, int K, int ldc, int mode, int32_t* status,
                             cudaStream_t s, const QkvRope* qr) {
  if (mode == EPI_QKV_ROPE &&
      (!qr || split0 != qr->q_width || split1 != qr->q_width + qr->kvw || N != split1 + qr->kvw || qr->kvw % 128 != 0))
    return cudaErrorInvalidValue;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const bool swiglu = mode == EPI_SWIGLU;
  CUtensorMap mx, mw0, mw1, mw2, mc;
  if (!encode_tmap(&mx, BF, A, K, M, static_cast<uint64_t>(K) * 2, pr::BK, g.bt / 2, SW)) return cudaErrorInvalidValue;
  if (swiglu) {
    if (!encode_tmap(&mw0, BF, B0, K, N / 2, static_cast<uint64_t>(K) * 2, pr::BK, 64, SW) ||
        !encode_tmap(&mw1, BF, B1, K, N / 2, static_cast<uint64_t>(K) * 2, pr::BK, 64, SW))
      return cudaErrorInvalidValue;
    mw2 = mw1;
    // bf16 C [M][ldc]: 16 tokens x 64 features per store (16-byte aligned, ldc % 8 == 0)
    if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 || ldc % 8 != 0 ||
        !encode_tmap(&mc, BF, C, N / 2, M, static_cast<uint64_t>(ldc) * 2, 64, 16, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    const int r0 = split0, r1 = split1 - split0, r2 = N - split1;
    if (!encode_tmap(&mw0, BF, B0, K, r0, static_cast<uint64_t>(K) * 2, pr::BK, 64, SW)) return cudaErrorInvalidValue;
    mw1 = mw0;
    mw2 = mw0;
    if (r1 > 0 && !encode_tmap(&mw1, BF, B1, K, r1, static_cast<uint64_t>(K) * 2, pr::BK, 64, SW))
      return cudaErrorInvalidValue;
    if (r2 > 0 && !encode_tmap(&mw2, BF, B2, K, r2, static_cast<uint64_t>(K) * 2, pr::BK, 64, SW))
      return cudaErrorInvalidValue;
    if (mode == EPI_QKV_ROPE) {
      // q and k rows of a head interleaved as (i, i + 64): 4-D maps {K, 2 (i or i + 64), 64 (i),
      // heads}, 64 rows per box (a driver that refuses the layout leaves the caller the separate
      // kernels)
      if (!encode_rope_rows(&mw0, B0, K, split0 / 128) || !encode_rope_rows(&mw1, B1, K, r1 / 128))
        return cudaErrorNotSupported;
      // bf16 q_out [M][q_width]: 16 tokens x one head of 128 per store
      if ((reinterpret_cast<uintptr_t>(qr->q_out) & 15u) != 0 ||
          !encode_tmap(&mc, BF, qr->q_out, qr->q_width, M, static_cast<uint64_t>(qr->q_width) * 2, pr::ROWS, 16,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    } else if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 || ldc % 4 != 0 ||
               !encode_tmap(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M, static_cast<uint64_t>(ldc) * 4, pr::ROWS,
                            pr::F32_SLAB_TOK, CU_TENSOR_MAP_SWIZZLE_NONE)) {
      // fp32 C [M][ldc]: 8 tokens x 128 features per store (16-byte aligned, ldc % 4 == 0)
      return cudaErrorInvalidValue;
    }
  }
  const pr::Layout l = pr::layout(g.bt, g.ksub, mode);
  if (l.stages < 3) return cudaErrorInvalidValue;
  pr::Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.mode = mode;
  p.out = C;
  p.ldc = ldc;
  p.split0 = split0;
  p.split1 = split1;
  p.status = status;
  p.bt = g.bt;
  p.tok_tiles = (M + g.bt - 1) / g.bt;
  p.tok_groups = (p.tok_tiles + g.cl / 2 - 1) / (g.cl / 2);
  p.units = g.w_tiles * p.tok_groups;
  p.ksub = g.ksub;
  p.n_kb = K / (pr::BK * g.ksub);
  p.stage_bytes = l.stage_bytes;
  p.stages = l.stages;
  p.stg_off = l.stg_off;
  p.slabs = l.slabs;
  if (qr) p.qr = *qr;
  if (mode == EPI_QKV_ROPE) {
    if (g.cl == 4) return launch_pair_cl<4, true>(mx, mw0, mw1, mw2, mc, p, g.clusters, s);
    return launch_pair_cl<2, true>(mx, mw0, mw1, mw2, mc, p, g.clusters, s);
  }
  if (g.cl == 4) return launch_pair_cl<4, false>(mx, mw0, mw1, mw2, mc, p, g.clusters, s);
  return launch_pair_cl<2, false>(mx, mw0, mw1, mw2, mc, p, g.clusters, s);
}

// Process-wide: the blend's uncompacted layers take QKV, RoPE and the scatter in one launch
// (default), or the GEMM and the post-QKV kernel (tests compare the two, tuning).
static std::atomic<bool> g_qkv_fusion{true};
void set_qkv_fusion(bool enabled) { g_qkv_fusion.store(enabled); }
bool qkv_fusion() { return g_qkv_fusion.load(); }

cudaError_t launch_qkv_rope_gemm(const void* x, const void* wq, const void* wk, const void* wv, int M, int d,
                                 const QkvRope& qr, int32_t* status, const void* scratch, size_t scratch_bytes,
                                 cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  const int N = qr.q_width + 2 * qr.kvw;
  PairPlan pp;
  if (!gemm_store_pair_plan(x, wq, wk, wv, qr.q_width, qr.q_width + qr.kvw, M, N, d, scratch, scratch_bytes, &pp) ||
      pr::layout(pp.bt, pp.ksub, EPI_QKV_ROPE).stages < 3)
    return cudaErrorNotSupported;
  return launch_gemm_pair(pp, x, wq, wk, wv, qr.q_width, qr.q_width + qr.kvw, nullptr, M, N, d, N, EPI_QKV_ROPE, status,
                          s, &qr);
}
}  // namespace cb
