// Dense projections C = A . B^T of the blended prefill.
//
// bf16: a tcgen05 kernel.  One 128 x BN output tile per CTA; operands staged by TMA
// (128-byte swizzle, K-major) through a shared-memory ring guarded by
// mbarriers; one elected thread issues tcgen05.mma (kind::f16, M=128, N=BN, K=16) into a
// fp32 accumulator in tensor memory; four epilogue warps read it back with tcgen05.ld,
// apply the fused epilogue (store fp32, residual add, or SiLU(gate) * up -> bf16).  The
// fp32 epilogues stage each 32-column slab of the tile in shared memory, from where one
// thread writes it with a TMA tile store (residual add: a TMA fp32 add-reduction), so
// that global writes are whole lines instead of one 32-byte piece per row.
//   warp 0: TMA producer   warp 1: TMEM owner + MMA issuer   warps 2-5: epilogue
// The B operand may come from up to three tensors split along N (q | k | v weights), or
// from two tensors interleaved per tile (gate rows then up rows) for the SwiGLU epilogue.
// Every mbarrier wait is bounded: on timeout the kernel records ST_WAIT_TIMEOUT, lets
// its in-flight copies land, frees its tensor memory and returns.
//
// fp32: a plain shared-memory-tiled FFMA kernel with the same epilogues (used by the
// fp32 configuration, whose 1e-4 tolerance rules out TF32).
#include <algorithm>
#include <cstdio>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace cb {


// ============================================================================= tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major [rows][inner] tensor with a row pitch of `pitch` bytes.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                 uint64_t pitch, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = get_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                           uint64_t pitch, uint32_t box_inner, uint32_t box_rows,
                           CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  return encode_tmap(map, dt, base, inner, rows, pitch, box_inner, box_rows, swz);
}

bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                         uint32_t box_rows) {
  EncodeTiledFn fn = get_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


// ============================================================================= tcgen05 kernel
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                    // one 128-byte swizzle atom of bf16 along K
constexpr int A_STAGE = BM * BK * 2;      // 16 KiB
constexpr int THREADS = 192;
constexpr int MAX_CTAS = 256;             // bound of the persistent grid
constexpr int FLAG_BYTES = MAX_CTAS * 4;  // stream-K flags at the head of the scratch, partial slots after

// Work division.  Tiles t = m + n * m_tiles (consecutive tiles share a weight tile).
// Tiles [0, dp_tiles) go round-robin to the CTAs (data-parallel).  The k-iterations of the
// rest are split evenly (stream-K) over groups of sk_group CTAs: with sk_group = 1 over the
// remaining tiles; with sk_group = m_tiles (and no data-parallel tiles) over the weight
// tiles n, the CTAs of a group taking the m_tiles token tiles of the same weight tile and
// k-range at the same time, so that the weight stream is still read from DRAM once.
struct Params {
  int M, N, K;
  int mode;
  void* out;
  int ldc;
  int split0, split1;  // B columns [0,split0) from map 0, [split0,split1) map 1, rest map 2
  int32_t* status;
  int m_tiles, kb_per_tile;
  int dp_tiles, tiles;
  long long sk_iters;
  float* partials;     // [gridDim.x][128 KiB] fp32: stream-K partial tiles
  int* flags;          // [gridDim.x], zero between launches
  int bt;              // weight-rows orientation: tokens per tile (multiple of 16, <= 256)
  int stages;          // ring depth
  int stage_bytes;     // A_STAGE + slot B bytes (a multiple of 2 KiB)
  int sk_group;        // stream-K: CTAs that move through the k-iterations in lockstep
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused for this layout)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version (sm_100 family)
  d |= static_cast<uint64_t>(2) << 61;                  // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major, M = 128, N = bn.
__host__ __device__ constexpr uint32_t idesc_bf16(int bn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(bn >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

// Shared memory: barriers, the epilogue's staging buffer, then the operand ring.  A ring
// stage is slot A (128 rows x 64 bf16 = 16 KiB) followed by slot B (rows x 64 bf16); its
// depth is what fits (at most MAX_STAGES): the deeper the ring, the more weight bytes are
// in flight per SM, which is what bounds a launch whose tiles stream weights from DRAM.
constexpr int MAX_STAGES = 12;
constexpr int L2_AHEAD = 6;   // k-blocks of weights prefetched into L2 beyond the ring
constexpr int FIX_BUFS = 16;  // stream-K fix-up: slab steps in flight
constexpr int OFF_BAR = 0;
constexpr int OFF_STG = 1024;          // epilogue staging: two 16 KiB buffers
constexpr int STG_BYTES = 32768;
constexpr int OFF_RING = OFF_STG + STG_BYTES;
constexpr int SMEM_ALLOC = 232448;     // the per-block maximum (227 KiB)
constexpr int RING_BYTES = SMEM_ALLOC - 1024 - OFF_RING;  // 1 KiB of slack aligns the base

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }

enum { ITEM_FULL = 0, ITEM_PARTIAL = 1, ITEM_OWNER = 2 };

struct Item {
  int tile, kb0, kb1, kind;
  // contributors of an ITEM_OWNER tile: CTAs first, first + stride, ..., last (none when
  // first > last)
  int first, last, stride;
};

// The idx-th work item of CTA g (false when there is none).
__device__ __forceinline__ bool get_item(const Params& p, int g, int G, int idx, Item& it) {
  const int KB = p.kb_per_tile;
  const int n_dp = p.dp_tiles > g ? (p.dp_tiles - g + G - 1) / G : 0;
  if (idx < n_dp) {
    it.tile = g + idx * G;
    it.kb0 = 0;
    it.kb1 = KB;
    it.kind = ITEM_FULL;
    it.first = g + 1;
    it.last = g;
    it.stride = 1;
    return true;
  }
  if (p.sk_iters <= 0) return false;
  const int S = p.sk_group;
  const int NG = G / S, gi = g / S, mem = g - gi * S;
  if (gi >= NG) return false;
  const long long I = p.sk_iters;
  const long long a = static_cast<long long>(gi) * I / NG, b = static_cast<long long>(gi + 1) * I / NG;
  const int j = idx - n_dp;
  const long long start = j == 0 ? a : (a / KB + j) * KB;
  if (start >= b) return false;
  const long long tile_lo = (start / KB) * KB, tile_hi = tile_lo + KB;
  const long long end = b < tile_hi ? b : tile_hi;
  it.tile = p.dp_tiles + mem + static_cast<int>(start / KB) * S;
  it.kb0 = static_cast<int>(start - tile_lo);
  it.kb1 = static_cast<int>(end - tile_lo);
  it.first = g + S;
  it.last = g;
  it.stride = S;
  if (it.kb0 == 0 && it.kb1 == KB) {
    it.kind = ITEM_FULL;
  } else if (it.kb0 == 0) {
    it.kind = ITEM_OWNER;
    int gl = gi;
    while (gl + 1 < NG && static_cast<long long>(gl + 1) * I / NG < tile_hi) ++gl;
    it.last = gl * S + mem;
  } else {
    it.kind = ITEM_PARTIAL;
  }
  return true;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }


// Two tile orientations.  TOKEN_ROWS (WROWS = false): the MMA's 128 rows are tokens
// (rows of A) and its N = BN columns are output features.  WEIGHT_ROWS (WROWS = true): the
// MMA's 128 rows are output features (rows of B; for SwiGLU 64 gate rows then the 64 up
// rows of the same features) and its N = p.bt columns are tokens, so that a token count
// that is not a multiple of 128 is covered in steps of 16 and a few hundred tokens still
// yield one tile per SM.  In both, shared-memory slot A holds the MMA's rows (128 x 64 bf16)
// and slot B its columns (<= 256 x 64 bf16).
template <int BN, bool WROWS>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_bf16_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                 const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                 const __grid_constant__ CUtensorMap tmC, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* acc_full = empty + MAX_STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* fix_full = reinterpret_cast<uint64_t*>(smem + OFF_BAR + 256);  // [FIX_BUFS] stream-K fix-up slabs

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, G = gridDim.x;

  const uint32_t stages = static_cast<uint32_t>(p.stages);
  uint8_t* ring = smem + OFF_RING;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    for (int f = 0; f < FIX_BUFS; ++f) mbar_init(&fix_full[f], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (p.mode == EPI_SWIGLU || p.split0 < p.N) prefetch_tmap(&tmB1);
    if (p.mode != EPI_SWIGLU) prefetch_tmap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // (everything above touches only this CTA's shared and tensor memory: it overlaps the
  // previous kernel's tail under programmatic dependent launch)
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    uint32_t c = 0;            // k-blocks issued so far
    uint32_t s = 0, ph = 0;    // ring position of k-block c (no division in the loop)
    Item it;
    bool ok = true;
    // rows of the tile in the token dimension (TOKEN_ROWS: 128; WEIGHT_ROWS: p.bt)
    const int tok_rows = WROWS ? p.bt : BM;
    const uint32_t stage_bytes = static_cast<uint32_t>(p.stage_bytes);
    for (int idx = 0; ok && get_item(p, g, G, idx, it); ++idx) {
      const int t0 = (it.tile % p.m_tiles) * tok_rows;  // first token of the tile
      const int wt = it.tile / p.m_tiles;               // weight tile
      // weight rows: WEIGHT_ROWS takes 128 output features (SwiGLU: 64 gate + 64 up),
      // TOKEN_ROWS BN of them (SwiGLU: BN/2 + BN/2)
      const int w_rows = WROWS ? BM : BN;
      const int n0 = wt * w_rows;  // first output column (of the gate|up concatenation for SwiGLU)
      const CUtensorMap* mb = &tmB0;
      int brow = n0;
      if (p.mode != EPI_SWIGLU) {
        if (n0 >= p.split1) {
          mb = &tmB2;
          brow = n0 - p.split1;
        } else if (n0 >= p.split0) {
          mb = &tmB1;
          brow = n0 - p.split0;
        }
      }
      // When several token tiles share a weight tile, the first of them pulls the weights into
      // L2 L2_AHEAD k-blocks ahead of its ring, so that the weight tile's DRAM latency is not
      // paid once per ring's worth of stages (measured on GB300, 535 tokens: the down projection
      // 76.5 -> 68.7 us).  A weight tile with one token tile gets no prefetch: there it only
      // added copy-unit traffic (seam repair, 176 tokens: 7.49 -> 7.73 ms per blend).
      const bool lead = p.m_tiles >= 2 && (it.tile % p.m_tiles) == 0;
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        if (lane == 0) ok = mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          const int kp = kb + L2_AHEAD;
          if (lead && kp < it.kb1) {
            if (p.mode == EPI_SWIGLU) {
              tma_prefetch_l2_2d(&tmB0, kp * BK, n0 / 2);
              tma_prefetch_l2_2d(&tmB1, kp * BK, n0 / 2);
            } else {
              tma_prefetch_l2_2d(mb, kp * BK, brow);
            }
          }
          uint8_t* sa = ring + s * stage_bytes;
          uint8_t* sb = sa + A_STAGE;
          uint8_t* sw_dst = WROWS ? sa : sb;  // weights
          uint8_t* sx_dst = WROWS ? sb : sa;  // tokens
          const int w_half = WROWS ? A_STAGE / 2 : BN * BK;  // SwiGLU: where the up rows start
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          tma_load_2d(sx_dst, &tmA, &full[s], kb * BK, t0);
          if (p.mode == EPI_SWIGLU) {
            tma_load_2d(sw_dst, &tmB0, &full[s], kb * BK, n0 / 2);
            tma_load_2d(sw_dst + w_half, &tmB1, &full[s], kb * BK, n0 / 2);
          } else {
            tma_load_2d(sw_dst, mb, &full[s], kb * BK, brow);
          }
        }
        __syncwarp();
        ++c;
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      set_status(p.status, ST_WAIT_TIMEOUT);
    }
    // Let every copy this warp issued land before the block can exit: only the last
    // `stages` k-blocks can still be in flight (an earlier one's stage was reused).
    if (lane == 0) {
      for (uint32_t j = c > stages ? c - stages : 0; j < c; ++j)
        mbar_wait_bounded(&full[j % stages], (j / stages) & 1u, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16(WROWS ? p.bt : BN);
    const uint32_t ring_u32 = smem_u32(ring);
    uint32_t s = 0, ph = 0, sa = ring_u32;  // ring position and its slot-A address
    Item it;
    bool ok = true;
    for (int idx = 0; ok && get_item(p, g, G, idx, it); ++idx) {
      const int b = idx & 1;
      const uint32_t use = static_cast<uint32_t>(idx >> 1);
      if (lane == 0) ok = mbar_wait_bounded(&acc_empty[b], (use & 1u) ^ 1u, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem + static_cast<uint32_t>(b * BN);
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        if (lane == 0) ok = mbar_wait_bounded(&full[s], ph, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t da = sw128_desc(sa);
          const uint64_t db = sw128_desc(sa + A_STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes along K per step (encoded >> 4)
            tc_mma_f16(tacc, da + 2 * kk, db + 2 * kk, idesc, (kb > it.kb0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[s]);  // frees the stage once these MMAs have read it
        }
        __syncwarp();
        sa += static_cast<uint32_t>(p.stage_bytes);
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
          sa = ring_u32;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&acc_full[b]);  // accumulator b complete
      __syncwarp();
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      set_status(p.status, ST_WAIT_TIMEOUT);
    }
    // no MMA may still be running when the tensor memory is released
    if (lane == 0) {
      tc_commit(drain);
      mbar_wait_bounded(drain, 0u, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
    const int r_loc = quarter * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..127 within the epilogue warps
    volatile int* go = abort_flag + 1;   // [2]: per-item decision, written by et == 0
    int slab_par = 0;                    // staging slabs issued (double buffer parity)
    // Stream-K partial slot of CTA `slot` (128 KiB), written straight from registers in a
    // layout where each warp store covers 512 contiguous bytes: token rows as 32-column
    // chunks [chunk][8 float4 groups][128 rows], weight rows as 16-token chunks
    // [chunk][4 float4 groups][128 features].  A chunk (16 / 8 KiB) is contiguous, so the
    // owner fetches it with one bulk copy.
    auto write_slot = [&](uint32_t tb, int slot) {
      float4* base = reinterpret_cast<float4*>(p.partials + static_cast<size_t>(slot) * (BM * 256));
      if (WROWS) {
#pragma unroll 1
        for (int c = 0; c < p.bt; c += 16) {
          float v[16];
          tmem_ld16(tb + c, v);
          float4* dst = base + static_cast<size_t>(c / 16) * 4 * BM + r_loc;
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q * BM] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(tb + c, v);
          float4* dst = base + static_cast<size_t>(c / 32) * 8 * BM + r_loc;
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q * BM] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
    };
    // The owner's fix-up.  An owner item is the last item of its CTA, so the operand ring is
    // idle: the contributors' partial slots come in through TMA, a column slab at a time,
    // as many steps ahead as the ring holds (up to FIX_BUFS), and are added, in contributor
    // order, to the owner's accumulator read from tensor memory; then the tile goes out as
    // in the whole-tile epilogue.
    auto owner_fixup = [&](const Item& it, uint32_t tb, int first, int last, int stride) {
      const int nc = (last - first) / stride + 1;
      const bool swig = p.mode == EPI_SWIGLU;
      // token rows: 32-column chunks of 128 rows (16 KiB); weight rows: 16-token chunks of
      // 128 features (8 KiB); SwiGLU token rows take the gate and the up chunk together
      const int slab = WROWS ? 16 * BM * 4 : BM * 32 * 4;
      const int per = nc * ((swig && !WROWS) ? 2 : 1);
      const int ring_bytes = p.stages * p.stage_bytes;
      const int steps = WROWS ? (min(p.bt, p.M - (it.tile % p.m_tiles) * p.bt) + 15) / 16 : (swig ? BN / 2 : BN) / 32;
      const int depth = min(min(steps, FIX_BUFS), ring_bytes / (per * slab));
      if (depth < 1) {  // the planner keeps contributors below this (uniform)
        if (et == 0) set_status(p.status, ST_RANGE);
        return;
      }
      auto issue = [&](int k, int buf) {
        if (et != 0) return;
        uint8_t* dst = ring + static_cast<size_t>(buf) * per * slab;
        mbar_arrive_expect_tx(&fix_full[buf], static_cast<uint32_t>(per * slab));
        int n = 0;
        for (int q = first; q <= last; q += stride) {
          const uint8_t* src = reinterpret_cast<const uint8_t*>(p.partials + static_cast<size_t>(q) * (BM * 256));
          bulk_load(dst + (n++) * slab, src + static_cast<size_t>(k) * slab, slab, &fix_full[buf]);
          if (!WROWS && swig)
            bulk_load(dst + (n++) * slab, src + static_cast<size_t>(k + BN / 64) * slab, slab, &fix_full[buf]);
        }
      };
      if (et == 0) fence_proxy_async_global();
      for (int k = 0; k < depth; ++k) issue(k, k);
      const int sw = r_loc & 7;
      for (int k = 0; k < steps; ++k) {
        const int buf = k % depth;
        mbar_wait_bounded(&fix_full[buf], static_cast<uint32_t>((k / depth) & 1), abort_flag);
        const uint8_t* src = ring + static_cast<size_t>(buf) * per * slab;
        if (WROWS) {
          const int t0 = (it.tile % p.m_tiles) * p.bt, nt = min(p.bt, p.M - t0), wt = it.tile / p.m_tiles;
          const int c = k * 16;
          float v[16];
          tmem_ld16(tb + c, v);
          for (int n = 0; n < nc; ++n) {
            const float4* sl = reinterpret_cast<const float4*>(src + n * slab) + r_loc;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 y = sl[q * BM];
              v[4 * q] += y.x;
              v[4 * q + 1] += y.y;
              v[4 * q + 2] += y.z;
              v[4 * q + 3] += y.w;
            }
          }
          if (swig) {
            float* xch = reinterpret_cast<float*>(smem + OFF_STG);  // [64][17]
            if (quarter >= 2) {
#pragma unroll
              for (int j = 0; j < 16; ++j) xch[(r_loc - 64) * 17 + j] = v[j];
            }
            epi_bar();
            if (quarter < 2) {
              bf16* dst = static_cast<bf16*>(p.out) + static_cast<size_t>(t0 + c) * p.ldc + wt * (BM / 2) + r_loc;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c + j < nt)
                  dst[static_cast<size_t>(j) * p.ldc] = __float2bfloat16_rn(silu_f(v[j]) * xch[r_loc * 17 + j]);
            }
          } else {
            float* sbuf = reinterpret_cast<float*>(smem + OFF_STG) + (slab_par & 1) * (16 * BM);
            if (et == 0) bulk_wait_read_all_but_1();
            epi_bar();
#pragma unroll
            for (int j = 0; j < 16; ++j) sbuf[j * BM + r_loc] = v[j];
            fence_proxy_async_smem();
            epi_bar();
            if (et == 0) {
              if (p.mode == EPI_ADD_F32)
                tma_reduce_add_2d(&tmC, sbuf, wt * BM, t0 + c);
              else
                tma_store_2d(&tmC, sbuf, wt * BM, t0 + c);
              bulk_commit();
            }
            ++slab_par;
          }
        } else {
          const int m0 = (it.tile % p.m_tiles) * BM, n0 = (it.tile / p.m_tiles) * BN;
          const int c = k * 32;
          float v[32];
          tmem_ld32(tb + c, v);
          auto add_slab = [&](float* x, const uint8_t* sl) {
            const float4* row = reinterpret_cast<const float4*>(sl) + r_loc;
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
              const float4 y = row[q8 * BM];
              x[4 * q8] += y.x;
              x[4 * q8 + 1] += y.y;
              x[4 * q8 + 2] += y.z;
              x[4 * q8 + 3] += y.w;
            }
          };
          if (swig) {
            float u[32];
            tmem_ld32(tb + BN / 2 + c, u);
            for (int n = 0; n < nc; ++n) {
              add_slab(v, src + (2 * n) * slab);
              add_slab(u, src + (2 * n + 1) * slab);
            }
            const int row = m0 + r_loc;
            if (row < p.M) {
              bf16* dst = static_cast<bf16*>(p.out) + static_cast<size_t>(row) * p.ldc + n0 / 2 + c;
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = silu_f(v[j + e]) * u[j + e];
                store8(dst + j, f);
              }
            }
          } else {
            for (int n = 0; n < nc; ++n) add_slab(v, src + n * slab);
            uint8_t* stg = smem + OFF_STG + (slab_par & 1) * 16384;
            ++slab_par;
            uint8_t* srow = stg + r_loc * 128;
            if (et == 0) bulk_wait_read_all_but_1();
            epi_bar();
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8)
              *reinterpret_cast<float4*>(srow + ((q8 ^ sw) << 4)) =
                  make_float4(v[4 * q8], v[4 * q8 + 1], v[4 * q8 + 2], v[4 * q8 + 3]);
            fence_proxy_async_smem();
            epi_bar();
            if (et == 0) {
              if (p.mode == EPI_ADD_F32)
                tma_reduce_add_2d(&tmC, stg, n0 + c, m0);
              else
                tma_store_2d(&tmC, stg, n0 + c, m0);
              bulk_commit();
            }
          }
        }
        epi_bar();  // every thread is done with this step's slabs before they are refilled
        if (k + depth < steps) issue(k + depth, buf);
      }
    };
    Item it;
    for (int idx = 0; get_item(p, g, G, idx, it); ++idx) {
      const int b = idx & 1;
      const uint32_t use = static_cast<uint32_t>(idx >> 1);
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(&acc_full[b], use & 1u, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok && lane == 0) {
        *abort_flag = 1;
        set_status(p.status, ST_WAIT_TIMEOUT);
      }
      // one decision for all four epilogue warps, so that every named barrier below is
      // reached by all of them: failures are recorded before the first barrier, read by
      // one thread between the two, and the slot of item idx is rewritten at idx + 2 only
      epi_bar();
      if (et == 0) go[b] = !*abort_flag;
      epi_bar();
      if (!go[b]) break;
      tc_fence_after();
      const int m0 = (it.tile % p.m_tiles) * BM;
      const int n0 = (it.tile / p.m_tiles) * BN;
      const int row = m0 + r_loc;
      const uint32_t tbase = tmem + static_cast<uint32_t>(b * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      if (it.kind != ITEM_FULL) {
        // Stream-K: this CTA's accumulator -> its partial slot; the owner of the tile adds
        // the slots to its own accumulator in a fixed order.
        if (it.kind == ITEM_PARTIAL) {
          write_slot(tbase, g);
          __threadfence();  // every thread's slot stores before the flag
          epi_bar();
          if (et == 0) atomicExch(&p.flags[g], 1);
        } else {
          const int first = it.first, last = it.last, stride = it.stride;
          if (et == 0) {  // the later contributors, in order (bounded)
            for (int q = first; q <= last; q += stride) {
              const uint64_t t0 = global_ns();
              while (atomicAdd(&p.flags[q], 0) == 0) {
                if (global_ns() - t0 > 2000000000ull || *abort_flag) {
                  set_status(p.status, ST_WAIT_TIMEOUT);
                  break;
                }
              }
            }
            __threadfence();
          }
          epi_bar();
          owner_fixup(it, tbase, first, last, stride);
          if (et == 0)
            for (int q = first; q <= last; q += stride) atomicExch(&p.flags[q], 0);
        }
      } else {
        if (WROWS) {
          // lanes = output features, columns = the tile's tokens t0 .. t0 + nt - 1
          const int t0 = (it.tile % p.m_tiles) * p.bt;
          const int nt = min(p.bt, p.M - t0);
          const int wt = it.tile / p.m_tiles;
          if (p.mode == EPI_SWIGLU) {
            // lanes 0-63 hold the gate and lanes 64-127 the up projection of features
            // f0 .. f0 + 63: the up warps pass their values through shared memory
            float* xch = reinterpret_cast<float*>(smem + OFF_STG);  // [64][17]
            const int f0 = wt * (BM / 2);
            bf16* out = static_cast<bf16*>(p.out);
#pragma unroll 1
            for (int c = 0; c < nt; c += 16) {
              float v[16];
              tmem_ld16(tbase + c, v);
              if (quarter >= 2) {
#pragma unroll
                for (int j = 0; j < 16; ++j) xch[(r_loc - 64) * 17 + j] = v[j];
              }
              epi_bar();
              if (quarter < 2) {
                bf16* dst = out + static_cast<size_t>(t0 + c) * p.ldc + f0 + r_loc;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (c + j < nt)
                    dst[static_cast<size_t>(j) * p.ldc] = __float2bfloat16_rn(silu_f(v[j]) * xch[r_loc * 17 + j]);
              }
              epi_bar();
            }
          } else {
            // 16-token x 128-feature fp32 slabs, double-buffered, one TMA store (or
            // add-reduction) each
            const int f0 = wt * BM;
            float* stg = reinterpret_cast<float*>(smem + OFF_STG);
#pragma unroll 1
            for (int c = 0; c < nt; c += 16, ++slab_par) {
              float v[16];
              tmem_ld16(tbase + c, v);
              float* sbuf = stg + (slab_par & 1) * (16 * BM);
              if (et == 0) bulk_wait_read_all_but_1();  // the store from this buffer two slabs ago
              epi_bar();
#pragma unroll
              for (int j = 0; j < 16; ++j) sbuf[j * BM + r_loc] = v[j];
              fence_proxy_async_smem();
              epi_bar();
              if (et == 0) {
                if (p.mode == EPI_ADD_F32)
                  tma_reduce_add_2d(&tmC, sbuf, f0, t0 + c);
                else
                  tma_store_2d(&tmC, sbuf, f0, t0 + c);
                bulk_commit();
              }
            }
          }
        } else if (p.mode != EPI_SWIGLU) {
          // stage a 128-row x 32-column slab in shared memory (128-byte swizzle: 16-byte
          // chunk q of row r at chunk q ^ (r & 7), conflict-free), then one thread stores
          // it; two staging buffers, each reused once its previous store has read it
          const int sw = r_loc & 7;
#pragma unroll 1
          for (int c = 0; c < BN; c += 32, ++slab_par) {
            float v[32];
            tmem_ld32(tbase + c, v);
            uint8_t* stg = smem + OFF_STG + (slab_par & 1) * 16384;
            uint8_t* srow = stg + r_loc * 128;
            if (et == 0) bulk_wait_read_all_but_1();
            epi_bar();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4*>(srow + ((q ^ sw) << 4)) =
                  make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            fence_proxy_async_smem();
            epi_bar();
            if (et == 0) {
              if (p.mode == EPI_ADD_F32)
                tma_reduce_add_2d(&tmC, stg, n0 + c, m0);
              else
                tma_store_2d(&tmC, stg, n0 + c, m0);
              bulk_commit();
            }
          }
        } else {  // EPI_SWIGLU, direct stores
          bf16* out = static_cast<bf16*>(p.out);
#pragma unroll 1
          for (int c = 0; c < BN / 2; c += 32) {
            float gv[32], uv[32];
            tmem_ld32(tbase + c, gv);
            tmem_ld32(tbase + BN / 2 + c, uv);
            if (row < p.M) {
              bf16* dst = out + static_cast<size_t>(row) * p.ldc + n0 / 2 + c;
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = silu_f(gv[j + e]) * uv[j + e];
                store8(dst + j, f);
              }
            }
          }
        }
      }
      // accumulator b may be overwritten once every epilogue warp has read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
    if (et == 0) bulk_wait_all();  // the tile stores have completed before the grid does
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
}

}  // namespace tc

// ============================================================================= fp32 SIMT kernel
namespace simt {

constexpr int TM = 64, TN = 64, TK = 16;

template <bool SWIGLU>
__global__ void __launch_bounds__(256) gemm_f32(const float* __restrict__ A, const float* __restrict__ B0,
                                                const float* __restrict__ B1, const float* __restrict__ B2,
                                                int split0, int split1, float* __restrict__ C, int M, int N, int K,
                                                int ldc, int mode) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  __shared__ float Us[SWIGLU ? TK : 1][TN + 4];
  const int m0 = blockIdx.x * TM, n0 = blockIdx.y * TN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {}, accu[4][4] = {};
  const int Nb = SWIGLU ? N : N;  // output columns (gate/up rows) of this call
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      const int r = i / TK, kk = i % TK;
      const int gm = m0 + r, gk = k0 + kk;
      As[kk][r] = (gm < M && gk < K) ? A[static_cast<size_t>(gm) * K + gk] : 0.f;
      const int gn = n0 + r;
      // B row gn: from B0 (gate when SWIGLU), or split across B0 | B1 | B2 along N
      const float* brow = nullptr;
      if (gn < Nb && gk < K) {
        if (SWIGLU || gn < split0)
          brow = B0 + static_cast<size_t>(gn) * K;
        else if (gn < split1)
          brow = B1 + static_cast<size_t>(gn - split0) * K;
        else
          brow = B2 + static_cast<size_t>(gn - split1) * K;
      }
      Bs[kk][r] = brow ? brow[gk] : 0.f;
      if (SWIGLU) Us[kk][r] = brow ? B1[static_cast<size_t>(gn) * K + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4], u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
        if (SWIGLU) u[i] = Us[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (SWIGLU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= Nb) continue;
      float* dst = C + static_cast<size_t>(gm) * ldc + gn;
      if (SWIGLU) {
        const float g = acc[i][j];
        *dst = g / (1.0f + expf(-g)) * accu[i][j];
      } else if (mode == EPI_ADD_F32) {
        *dst += acc[i][j];
      } else {
        *dst = acc[i][j];
      }
    }
  }
}

}  // namespace simt

// ============================================================================= launcher
static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  }
  return n;
}

// Scratch that lets every shape use its preferred schedule: the flags plus one 128 KiB
// fp32 partial slot per SM.
size_t gemm_scratch_bytes() {
  return tc::FLAG_BYTES + static_cast<size_t>(std::min(sm_count(), tc::MAX_CTAS)) * tc::BM * 256 * sizeof(float);
}

// 0: time model; 1: token rows; 2: weight rows with the model's token tile; 16..256
// (multiple of 16): weight rows with that token tile.
static std::atomic<int> g_orientation{0};
void gemm_set_orientation(int o) { g_orientation.store(o); }

// Schedule of one bf16 GEMM.
struct GemmPlan {
  bool wrows;     // weight-rows orientation
  int bn;         // token-rows: output features per tile (256 or 128)
  int bt;         // weight-rows: tokens per tile
  int tok_tiles;  // tiles along the tokens
  int tiles;
  int grid;
  int dp_tiles;
  long long sk_iters;
  int sk_group;         // CTAs per stream-K group (1: plain stream-K)
  size_t scratch_used;  // bytes of scratch the stream-K split touches (0: data-parallel)
  double us;            // the time model's estimate
};

// Time model used to pick the orientation, the token tile and the schedule.  A tile takes
// K/64 k-blocks.  Measured on GB300 (one CTA per SM, this kernel): a k-block takes ~0.31 us
// for any N below 256 and 0.336 us at N = 256.  The MMAs alone would take 128 cycles per
// N = 256 instruction and proportionally less for narrower ones; what sets the k-block time
// here is the stage landing in time and the shared-memory bandwidth that the copies and the
// MMA operand reads share, so narrow tiles buy little.  A k-block therefore costs about
// max(0.336 * N / 256, 0.31) us (with a slight
// slope below the floor, so that of two plans with as many waves the one spreading the
// tokens over more SMs wins), and the choice is about padding and filling the SMs.
// Data-parallel: tiles go round-robin over at most one CTA per SM, ceil(tiles / SMs) tile
// times.  Stream-K (when the tiles fill at most half of the SMs): the k-blocks of all tiles
// are divided evenly over up to 8 CTAs per tile, and every token tile of a weight tile
// then streams that weight tile from DRAM on its own (6.5 TB/s).  Token rows pad the
// tokens to a multiple of 128; weight rows pad them to a multiple of 16 per tile.
static double kblock_us(int n_cols) { return std::max(0.336 * n_cols / 256.0, 0.31 + 0.02 * n_cols / 256.0); }

struct Sched {
  int grid, dp_tiles, sk_group;
  long long sk_iters;
  size_t scratch;
  double us;
};

// tiles = tok_tiles x w_tiles, each of kb k-blocks; weight_bytes read once per token tile
// under stream-K.
static Sched schedule(int tok_tiles, int w_tiles, int kb, double kb_us, double weight_bytes, int sms,
                      long long slots) {
  Sched r{};
  const int tiles = tok_tiles * w_tiles;
  r.grid = std::min(sms, tiles);
  r.dp_tiles = tiles;
  r.sk_group = 1;
  r.sk_iters = 0;
  r.scratch = 0;
  r.us = ((tiles + sms - 1) / sms) * kb * kb_us;
  if (2 * tiles <= sms) {
    const long long iters = static_cast<long long>(tiles) * kb;
    // at most ~4 CTAs share one tile, one partial slot per CTA, at least 8 k-blocks each
    const int g_sk = static_cast<int>(std::min<long long>(std::min(sms, 4 * tiles), slots));
    if (g_sk >= 2 * tiles && iters >= 8LL * g_sk) {
      r.grid = g_sk;
      r.dp_tiles = 0;
      r.sk_iters = iters;
      r.scratch = tc::FLAG_BYTES + static_cast<size_t>(g_sk) * tc::BM * 256 * sizeof(float);
      // (+0.5 us per extra token tile: their CTAs no longer share the weight stream)
      r.us = std::max(((iters + g_sk - 1) / g_sk) * kb_us, weight_bytes * tok_tiles / 6.5e6) + 0.5 * (tok_tiles - 1);
    }
  }
  // Grouped stream-K: groups of tok_tiles CTAs divide the (weight tile, k-block) iterations
  // evenly; the members of a group take the token tiles of the same weight tile and k-range
  // together, so weights are still streamed once, and every SM gets the same number of
  // k-blocks (a few hundred tokens otherwise leave SMs idle or a wave ragged).  At most 4
  // groups share one weight tile; +8 us for writing and summing the split tiles (measured
  // on GB300 with one owner per tile: ~3 us to write a partial, ~6 us for the owner's
  // eight 32-column steps), so it only pays off on long k ranges.
  if (tok_tiles >= 2) {
    const long long iters = static_cast<long long>(w_tiles) * kb;
    const int ng = static_cast<int>(
        std::min<long long>(std::min<long long>(sms / tok_tiles, slots / tok_tiles), 4LL * w_tiles));
    if (ng >= 2 && iters >= 8LL * ng) {
      const double us = ((iters + ng - 1) / ng) * kb_us + 8.0;
      if (us < 0.9 * r.us) {
        r.grid = ng * tok_tiles;
        r.dp_tiles = 0;
        r.sk_group = tok_tiles;
        r.sk_iters = iters;
        r.scratch = tc::FLAG_BYTES + static_cast<size_t>(r.grid) * tc::BM * 256 * sizeof(float);
        r.us = us;
      }
    }
  }
  return r;
}

static GemmPlan plan_gemm(int M, int N, int K, int split0, int split1, long long slots) {
  const int sms = std::min(sm_count(), tc::MAX_CTAS);
  const int kb = K / tc::BK;
  const double wbytes = 2.0 * N * K;
  GemmPlan g{};
  g.bn = (N % 256 == 0 && split0 % 256 == 0 && split1 % 256 == 0) ? 256 : 128;
  const int mt = (M + tc::BM - 1) / tc::BM;
  const Sched st = schedule(mt, N / g.bn, kb, kblock_us(g.bn), wbytes, sms, slots);
  const int nw = N / tc::BM;
  const int forced = g_orientation.load();
  const bool w_ok = split0 % tc::BM == 0 && split1 % tc::BM == 0;
  Sched sw{};
  int best_bt = 0;
  if (w_ok) {
    for (int t = (M + 255) / 256; t <= M; ++t) {
      const int bt = ((M + t - 1) / t + 15) / 16 * 16;
      if (bt > 256) continue;
      if (forced >= 16 && bt != forced) {
        if (bt <= 16) break;
        continue;
      }
      const Sched c = schedule((M + bt - 1) / bt, nw, kb, kblock_us(bt), wbytes, sms,
                               slots);
      if (best_bt == 0 || c.us < sw.us) {
        sw = c;
        best_bt = bt;
      }
      if (bt <= 16) break;
    }
    if (forced >= 16 && best_bt == 0) {  // a forced tile the enumeration did not produce
      best_bt = forced;
      sw = schedule((M + forced - 1) / forced, nw, kb, kblock_us(forced), wbytes,
                    sms, slots);
    }
  }
  g.wrows = best_bt > 0 && (forced >= 2 || (forced == 0 && sw.us < st.us));
  const Sched& c = g.wrows ? sw : st;
  g.bt = g.wrows ? best_bt : 0;
  g.tok_tiles = g.wrows ? (M + g.bt - 1) / g.bt : mt;
  g.tiles = g.tok_tiles * (g.wrows ? nw : N / g.bn);
  g.grid = c.grid;
  g.dp_tiles = c.dp_tiles;
  g.sk_iters = c.sk_iters;
  g.sk_group = c.sk_group;
  g.scratch_used = c.scratch;
  g.us = c.us;
  return g;
}

template <int BN, bool WROWS>
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& b2,
                             const CUtensorMap& c, tc::Params p, const GemmPlan& g, void* scratch, cudaStream_t s) {
  static DeviceOnce configured;
  cudaError_t e = max_dynamic_smem_once(reinterpret_cast<const void*>(tc::gemm_bf16_tc<BN, WROWS>), tc::SMEM_ALLOC,
                                        configured);
  if (e != cudaSuccess) return e;
  p.m_tiles = g.tok_tiles;
  p.kb_per_tile = p.K / tc::BK;
  p.tiles = g.tiles;
  p.dp_tiles = g.dp_tiles;
  p.sk_iters = g.sk_iters;
  p.sk_group = g.sk_group;
  p.bt = g.bt;
  p.stage_bytes = tc::A_STAGE + (WROWS ? g.bt : BN) * tc::BK * 2;
  p.stages = std::min(tc::MAX_STAGES, tc::RING_BYTES / p.stage_bytes);
  p.flags = scratch ? static_cast<int*>(scratch) : nullptr;
  p.partials = scratch ? reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + tc::FLAG_BYTES) : nullptr;
  // request only what the ring uses (+1 KiB to align the base)
  const int smem = tc::OFF_RING + p.stages * p.stage_bytes + 1024;
  launch_chain(tc::gemm_bf16_tc<BN, WROWS>, dim3(g.grid), dim3(tc::THREADS), smem, s, a, b0, b1, b2, c, p);
  return cudaGetLastError();
}

// Stream-K partial slots that scratch_bytes of scratch holds (after the flags).
static long long scratch_slots(const void* scratch, size_t scratch_bytes) {
  const size_t slot_bytes = static_cast<size_t>(tc::BM) * 256 * sizeof(float);
  return scratch && scratch_bytes > static_cast<size_t>(tc::FLAG_BYTES)
             ? static_cast<long long>((scratch_bytes - tc::FLAG_BYTES) / slot_bytes)
             : 0;
}

// Whether launch_gemm runs these operands on CTA pairs (the paired kernel takes no scratch):
// forced by the pairing hook, else when the time model prefers it and no orientation is forced.
static bool use_pair(const GemmPlan& g, int M, int N, int K, int split0, int split1, int mode, PairPlan* pp) {
  const int pm = gemm_pairing();
  const int forced = g_orientation.load();
  if (pm == 1 || (pm == 0 && forced != 0)) return false;
  if (!plan_gemm_pair(M, N, K, split0, split1, mode, forced >= 16 ? forced : 0, pp)) return false;
  // The single-CTA model is optimistic: measured launches take ~1.2x its estimate plus a
  // fixed ~8 us that it leaves out (GB300, CUDA events, 40 projection shapes of the blends from
  // 535 to 3536 rows: with this rule the faster kernel is taken at all but one, 2.4 % apart)
  return pm >= 2 || pp->us < 1.2 * g.us + 8.0;
}

// The paired plan launch_gemm takes for this bf16 store-mode GEMM (false when it would run the
// GEMV or the single-CTA kernel).
bool gemm_store_pair_plan(const void* A, const void* B0, const void* B1, const void* B2, int split0, int split1, int M,
                          int N, int K, const void* scratch, size_t scratch_bytes, PairPlan* pp) {
  if (M <= 0 || gemv_applies(M, K, CB_BF16, A, B0, B1, B2)) return false;
  const GemmPlan g = plan_gemm(M, N, K, split0, split1, scratch_slots(scratch, scratch_bytes));
  return use_pair(g, M, N, K, split0, split1, EPI_STORE_F32, pp);
}

// Scratch bytes the schedule of launch_gemm would use for a single-tensor B of N output
// columns with unlimited scratch (0 when the shape runs data-parallel).
size_t gemm_scratch_needed(int N, int M, int K, cb_dtype dt) {
  if (dt != CB_BF16 || M <= 0) return 0;
  return plan_gemm(M, N, K, N, N, 1LL << 40).scratch_used;
}

// Scratch bytes launch_gemm uses for these operands when it is given scratch_bytes of
// scratch: 0 on the paths that take none (no rows, the few-row GEMV, fp32), otherwise
// what the schedule narrowed to the slots that scratch holds uses (never more than it).
size_t gemm_scratch_used(const void* A, const void* B0, const void* B1, const void* B2, int split0, int split1, int M,
                         int N, int K, int mode, cb_dtype dt, size_t scratch_bytes) {
  if (M <= 0 || dt != CB_BF16 || gemv_applies(M, K, dt, A, B0, B1, B2)) return 0;
  const long long slots = scratch_slots(reinterpret_cast<const void*>(1), scratch_bytes);
  const GemmPlan g = plan_gemm(M, N, K, split0, split1, slots);
  PairPlan pp;
  if (use_pair(g, M, N, K, split0, split1, mode, &pp)) return 0;
  return g.scratch_used;
}

// The schedule launch_gemm picks for a bf16 GEMM with scratch_bytes of scratch, as text.
int gemm_describe(int M, int N, int K, int mode, size_t scratch_bytes, char* buf, size_t len) {
  if (M <= 0 || N <= 0 || K <= 0) return snprintf(buf, len, "empty");
  const long long slots = scratch_slots(reinterpret_cast<const void*>(1), scratch_bytes);
  const GemmPlan g = plan_gemm(M, N, K, N, N, slots);
  PairPlan pp;
  if (use_pair(g, M, N, K, N, N, mode, &pp)) {
    const int stage_bytes = pp.ksub * (16384 + pp.bt * 64);
    return snprintf(buf, len, "pairs cluster=%d token_tile=%d k_atoms_per_stage=%d stage_bytes=%d clusters=%d model_us=%.1f",
                    pp.cl, pp.bt, pp.ksub, stage_bytes, pp.clusters, pp.us);
  }
  return snprintf(buf, len,
                  "single orientation=%s token_tile=%d feature_tile=%d grid=%d data_parallel_tiles=%d stream_k_iters=%lld "
                  "stream_k_group=%d model_us=%.1f",
                  g.wrows ? "weight-rows" : "token-rows", g.wrows ? g.bt : 128, g.wrows ? 128 : g.bn, g.grid, g.dp_tiles,
                  g.sk_iters, g.sk_group, g.us);
}

// mode: EPI_STORE_F32 / EPI_ADD_F32 (C fp32 [M][ldc]) or EPI_SWIGLU (C dtype [M][ldc], N/2 columns).
// B0/B1/B2: weight tensors [rows][K]; for STORE/ADD the output columns [0,split0) come from
// B0, [split0,split1) from B1 and [split1,N) from B2; for SWIGLU B0 = gate, B1 = up, each
// [N/2][K].  scratch (may be null: data-parallel only) holds stream-K partial tiles and
// flags; its flags must be zero before the first use and are left zero.
cudaError_t launch_gemm(const void* A, const void* B0, const void* B1, const void* B2, int split0, int split1, void* C,
                        int M, int N, int K, int ldc, int mode, cb_dtype dt, int32_t* status, void* scratch,
                        size_t scratch_bytes, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (gemv_applies(M, K, dt, A, B0, B1, B2))
    return launch_gemv(A, B0, B1, B2, split0, split1, C, M, N, K, ldc, mode, dt, s);
  if (dt == CB_F32) {
    if (mode == EPI_SWIGLU) {
      dim3 grid((M + simt::TM - 1) / simt::TM, (N / 2 + simt::TN - 1) / simt::TN);
      simt::gemm_f32<true><<<grid, 256, 0, s>>>(static_cast<const float*>(A), static_cast<const float*>(B0),
                                                static_cast<const float*>(B1), nullptr, 0, 0, static_cast<float*>(C), M,
                                                N / 2, K, ldc, mode);
    } else {
      dim3 grid((M + simt::TM - 1) / simt::TM, (N + simt::TN - 1) / simt::TN);
      simt::gemm_f32<false><<<grid, 256, 0, s>>>(static_cast<const float*>(A), static_cast<const float*>(B0),
                                                 static_cast<const float*>(B1), static_cast<const float*>(B2), split0,
                                                 split1, static_cast<float*>(C), M, N, K, ldc, mode);
    }
    return cudaGetLastError();
  }
  // bf16 on tcgen05
  const long long slots = scratch_slots(scratch, scratch_bytes);
  const GemmPlan g = plan_gemm(M, N, K, split0, split1, slots);
  PairPlan pp;
  if (use_pair(g, M, N, K, split0, split1, mode, &pp))
    return launch_gemm_pair(pp, A, B0, B1, B2, split0, split1, C, M, N, K, ldc, mode, status, s);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  // token rows: A box 128 rows, weight box BN rows (SwiGLU BN/2 + BN/2);
  // weight rows: A box bt rows, weight box 128 rows (SwiGLU 64 + 64)
  const uint32_t a_rows = g.wrows ? static_cast<uint32_t>(g.bt) : static_cast<uint32_t>(tc::BM);
  const uint32_t w_rows = g.wrows ? static_cast<uint32_t>(tc::BM) : static_cast<uint32_t>(g.bn);
  CUtensorMap ma, mb0, mb1, mb2;
  if (!encode_tmap_2d(&ma, BF, A, K, M, static_cast<uint64_t>(K) * 2, tc::BK, a_rows, SW)) return cudaErrorInvalidValue;
  if (mode == EPI_SWIGLU) {
    if (!encode_tmap_2d(&mb0, BF, B0, K, N / 2, static_cast<uint64_t>(K) * 2, tc::BK, w_rows / 2, SW))
      return cudaErrorInvalidValue;
    if (!encode_tmap_2d(&mb1, BF, B1, K, N / 2, static_cast<uint64_t>(K) * 2, tc::BK, w_rows / 2, SW))
      return cudaErrorInvalidValue;
    mb2 = mb1;
  } else {
    const int r0 = split0, r1 = split1 - split0, r2 = N - split1;
    if (!encode_tmap_2d(&mb0, BF, B0, K, r0, static_cast<uint64_t>(K) * 2, tc::BK, w_rows, SW))
      return cudaErrorInvalidValue;
    mb1 = mb0;
    mb2 = mb0;
    if (r1 > 0 && !encode_tmap_2d(&mb1, BF, B1, K, r1, static_cast<uint64_t>(K) * 2, tc::BK, w_rows, SW))
      return cudaErrorInvalidValue;
    if (r2 > 0 && !encode_tmap_2d(&mb2, BF, B2, K, r2, static_cast<uint64_t>(K) * 2, tc::BK, w_rows, SW))
      return cudaErrorInvalidValue;
  }
  // fp32 output tensor map: token rows store 128 tokens x 32 features (128-byte swizzle),
  // weight rows 16 tokens x 128 features.  SwiGLU keeps direct stores: in token rows its
  // CTAs run several tiles, so the epilogue overlaps the next tile's main loop, and it
  // measured slower with TMA stores sharing the copy unit with the loads.
  // (fp32 C: 16-byte aligned, ldc % 4 == 0)
  CUtensorMap mc = ma;
  if (mode != EPI_SWIGLU &&
      ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 || ldc % 4 != 0 ||
       !encode_tmap_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M, static_cast<uint64_t>(ldc) * 4,
                       g.wrows ? tc::BM : 32, g.wrows ? 16 : tc::BM, g.wrows ? CU_TENSOR_MAP_SWIZZLE_NONE : SW)))
    return cudaErrorInvalidValue;
  tc::Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.mode = mode;
  p.out = C;
  p.ldc = ldc;
  p.split0 = split0;
  p.split1 = split1;
  p.status = status;
  if (g.wrows) return launch_tc<256, true>(ma, mb0, mb1, mb2, mc, p, g, scratch, s);
  if (g.bn == 256) return launch_tc<256, false>(ma, mb0, mb1, mb2, mc, p, g, scratch, s);
  return launch_tc<128, false>(ma, mb0, mb1, mb2, mc, p, g, scratch, s);
}

}  // namespace cb
