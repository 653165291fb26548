// Dense projections C = A . B^T of the blended prefill.
//
// bf16: a tcgen05 kernel.  One 128 x BN output tile per CTA; operands staged by TMA
// (128-byte swizzle, K-major) through a STAGES-deep shared-memory ring guarded by
// mbarriers; one elected thread issues tcgen05.mma (kind::f16, M=128, N=BN, K=16) into a
// fp32 accumulator in tensor memory; four epilogue warps read it back with tcgen05.ld and
// apply the fused epilogue (store fp32, residual add, or SiLU(gate) * up -> bf16).
//   warp 0: TMA producer   warp 1: TMEM owner + MMA issuer   warps 2-5: epilogue
// The B operand may come from up to three tensors split along N (q | k | v weights), or
// from two tensors interleaved per tile (gate rows then up rows) for the SwiGLU epilogue.
// Every mbarrier wait is bounded: on timeout the kernel records ST_WAIT_TIMEOUT, lets
// its in-flight copies land, frees its tensor memory and returns.
//
// fp32: a plain shared-memory-tiled FFMA kernel with the same epilogues (used by the
// fp32 configuration, whose 1e-4 tolerance rules out TF32).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace cb {

enum { EPI_STORE_F32 = 0, EPI_ADD_F32 = 1, EPI_SWIGLU = 2 };

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
// Tiles [0, dp_tiles) go round-robin to the CTAs (data-parallel); the k-iterations of the
// remaining tiles are split evenly over the CTAs (stream-K): CTA g owns iterations
// [g*I/G, (g+1)*I/G) of the I = (tiles - dp_tiles) * kb_per_tile tail iterations.
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
  float* partials;     // [gridDim.x][BM][BN] fp32, stream-K partial tiles
  int* flags;          // [gridDim.x], zero between launches
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

template <int BN, int STAGES>
struct Layout {
  static constexpr int B_STAGE = BN * BK * 2;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = STAGES * A_STAGE;
  static constexpr int OFF_BAR = OFF_B + STAGES * B_STAGE;
  static constexpr int BYTES = OFF_BAR + 256;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 B
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }

enum { ITEM_FULL = 0, ITEM_PARTIAL = 1, ITEM_OWNER = 2 };

struct Item {
  int tile, kb0, kb1, kind;
  int last;  // ITEM_OWNER: last contributing CTA
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
    it.last = g;
    return true;
  }
  if (p.sk_iters <= 0) return false;
  const long long I = p.sk_iters;
  const long long a = static_cast<long long>(g) * I / G, b = static_cast<long long>(g + 1) * I / G;
  const int j = idx - n_dp;
  const long long start = j == 0 ? a : (a / KB + j) * KB;
  if (start >= b) return false;
  const long long tile_lo = (start / KB) * KB, tile_hi = tile_lo + KB;
  const long long end = b < tile_hi ? b : tile_hi;
  it.tile = p.dp_tiles + static_cast<int>(start / KB);
  it.kb0 = static_cast<int>(start - tile_lo);
  it.kb1 = static_cast<int>(end - tile_lo);
  it.last = g;
  if (it.kb0 == 0 && it.kb1 == KB) {
    it.kind = ITEM_FULL;
  } else if (it.kb0 == 0) {
    it.kind = ITEM_OWNER;
    int last = g;
    while (last + 1 < G && static_cast<long long>(last + 1) * I / G < tile_hi) ++last;
    it.last = last;
  } else {
    it.kind = ITEM_PARTIAL;
  }
  return true;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int BN, int STAGES>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_bf16_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                 const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2, Params p) {
  using L = Layout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (p.mode == EPI_SWIGLU || p.split0 < p.N) prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    int issued_phase[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued_phase[s] = -1;
    uint32_t c = 0;  // k-blocks issued so far (ring position)
    Item it;
    bool ok = true;
    for (int idx = 0; ok && get_item(p, g, G, idx, it); ++idx) {
      const int m0 = (it.tile % p.m_tiles) * BM;
      const int n0 = (it.tile / p.m_tiles) * BN;
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
      for (int kb = it.kb0; kb < it.kb1; ++kb, ++c) {
        const int s = static_cast<int>(c % STAGES);
        const uint32_t ph = (c / STAGES) & 1u;
        if (lane == 0) ok = mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* sa = smem + L::OFF_A + s * A_STAGE;
          uint8_t* sb = smem + L::OFF_B + s * L::B_STAGE;
          mbar_arrive_expect_tx(&full[s], A_STAGE + L::B_STAGE);
          tma_load_2d(sa, &tmA, &full[s], kb * BK, m0);
          if (p.mode == EPI_SWIGLU) {
            tma_load_2d(sb, &tmB0, &full[s], kb * BK, n0 / 2);
            tma_load_2d(sb + L::B_STAGE / 2, &tmB1, &full[s], kb * BK, n0 / 2);
          } else {
            tma_load_2d(sb, mb, &full[s], kb * BK, brow);
          }
        }
        issued_phase[s] = static_cast<int>(ph);
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      set_status(p.status, ST_WAIT_TIMEOUT);
    }
    // Let every copy this warp issued land before the block can exit.
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s)
        if (issued_phase[s] >= 0) mbar_wait_bounded(&full[s], static_cast<uint32_t>(issued_phase[s]), nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16(BN);
    uint32_t c = 0;
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
      for (int kb = it.kb0; kb < it.kb1; ++kb, ++c) {
        const int s = static_cast<int>(c % STAGES);
        const uint32_t ph = (c / STAGES) & 1u;
        if (lane == 0) ok = mbar_wait_bounded(&full[s], ph, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t da = sw128_desc(smem_u32(smem + L::OFF_A + s * A_STAGE));
          const uint64_t db = sw128_desc(smem_u32(smem + L::OFF_B + s * L::B_STAGE));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes along K per step (encoded >> 4)
            tc_mma_f16(tacc, da + 2 * kk, db + 2 * kk, idesc, (kb > it.kb0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[s]);  // frees the stage once these MMAs have read it
        }
        __syncwarp();
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
      if (it.kind == ITEM_PARTIAL) {
        // write the partial accumulator of this tile to this CTA's slot, then publish it
        float* slot = p.partials + (static_cast<size_t>(g) * BM + r_loc) * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(tbase + c, v);
#pragma unroll
          for (int j = 0; j < 32; j += 8) store8(slot + c + j, v + j);
        }
        __threadfence();
        epi_bar();
        if (et == 0) atomicExch(&p.flags[g], 1);
      } else {
        const int first = g + 1, last = it.kind == ITEM_OWNER ? it.last : g;
        if (it.kind == ITEM_OWNER) {
          // wait for the later contributors of this tile (bounded), in order
          if (et == 0) {
            for (int q = first; q <= last; ++q) {
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
        }
        auto add_partials = [&](float* v, int col) {
          for (int q = first; q <= last; ++q) {
            const float* src = p.partials + (static_cast<size_t>(q) * BM + r_loc) * BN + col;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 t = __ldcg(reinterpret_cast<const float4*>(src + j));
              v[j] += t.x;
              v[j + 1] += t.y;
              v[j + 2] += t.z;
              v[j + 3] += t.w;
            }
          }
        };
        if (p.mode == EPI_SWIGLU) {
          bf16* out = static_cast<bf16*>(p.out);
#pragma unroll 1
          for (int c = 0; c < BN / 2; c += 32) {
            float gv[32], uv[32];
            tmem_ld32(tbase + c, gv);
            tmem_ld32(tbase + BN / 2 + c, uv);
            add_partials(gv, c);
            add_partials(uv, BN / 2 + c);
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
        } else {
          float* out = static_cast<float*>(p.out);
#pragma unroll 1
          for (int c = 0; c < BN; c += 32) {
            float v[32];
            tmem_ld32(tbase + c, v);
            add_partials(v, c);
            if (row < p.M) {
              float* dst = out + static_cast<size_t>(row) * p.ldc + n0 + c;
              if (p.mode == EPI_ADD_F32) {
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                  float o[8];
                  load8(dst + j, o);
#pragma unroll
                  for (int e = 0; e < 8; ++e) o[e] += v[j + e];
                  store8(dst + j, o);
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; j += 8) store8(dst + j, v + j);
              }
            }
          }
        }
        if (it.kind == ITEM_OWNER) {
          epi_bar();  // every thread has read the partials
          if (et == 0)
            for (int q = first; q <= last; ++q) atomicExch(&p.flags[q], 0);
        }
      }
      // accumulator b may be overwritten once every epilogue warp has read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
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

// Scratch that lets every shape use its preferred schedule: the flags plus one 128 x 256
// fp32 partial slot per SM.
size_t gemm_scratch_bytes() {
  return tc::FLAG_BYTES + static_cast<size_t>(std::min(sm_count(), tc::MAX_CTAS)) * tc::BM * 256 * sizeof(float);
}

template <int BN, int STAGES>
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& b2,
                             tc::Params p, void* scratch, size_t scratch_bytes, cudaStream_t s) {
  using L = tc::Layout<BN, STAGES>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(tc::gemm_bf16_tc<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::ALLOC);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  // Persistent grid: one CTA per SM, whole tiles round-robin (data-parallel).  When the
  // tiles fill at most half of the SMs, the k-iterations are instead divided evenly over
  // all SMs (stream-K), which needs scratch for the partial tiles.  Measured on GB300:
  // with five or more CTAs sharing each weight tile (M >= ~512), stream-K desynchronises
  // them and re-reads weights from DRAM (1.66x the bytes), so it is kept to the sparse
  // case where most SMs would otherwise idle.
  const int sms = std::min(sm_count(), tc::MAX_CTAS);
  p.m_tiles = (p.M + tc::BM - 1) / tc::BM;
  p.kb_per_tile = p.K / tc::BK;
  p.tiles = p.m_tiles * (p.N / BN);
  const size_t slot_bytes = static_cast<size_t>(tc::BM) * BN * sizeof(float);
  const long long slots =
      scratch && scratch_bytes > static_cast<size_t>(tc::FLAG_BYTES) ? (scratch_bytes - tc::FLAG_BYTES) / slot_bytes : 0;
  int G = std::min(sms, p.tiles);
  p.dp_tiles = p.tiles;
  p.sk_iters = 0;
  if (2 * p.tiles <= sms) {
    const long long iters = static_cast<long long>(p.tiles) * p.kb_per_tile;
    // at most ~8 CTAs share one tile, one partial slot per CTA, at least 8 k-blocks each
    const int g_sk = static_cast<int>(std::min<long long>(std::min(sms, 8 * p.tiles), slots));
    if (g_sk >= 2 * p.tiles && iters >= 8LL * g_sk) {
      G = g_sk;
      p.dp_tiles = 0;
      p.sk_iters = iters;
    }
  }
  p.flags = scratch ? static_cast<int*>(scratch) : nullptr;
  p.partials = scratch ? reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + tc::FLAG_BYTES) : nullptr;
  tc::gemm_bf16_tc<BN, STAGES><<<G, tc::THREADS, L::ALLOC, s>>>(a, b0, b1, b2, p);
  return cudaGetLastError();
}

// Scratch bytes the schedule of launch_gemm would use for a single-tensor B of N output
// columns with unlimited scratch (0 when the shape runs data-parallel).
size_t gemm_scratch_needed(int N, int M, int K, cb_dtype dt) {
  if (dt != CB_BF16 || M <= 0) return 0;
  const int BN = N % 256 == 0 ? 256 : 128;
  const int sms = std::min(sm_count(), tc::MAX_CTAS);
  const int tiles = ((M + tc::BM - 1) / tc::BM) * (N / BN);
  if (2 * tiles > sms) return 0;
  const long long iters = static_cast<long long>(tiles) * (K / tc::BK);
  const int g_sk = std::min(sms, 8 * tiles);
  if (g_sk < 2 * tiles || iters < 8LL * g_sk) return 0;
  return tc::FLAG_BYTES + static_cast<size_t>(g_sk) * tc::BM * BN * sizeof(float);
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
  const int BN = (N % 256 == 0 && split0 % 256 == 0 && split1 % 256 == 0) ? 256 : 128;
  CUtensorMap ma, mb0, mb1, mb2;
  if (!encode_tmap_bf16_2d(&ma, A, K, M, tc::BK, tc::BM)) return cudaErrorInvalidValue;
  if (mode == EPI_SWIGLU) {
    if (!encode_tmap_bf16_2d(&mb0, B0, K, N / 2, tc::BK, BN / 2)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16_2d(&mb1, B1, K, N / 2, tc::BK, BN / 2)) return cudaErrorInvalidValue;
    mb2 = mb1;
  } else {
    const int r0 = split0, r1 = split1 - split0, r2 = N - split1;
    if (!encode_tmap_bf16_2d(&mb0, B0, K, r0, tc::BK, BN)) return cudaErrorInvalidValue;
    mb1 = mb0;
    mb2 = mb0;
    if (r1 > 0 && !encode_tmap_bf16_2d(&mb1, B1, K, r1, tc::BK, BN)) return cudaErrorInvalidValue;
    if (r2 > 0 && !encode_tmap_bf16_2d(&mb2, B2, K, r2, tc::BK, BN)) return cudaErrorInvalidValue;
  }
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
  if (BN == 256) return launch_tc<256, 4>(ma, mb0, mb1, mb2, p, scratch, scratch_bytes, s);
  return launch_tc<128, 6>(ma, mb0, mb1, mb2, p, scratch, scratch_bytes, s);
}

}  // namespace cb
