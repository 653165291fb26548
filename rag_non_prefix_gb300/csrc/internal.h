// Host-side declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "cacheblend.h"

namespace cb {

// One re-rotation job: n_rows rows of one chunk/layer moved by `delta` positions.
struct RerotSeg {
  const void* k_src;
  const void* v_src;  // may be null (no V copy)
  void* k_dst;
  void* v_dst;
  int n_rows;
  int delta;
};

// Byte offsets inside one layer block of a quantised chunk (the layout cacheblend.h
// documents at cb_codec_layer_bytes): key codes, value codes, key scales and minima per
// channel, value scales and minima per (token, head) row; regions 16-byte aligned, the
// block padded to 256 bytes.
struct CodecLayout {
  size_t kc, vc, ks, kz, vs, vz, bytes;
};
__host__ __device__ inline size_t codec_align(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline CodecLayout codec_layout(int n, int n_kv_heads, int head_dim, int bits) {
  const size_t rows = static_cast<size_t>(n) * n_kv_heads;
  const size_t codes = codec_align(rows * head_dim * bits / 8, 16);
  const size_t chan = codec_align(static_cast<size_t>(n_kv_heads) * head_dim * 4, 16);
  const size_t per_row = codec_align(rows * 4, 16);
  CodecLayout l;
  l.kc = 0;
  l.vc = codes;
  l.ks = 2 * codes;
  l.kz = l.ks + chan;
  l.vs = l.kz + chan;
  l.vz = l.vs + per_row;
  l.bytes = codec_align(l.vz + per_row, 256);
  return l;
}

// One quantised chunk-layer block decoded into its fused-cache rows, keys turned by delta.
struct CodecSeg {
  const uint8_t* block;
  void* k_dst;
  void* v_dst;
  int n;
  int delta;
  int bits;  // 8 or 4
  int pad;
};

// Per request, per layer: where its rows sit in the batched R and S row lists.
struct PlanEntry {
  int r_off, r_n;   // rows of R_i (layer input) of this request
  int s_off, s_n;   // rows of S_i (kept / recomputed) of this request
  int k;            // cached tokens kept at a check layer
  int check;        // 1: deviation + selection at this layer
  int forced_off;   // offset of forced selection (token positions) in the forced buffer, -1 if none
  int pad;
};

// Per request: its fused cache and prompt sizes.
struct ReqDev {
  void* k;                 // fused K [n_layers][N][Hkv][dh] (or one layer when layer_stride == 0)
  void* v;
  long long layer_stride;  // elements between consecutive layers of the fused cache
  int n_tokens;            // N
  int n_cached;            // Nc: tokens 0..Nc-1 are cached, Nc..N-1 the query
};

// Attention work item: `count` query rows of S starting at `row0`, one request.
struct AttnTile {
  int req;
  int row0;
  int count;
  int pad;
};

// Launches of the blended-prefill chain go through launch_chain: with programmatic
// dependent launch enabled (the default; cb_set_launch_overlap), a kernel may start while
// the previous one drains, and runs its prologue up to its pdl_wait.  Every kernel
// launched this way calls pdl_wait before it touches memory that earlier kernels write.
bool launch_overlap_enabled();
void set_launch_overlap(bool on);

// cudaFuncSetAttribute applies to the current device only: kernels that need more than
// the default dynamic shared memory set it once per device (bit d of `done` for device d;
// devices past 63 set it on every launch).  Threads racing on the first launch both set
// it, which is harmless.
struct DeviceOnce {
  std::atomic<uint64_t> done{0};
};
inline cudaError_t max_dynamic_smem_once(const void* kernel, int bytes, DeviceOnce& once) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (once.done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) once.done.fetch_or(bit, std::memory_order_release);
  return e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_chain(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                         Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = launch_overlap_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_embed(const void* embed, const int32_t* ids, int n_rows, int d, int vocab, cb_dtype dt, float* h,
                         int32_t* status, cudaStream_t s);
cudaError_t launch_rerotate(const RerotSeg* segs, int n_segs, int max_rows, int n_kv_heads, int head_dim,
                            const float2* rope_table, int max_pos, cb_dtype dt, int32_t* status, cudaStream_t s);
cudaError_t launch_rerotate_single(const void* k_src, void* k_dst, const void* v_src, void* v_dst, int n_rows,
                                   int n_kv_heads, int head_dim, const float* cs_host, cb_dtype dt, cudaStream_t s);
cudaError_t launch_kv_encode(const void* k, const void* v, int L, int n, int n_kv_heads, int head_dim, int bits,
                             cb_dtype dt, void* blob, cudaStream_t s);
cudaError_t launch_codec_decode(const CodecSeg* segs, int n_segs, int max_n, int n_kv_heads, int head_dim,
                                const float2* rope_table, int max_pos, cb_dtype dt, int32_t* status, cudaStream_t s);
// cs_host: head_dim/2 (cos, sin) pairs of the rotation
cudaError_t launch_codec_decode_blob(const void* blob, int L, int n, int n_kv_heads, int head_dim, int bits,
                                     const float* cs_host, cb_dtype dt, void* k_out, void* v_out, cudaStream_t s);
// decode attention (one query per sequence over its cache rows 0..pos): key ranges of
// DECODE_KEYS keys, decode_splits() of them for the longest sequence; the partial buffers
// hold n_seq * n_heads * n_splits rows of head_dim floats and (max, sum) pairs.
constexpr int DECODE_KEYS = 128;
int decode_splits(int max_keys);
cudaError_t launch_decode_attention(const void* q, const int32_t* pos, const ReqDev* reqs, int n_seq, int layer,
                                    int n_heads, int n_kv_heads, int head_dim, int n_splits, float* part_o,
                                    float2* part_ml, void* out, cb_dtype dt, int32_t* status, cudaStream_t s);
cudaError_t launch_rmsnorm(const float* h, int n_rows, int d, float eps, void* x, cb_dtype dt, cudaStream_t s);
// (both rotate the fresh q / k of the fp32 projection output at each row's position)
cudaError_t launch_deviation_rows(const float* qkv, int n_rows, const int32_t* pos, const int32_t* req,
                                  const ReqDev* reqs, int layer, int n_heads, int n_kv_heads, int head_dim, int mode,
                                  const float2* rope_table, int max_pos, cb_dtype dt, float* dev, int32_t* status,
                                  cudaStream_t s);
cudaError_t launch_deviation_plain(const float* k_new, const float* v_new, const void* k_fus, const void* v_fus,
                                   const int32_t* idx, int n, int kv_width, int mode, cb_dtype dt, float* dev,
                                   cudaStream_t s);
cudaError_t launch_select_plain(const float* dev, const int32_t* cand, int n, int k, int32_t* sel_out,
                                int32_t* status, cudaStream_t s);
cudaError_t launch_select_batched(const float* dev, const int32_t* r_pos, const PlanEntry* plan, const ReqDev* reqs,
                                  const int32_t* forced, int n_req, int32_t* s_src, int32_t* s_pos, int32_t* s_req,
                                  int32_t* status, cudaStream_t s);
cudaError_t launch_post_qkv(const float* qkv, int n_s_rows, const int32_t* s_src, const int32_t* s_pos,
                            const int32_t* s_req, const ReqDev* reqs, int layer, int n_heads, int n_kv_heads,
                            int head_dim, const float2* rope_table, int max_pos, cb_dtype dt, void* q_out,
                            const float* h_in, float* h_out, int d, int32_t* status, cudaStream_t s);
cudaError_t launch_gemm(const void* A, const void* B0, const void* B1, const void* B2, int split0, int split1, void* C,
                        int M, int N, int K, int ldc, int mode, cb_dtype dt, int32_t* status, void* scratch,
                        size_t scratch_bytes, cudaStream_t s);
// Projections of at most GEMV_MAX_ROWS token rows stream the weights with a warp-per-feature
// kernel (launch_gemm takes that path by itself when gemv_applies).
constexpr int GEMV_MAX_ROWS = 2;  // measured: from 3-4 rows on the tensor-core tiles stream faster
bool gemv_applies(int M, int K, cb_dtype dt, const void* A, const void* B0, const void* B1, const void* B2);
cudaError_t launch_gemv(const void* A, const void* B0, const void* B1, const void* B2, int split0, int split1, void* C,
                        int M, int N, int K, int ldc, int mode, cb_dtype dt, cudaStream_t s);
// logits fp32 [M][vocab] = x fp32 [M][d] . W^T for M <= GEMV_MAX_ROWS (d % 8 == 0)
cudaError_t launch_gemv_f32a(const float* x, const void* W, int M, int vocab, int d, float* logits, cb_dtype dt,
                             cudaStream_t s);
// bytes of GEMM scratch (stream-K partial tiles + flags) that enable every schedule
size_t gemm_scratch_bytes();
void gemm_set_orientation(int o);  // 0 model, 1 token rows, 2 weight rows
// scratch the schedule of one single-B GEMM uses when scratch is unlimited (0: none)
size_t gemm_scratch_needed(int N, int M, int K, cb_dtype dt);
// scratch launch_gemm uses for these operands given scratch_bytes of it (<= scratch_bytes)
size_t gemm_scratch_used(const void* A, const void* B0, const void* B1, const void* B2, int split0, int split1, int M,
                         int N, int K, int mode, cb_dtype dt, size_t scratch_bytes);
// Device address of the status word that the standalone GEMM calls (cb_gemm,
// cb_gemm_noalloc) report device-side problems into, on the current device.
cudaError_t standalone_gemm_status(int32_t** out);
cudaError_t launch_attention(const void* q, const int32_t* s_pos, const int32_t* s_req, const ReqDev* reqs,
                             const AttnTile* tiles, int n_tiles, int layer, int n_heads, int n_kv_heads, int head_dim,
                             void* out, cb_dtype dt, cudaStream_t s);
int attention_tile_rows(int n_heads, int n_kv_heads, cb_dtype dt);
// tcgen05 attention (bf16, head_dim 128): tiles of request r are tiles[tile_off[r] .. tile_off[r+1]).
// When a layer's (tile, KV head) units leave SMs idle (one launch per layer) and part_o is given,
// the longest tiles get a second CTA (as many as the idle SMs hold, plus two per KV head), and such
// a tile of at least
// ATTN_SPLIT_MIN_BLOCKS 128-key blocks (known on the device only) is split into two key ranges,
// merged by whichever CTA finishes second: part_o holds
// ATTN_SPLIT_UNITS * 2 * 128 * 128 floats, part_ml as many * 128 (max, sum) pairs, part_cnt
// ATTN_SPLIT_UNITS counters that must be zero before the first launch (each launch leaves them zero).
constexpr int ATTN_SPLIT_UNITS = 256;
void attention_set_tiles(int tiles);  // 0 by the launch's size, 1 or 2 query tiles per CTA
constexpr int ATTN_SPLIT_MIN_BLOCKS = 12;
cudaError_t launch_attention_bf16(const void* q, const int32_t* s_pos, const AttnTile* tiles, const int* tile_off,
                                  const CUtensorMap* kmaps, const CUtensorMap* vmaps, const int* n_kv,
                                  const int* one_layer, int n_req, int layer, int n_heads, int n_kv_heads, void* out,
                                  int32_t* status, float* part_o, float2* part_ml, int* part_cnt, cudaStream_t s);
// 4-D tensor map over a bf16 KV cache [L][N][Hkv][128] (layer_stride_elems 0: one layer)
bool encode_kv_map(CUtensorMap* map, const void* base, int n_layers, int n_tokens, int n_kv_heads,
                   long long layer_stride_elems);
cudaError_t launch_last_rows_norm(const float* h, const int32_t* rows, int n, int d, float eps, float* x_out,
                                  cudaStream_t s);
cudaError_t launch_lm_head(const float* x, int n_req, int d, const void* w, int vocab, cb_dtype dt, float* logits,
                           cudaStream_t s);
cudaError_t launch_argmax(const float* logits, int n_req, int vocab, int32_t* const* outs, int32_t* out_dev,
                          cudaStream_t s);
cudaError_t launch_write_hidden(const float* h, const int32_t* s_pos, int row0, int n, int d, float* out,
                                cudaStream_t s);

enum { EPI_STORE_F32 = 0, EPI_ADD_F32 = 1, EPI_SWIGLU = 2, EPI_QKV_ROPE = 3 };

// EPI_QKV_ROPE (the paired GEMM only): the outputs are [q | k | v] of head_dim 128; q and k
// are rotated at each row's position (RoPE, the table's (cos, sin) of pairs i and i + 64), q
// goes to q_out [M][q_width] in bf16 and k, v to the fused cache row of that position, as the
// post-QKV scatter does for an uncompacted set.
struct QkvRope {
  const int32_t* s_pos;  // [M] token positions
  const int32_t* s_req;  // [M] request of each row
  const ReqDev* reqs;
  const float2* rope;    // [max_pos][64]
  int layer, max_pos;
  void* q_out;
  int q_width, kvw;
};

// Paired GEMM (gemm_pair.cu): clusters of one or two CTA pairs, weights on the tensor
// core's rows, 256 weight rows x bt tokens per pair.
struct PairPlan {
  int cl;               // CTAs per cluster (2 or 4)
  int bt;               // tokens per pair tile
  int ksub;             // 64-element atoms of K per ring stage
  int clusters;         // clusters resident at once
  int w_tiles;          // weight tiles (256 rows; SwiGLU 128 features)
  double us;            // the time model's estimate
};
// Whether the operands suit the paired kernel, and its best plan (forced_bt >= 16 fixes
// the token tile); false when they do not, or pairing is switched off.  The paired kernel
// takes no scratch.
bool plan_gemm_pair(int M, int N, int K, int split0, int split1, int mode, int forced_bt, PairPlan* out);
cudaError_t launch_gemm_pair(const PairPlan& g, const void* A, const void* B0, const void* B1, const void* B2,
                             int split0, int split1, void* C, int M, int N, int K, int ldc, int mode, int32_t* status,
                             cudaStream_t s, const QkvRope* qr = nullptr);
bool gemm_store_pair_plan(const void* A, const void* B0, const void* B1, const void* B2, int split0, int split1, int M,
                          int N, int K, const void* scratch, size_t scratch_bytes, PairPlan* pp);
// [q | k | v] = x [Wq; Wk; Wv]^T with RoPE and the scatter in the epilogue (EPI_QKV_ROPE), on the
// CTA-pair plan launch_gemm takes for the projection alone, so that every output is summed as
// there; cudaErrorNotSupported when launch_gemm would not take pairs (the caller then runs the
// GEMM and the post-QKV scatter).
cudaError_t launch_qkv_rope_gemm(const void* x, const void* wq, const void* wk, const void* wv, int M, int d,
                                 const QkvRope& qr, int32_t* status, const void* scratch, size_t scratch_bytes,
                                 cudaStream_t s);
void set_qkv_fusion(bool enabled);
bool qkv_fusion();
void gemm_set_pairing(int m);  // 0 model, 1 never, 2 clusters of one pair, 4 of two pairs
// launch_gemm's schedule for a bf16 GEMM (single-tensor B) as text; snprintf's return value
int gemm_describe(int M, int N, int K, int mode, size_t scratch_bytes, char* buf, size_t len);
int gemm_pairing();
// tensor-map encoder (driver entry point, resolved once)
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                 uint64_t pitch, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz);
bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                         uint32_t box_rows);

}  // namespace cb
