/*
 * cacheblend.h -- C ABI of the GB300 (sm_103a) blended-prefill library.
 *
 * CacheBlend ("cached knowledge fusion") reuses KV caches of RAG chunks that were
 * each prefilled alone from position 0.  For a prompt made of such chunks plus a
 * query it re-rotates the cached keys to their new positions and, layer by layer,
 * recomputes only the tokens whose cached KV deviates most from what a full
 * prefill would give.  Pages the comments below cite (by title and section):
 *
 *   [P1] "論文解説: CacheBlend - RAG向けKVキャッシュ融合によるLLM推論高速化" (0h-n0.github.io)
 *   [P2] "KVキャッシュを再利用してLLM推論を4.49倍高速化——KVBoostが切り拓く自宅サーバーLLMの新境地"
 *   [P3] "논문: CacheBlend: Fast Large Language Model Serving for RAG with Cached Knowledge Fusion" (jaehun.me)
 *   [P4] "LMCache: KV キャシを GPU の外へ" (ttlab.hopto.org)
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless the argument name ends in _host.
 *   - The caller owns every buffer (weights, KV caches, outputs, workspace) and
 *     every stream; the library owns only the context, its events, its chunk
 *     registry and a small rotary cos/sin table inside the workspace.
 *   - Streams are passed as void* holding a cudaStream_t (NULL = legacy default stream).
 *   - Calls never throw and never abort.  Arguments are checked synchronously
 *     (null pointers, sizes, 16-byte alignment of vector I/O, dtype) and a bad one
 *     returns an error before anything is enqueued.  Device-side problems (a NaN
 *     deviation, an index out of range, a bounded wait that ran out) set bits of a
 *     status word in the workspace; cb_get_status() reports them.
 *   - Everything is asynchronous on the given stream except cb_synchronize(),
 *     cb_get_status(), the *_size() queries, cb_create/cb_destroy and
 *     cb_set_workspace().
 *   - Row-major layouts; weights are [out_features][in_features].  KV caches are
 *     [n_layers][n_tokens][n_kv_heads][head_dim] of the model dtype.
 */
#ifndef CACHEBLEND_H
#define CACHEBLEND_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CB_OK = 0,
  CB_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad enum, out-of-range scalar */
  CB_ERR_SHAPE = 2,        /* sizes that do not fit the model or the kernels' tiling */
  CB_ERR_DTYPE = 3,        /* dtype not supported by this entry point */
  CB_ERR_NOT_FOUND = 4,    /* chunk id missing from the registry */
  CB_ERR_WORKSPACE = 5,    /* no workspace, or too small for the call */
  CB_ERR_CUDA = 6,         /* a CUDA runtime call failed (cb_last_error has its text) */
  CB_ERR_TIMEOUT = 7,      /* a host wait passed its deadline */
  CB_ERR_NAN = 8,          /* a deviation was NaN (reported by the device status word) */
  CB_ERR_DEVICE = 9,       /* another device-side check failed (index range, bounded wait) */
  CB_ERR_STATE = 10        /* call out of order (e.g. prefill_layer before blend_begin) */
} cb_status;

typedef enum { CB_F32 = 0, CB_BF16 = 1 } cb_dtype;

/* Decoder shape.  head_dim must be 128 for CB_BF16 (64 or 128 for CB_F32);
 * d_model, n_heads*head_dim and ffn_dim multiples of 128 for CB_BF16.
 * max_positions bounds token positions (rotary table size). */
typedef struct {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  double rope_theta;
  float rms_eps;
  cb_dtype dtype;
  int max_positions;
} cb_model_cfg;

/* Borrowed weight pointers (device, model dtype).  The per-layer members are HOST
 * arrays of n_layers device pointers; cb_create copies the arrays, not the weights.
 *   embed [vocab][d]   lm_head [vocab][d]
 *   wq [H*dh][d]  wk, wv [Hkv*dh][d]  wo [d][H*dh]  wgate, wup [ffn][d]  wdown [d][ffn]
 * RMSNorm weights are 1 and there are no biases. */
typedef struct {
  const void* embed;
  const void* lm_head;
  const void* const* wq;
  const void* const* wk;
  const void* const* wv;
  const void* const* wo;
  const void* const* wgate;
  const void* const* wup;
  const void* const* wdown;
} cb_weights;

typedef struct cb_ctx cb_ctx;

/* --------------------------------------------------------------------- lifetime */
cb_status cb_create(const cb_model_cfg* cfg, const cb_weights* weights, cb_ctx** out);
cb_status cb_destroy(cb_ctx* ctx);
const char* cb_status_string(cb_status s);
/* Text of the last error seen by this context (or by the standalone calls if ctx is NULL). */
const char* cb_last_error(const cb_ctx* ctx);

/* Workspace: device memory the caller allocates (e.g. with torch.empty) and hands
 * over.  max_tokens bounds the total prompt tokens of one call summed over its
 * requests; max_requests bounds the requests of one call. */
size_t cb_workspace_size(const cb_ctx* ctx, int max_tokens, int max_requests);
/* Binds the workspace; writes the rotary table into it (synchronous). */
cb_status cb_set_workspace(cb_ctx* ctx, void* ws, size_t bytes, int max_tokens, int max_requests);

/* --------------------------------------------------------------------- chunk cache
 * A chunk's KV cache is the chunk prefilled ALONE from position 0: [P3] "어떤 문제를
 * 해결하는가" and [P1] 背景と動機 (each retrieved document is precomputed on its own).
 * cb_precompute_chunk runs that prefill on the GPU and writes K (with rotary
 * embedding at local positions) and V for every layer:
 *   ids [n] int32;  k_out, v_out [n_layers][n][n_kv_heads][head_dim].  */
cb_status cb_precompute_chunk(cb_ctx* ctx, const int32_t* ids, int n, void* k_out, void* v_out, void* stream);

/* Registers a cached chunk under chunk_id (the pages key caches by text hash:
 * [P1] vLLMとの統合, hash table in CPU memory; [P3] loading controller).
 * ids: device int32[n] token ids (needed because layer 0 runs on every token).
 * k, v: [n_layers][n][n_kv_heads][head_dim]; device memory if on_host == 0, else
 * page-locked host memory (staged per layer by cb_fetch_kv).  Borrowed: the
 * caller keeps them alive while registered.  Re-registering an id replaces it. */
cb_status cb_register_chunk(cb_ctx* ctx, uint64_t chunk_id, const int32_t* ids, const void* k, const void* v,
                            int n, int on_host);
cb_status cb_unregister_chunk(cb_ctx* ctx, uint64_t chunk_id);
int cb_registered_chunks(const cb_ctx* ctx);

/* --------------------------------------------------------------------- loading controller
 * [P3] loading controller: it checks whether the chunks a retriever chose have caches and
 * where they are stored, and coordinates loading with recompute; the cache manager finds a
 * cache by a hash of its text ([P1] vLLMとの統合: a hash table in CPU memory).  The key used
 * here is the chunk's content only, so a chunk is found wherever it sits in a prompt. */

/* FNV-1a 64 (Fowler, Noll, Vo) of the token ids as little-endian int32 bytes (host array).
 * Intended as the chunk_id of cb_register_chunk / cb_request. */
uint64_t cb_chunk_hash(const int32_t* ids_host, int n);

enum { CB_TIER_MISSING = -1, CB_TIER_DEVICE = 0, CB_TIER_HOST = 1 };
enum { CB_ACT_USE = 0, CB_ACT_LOAD = 1, CB_ACT_RECOMPUTE = 2 };
typedef struct {
  int n_tokens;
  int tier;      /* CB_TIER_* */
  double bytes;  /* bytes a load moves (the chunk's KV, or its quantised blob) */
} cb_chunk_info;
/* What the registry holds under chunk_id: tier, tokens and bytes (CB_TIER_MISSING, 0, 0 if
 * it is not registered; the call still returns CB_OK). */
cb_status cb_chunk_info_of(const cb_ctx* ctx, uint64_t chunk_id, cb_chunk_info* out);

/* Costs the plan weighs, measured on the machine: the host->device link of the staging tier,
 * the full-prefill time per token, and the part of the blend's recompute time that does not
 * scale with the ratio (layer 0, the query, launch overheads). */
typedef struct {
  double link_bytes_per_s;
  double link_latency_s;       /* per chunk loaded */
  double prefill_s_per_token;
  double recompute_fixed_s;
  double r_min, r_max;         /* quality bounds of the ratio ([P1]: 5 % latency first ... 20 % quality first) */
} cb_cost_model;
/* Plan of one prompt (host arrays).  Per chunk ([P4] §5 損益分岐): a device-resident chunk is
 * used (CB_ACT_USE); a host-resident one is loaded when bytes / link + latency is below
 * n_tokens x prefill time per token, else recomputed; a missing one is recomputed (the caller
 * prefills it, e.g. with cb_precompute_chunk, and registers it).  The ratio ([P1] パイプライン化の設計,
 * 閾値チューニング): T_load = the summed load times, T_prefill = N x prefill time per token (N = all
 * chunk tokens + n_query), T_recompute(r) = recompute_fixed_s + r x T_prefill, and
 * *ratio_out = clamp((T_load - recompute_fixed_s) / T_prefill, r_min, r_max): the largest ratio
 * whose recompute still hides under the load (r_min when nothing is loaded).  t_load_out and
 * t_recompute_out (T_recompute at the chosen ratio) may be NULL.  Host-only; no GPU needed. */
cb_status cb_plan_loading(const cb_cost_model* model, const cb_chunk_info* chunks_host, int n_chunks, int n_query,
                          int32_t* actions_host, double* ratio_out, double* t_load_out, double* t_recompute_out);

/* --------------------------------------------------------------------- KV codec
 * KIVI-style asymmetric quantisation of a chunk's KV cache ([P2] KV量子化とメモリ管理 /
 * 非対称量子化: keys per channel, values per token, int8 or int4; about 2x / 4x fewer bytes
 * to keep or to stage).  A key group is one channel of one KV head of one layer over the
 * chunk's n tokens; a value group is one token's head_dim channels of one KV head.  Per group:
 * scale = (max - min) / (2^bits - 1), code = clamp(rint((x - min) / scale), 0, 2^bits - 1)
 * (0 when scale is 0), each step one IEEE float32 operation; decoding gives min + code * scale.
 *
 * A quantised chunk ("blob") is n_layers blocks of cb_codec_layer_bytes() bytes each.  With
 * rows = n * Hkv and code_bytes = rows * head_dim * bits / 8, one block holds, each region
 * starting at a multiple of 16 bytes (offsets rounded up) and the block padded to 256 bytes:
 *   key codes   [n][Hkv][head_dim * bits / 8] uint8    at 0
 *   value codes [n][Hkv][head_dim * bits / 8] uint8    at R16(code_bytes)
 *   key scale   [Hkv][head_dim] float32                at 2 * R16(code_bytes)
 *   key min     [Hkv][head_dim] float32                after the key scales (R16)
 *   value scale [n][Hkv] float32                       after the key minima (R16)
 *   value min   [n][Hkv] float32                       after the value scales (R16)
 * int4 packs channel 2j in the low and channel 2j + 1 in the high nibble of byte j.
 * head_dim must be 64 or 128. */
size_t cb_codec_layer_bytes(int n_tok, int n_kv_heads, int head_dim, int bits);  /* 0 for bad sizes */
/* Quantises k, v [n_layers][n_tok][n_kv_heads][head_dim] of dtype into blob (device, 16-byte
 * aligned, n_layers * cb_codec_layer_bytes() bytes). */
cb_status cb_kv_encode(const void* k, const void* v, int n_layers, int n_tok, int n_kv_heads, int head_dim,
                       cb_dtype dtype, int bits, void* blob, void* stream);
/* Dequantises a blob and re-rotates its keys by delta_pos positions (the rotation of
 * cb_rope_rerotate) in one pass: k_out, v_out [n_layers][n_tok][n_kv_heads][head_dim] of dtype. */
cb_status cb_kv_decode(const void* blob, int n_layers, int n_tok, int n_kv_heads, int head_dim, int bits,
                       int delta_pos, double theta, cb_dtype dtype, void* k_out, void* v_out, void* stream);
/* Registers a quantised chunk (a blob of cb_kv_encode) under chunk_id; ids as for
 * cb_register_chunk.  on_host == 0: the blob is in device memory and is decoded straight into
 * the fused caches when a batch begins.  on_host != 0: the blob is in page-locked host memory;
 * cb_fetch_kv copies each layer's block into the staging ring (cb_set_staging) and
 * cb_prefill_layer decodes it from there.  Borrowed, like cb_register_chunk. */
cb_status cb_register_chunk_codec(cb_ctx* ctx, uint64_t chunk_id, const int32_t* ids, const void* blob, int n,
                                  int bits, int on_host);
/* Device buffer (caller-owned, 16-byte aligned) for the staging ring of host-resident quantised
 * chunks.  A batch uses slots of S = the sum of cb_codec_layer_bytes() over the occurrences of
 * its host-resident quantised chunks; layer i goes to slot i mod (bytes / S).  A batch that
 * needs S > bytes fails at cb_blend_begin with CB_ERR_WORKSPACE.  With k slots, cb_fetch_kv of
 * layer i is accepted only after cb_prefill_layer of layer i - k was enqueued (CB_ERR_STATE
 * otherwise); cb_blend_prefill orders its calls that way.  NULL / 0 removes the buffer. */
cb_status cb_set_staging(cb_ctx* ctx, void* buf, size_t bytes);

/* --------------------------------------------------------------------- standalone kernels */

/* RoPE re-rotation of cached keys by delta_pos positions; V is copied.
 * [P1] 技術的詳細 / 位置エンコーディングの更新: K_new[j] = R(dp_j) . K_cached[j].
 * Rotary pairs are (i, i + head_dim/2) with angle delta_pos * theta^(-2i/head_dim),
 * evaluated in double precision on the host; the rotation runs in fp32.
 * k_src/k_dst, v_src/v_dst: [n_tok][n_kv_heads][head_dim] of dtype, 16-byte
 * aligned; in place (src == dst) is allowed.  v_src/v_dst may both be NULL. */
cb_status cb_rope_rerotate(const void* k_src, void* k_dst, const void* v_src, void* v_dst, int n_tok,
                           int n_kv_heads, int head_dim, int delta_pos, double theta, cb_dtype dtype,
                           void* stream);

/* Squared KV deviation of fresh rows against the fused cache.
 * [P1] 技術的詳細 / HKVD トークン選定: Delta_KV^(i)[j] = ||KV_cached^(i)[j] - KV_full^(i)[j]||_2
 * (squared: same ranking).  k_new, v_new: fp32 [n][kv_width] (fresh, after RoPE);
 * k_fus, v_fus: dtype [*][kv_width]; row j is compared with fused row idx[j]
 * (idx NULL: row j).  mode 0 = K and V, 1 = K only, 2 = V only (squared L2), 3 = 1 - cos
 * of the concatenated K and V rows ([P2] シーム修復戦略 / CacheBlendRecompute).
 * dev_out fp32 [n]; accumulation in fp32. */
cb_status cb_kv_deviation(const float* k_new, const float* v_new, const void* k_fus, const void* v_fus,
                          const int32_t* idx, int n, int kv_width, int mode, cb_dtype dtype, float* dev_out,
                          void* stream);

/* HKVD selection: the k candidates of largest deviation, ties to the smaller
 * candidate value, written to sel_out[k] in ASCENDING order.
 * [P1] 段階的フィルタリングスキーム (top r% by deviation).  dev fp32 [n]; cand int32 [n]
 * (token indices, distinct; NULL = 0..n-1).  n <= 65536, 0 <= k <= n.  A NaN
 * deviation sets CB_ERR_NAN in *status (device int32, may be NULL); the NaN ranks
 * below every number. */
cb_status cb_select_hkvd(const float* dev, const int32_t* cand, int n, int k, int32_t* sel_out, int32_t* status,
                         void* stream);

/* Dense GEMM used by the projections: C = A . B^T with A [M][K], B [N][K] of dtype,
 * fp32 accumulation.  epilogue 0: C fp32 [M][ldc] = acc;  1: C fp32 += acc
 * (residual add);  2: C (dtype) [M][N/2] = SiLU(acc[:, gate]) * acc[:, up] where
 * B2 (may not be NULL) holds the "up" rows and B the "gate" rows, each [N/2][K]
 * (then N counts both).  bf16 runs on the tcgen05 tensor cores (persistent, one CTA
 * per SM), fp32 on CUDA cores.  bf16 needs K % 64 == 0 and N % 128 == 0.
 * scratch: NULL (whole output tiles per CTA only) or device memory, zero-filled before
 * its first use, for the stream-K schedules (the k-iterations of the output tiles
 * divided evenly over the SMs, when whole tiles would leave SMs idle or a last wave
 * ragged; the sums of split tiles are formed in a fixed order, so results repeat
 * exactly): 1 KiB of flags, then one 128 KiB fp32 partial slot per CTA of the split (a smaller
 * scratch narrows the split).  cb_gemm_scratch_size() bytes allow every split.  The
 * call leaves the flags zeroed.  Calls sharing one scratch must not overlap on the GPU.
 * Device-side problems (a stream-K wait for a partial tile that gave up after 2 s) are
 * recorded in the standalone GEMM status word that cb_gemm_get_status() reads; after such
 * a report the output is not valid and the scratch's flags must be zeroed again. */
cb_status cb_gemm(const void* A, const void* B, const void* B2, void* C, int M, int N, int K, int ldc, int epilogue,
                  cb_dtype dtype, void* scratch, size_t scratch_bytes, void* stream);
size_t cb_gemm_scratch_size(void);

/* Tile orientation of the bf16 GEMMs, process-wide (a tuning and test hook; default 0).
 * 0: chosen per shape by the library's time model; 1: tokens (rows of A) as the 128
 * rows of each tensor-core tile; 2: output features (rows of B) as the tile rows and
 * tokens as its columns, in tiles of a multiple of 16 tokens (used where the q|k|v
 * split points are multiples of 128; otherwise 1); 16..256, a multiple of 16: as 2 with
 * that many tokens per tile.  Results agree to fp32 rounding of the same sums.  Other
 * values: CB_ERR_INVALID_ARG. */
cb_status cb_gemm_set_orientation(int orientation);

/* CTA pairs for the bf16 GEMMs, process-wide (a tuning and test hook; default 0).  A pair
 * of CTAs on two SMs computes 256 weight rows x a tile of tokens with one 256-row
 * tensor-core instruction (tcgen05 cta_group::2), each CTA staging 128 weight rows and half
 * of the tokens; a cluster of two pairs also shares the weight rows by multicast.
 * 0: chosen per shape by the library's time model (only while cb_gemm_set_orientation is
 * 0); 1: never; 2: clusters of one pair; 4: clusters of two pairs (2 and 4 apply where the
 * shape allows pairs: output features a multiple of 256 with the q|k|v split points
 * multiples of 128, SwiGLU features a multiple of 128, K a multiple of 64; a token tile
 * forced by cb_gemm_set_orientation applies to the pairs too).  Results agree to fp32
 * rounding of the same sums.  Other values: CB_ERR_INVALID_ARG. */
cb_status cb_gemm_set_pairing(int pairing);

/* The schedule a bf16 cb_gemm of M x N x K with `epilogue` and scratch_bytes of scratch
 * would run under the current hooks, as a NUL-terminated line of text in buf (at most len
 * bytes, truncated): the kernel (single CTAs or CTA pairs), its tiles, grid and the time
 * model's estimate.  For tuning and reports; no GPU work.  CB_ERR_INVALID_ARG for a null
 * buffer, a negative size or an unknown epilogue. */
cb_status cb_gemm_describe(int M, int N, int K, int epilogue, size_t scratch_bytes, char* buf, size_t len);

/* Fused QKV of the bf16 blend, process-wide (a tuning and test hook; default 1): 1 runs,
 * in a layer whose recomputed set is not re-selected (no check), the Q/K/V projection with
 * RoPE and the scatter of K and V into the fused cache in the GEMM's epilogue wherever the
 * projection runs on CTA pairs (head_dim 128), with the projection's own plan; 0 runs the
 * projection and the post-QKV kernel separately.  Both compute the same values in the same
 * order.  Other values: CB_ERR_INVALID_ARG. */
cb_status cb_set_qkv_fusion(int enabled);

/* Query tiles per CTA of the bf16 attention, process-wide (a tuning and test hook;
 * default 0).  0: two 128-row tiles of one KV head per CTA when a launch's tile pairs
 * times the KV heads fill the SMs (the tensor core then works for one tile while the
 * other's softmax runs, and each K/V block is loaded once for both), else one tile per
 * CTA with the longest tiles' key ranges split over two CTAs; 1 or 2: that many tiles
 * per CTA.  Results agree to the rounding of the same sums.  Other values:
 * CB_ERR_INVALID_ARG. */
cb_status cb_attention_set_tiles(int tiles);

/* Programmatic dependent launch of the blended-prefill kernels, process-wide (default
 * 1): each kernel of a layer may start while the previous one drains, running the part
 * of its prologue that touches only its own on-chip memory (barriers, tensor-memory
 * allocation, tensor-map prefetch) before it waits for the previous kernel's results.
 * 0 launches every kernel after the previous one has completed.  Results are identical
 * either way. */
cb_status cb_set_launch_overlap(int enabled);

/* Allocation-free variant of cb_gemm (no counterpart on the pages: an addition for
 * callers that cannot allocate device memory, e.g. a process held to a fixed device
 * budget after start-up, or code inside a framework that owns every allocation).
 * Same arguments and results as cb_gemm without the scratch arguments: its stream-K
 * scratch is a built-in device array of CB_GEMM_STATIC_SCRATCH_BYTES (4 MiB + 1 KiB:
 * the flags and 32 partial slots) that every GPU loading the library holds until the
 * process exits.  The schedule narrows its stream-K split to those 32 slots, as cb_gemm
 * does with a small scratch, so every shape cb_gemm accepts runs; the few-row GEMV and
 * data-parallel shapes use no scratch.  A schedule asking for more than the array would
 * be refused with CB_ERR_WORKSPACE.  Every non-OK return leaves its reason in
 * cb_gemm_noalloc_error() (an empty string after CB_OK).  The call allocates nothing;
 * its first call on a device looks up the array's device address (make that first call
 * before any stream capture), and each call that uses the array zeroes its flags first.
 * All calls share the array, so calls that overlap on the GPU (other streams, other
 * threads) race: order them on one stream.  Device-side problems go to the standalone
 * GEMM status word (cb_gemm_get_status). */
#define CB_GEMM_STATIC_SCRATCH_BYTES ((size_t)(4u << 20) + 1024u)
cb_status cb_gemm_noalloc(const void* A, const void* B, const void* B2, void* C, int M, int N, int K, int ldc,
                          int epilogue, cb_dtype dtype, void* stream);
const char* cb_gemm_noalloc_error(void);
/* Bytes of the built-in array that cb_gemm_noalloc uses for this shape on the current
 * device with 16-byte aligned operands (0: the few-row GEMV or whole output tiles, no
 * scratch; never more than CB_GEMM_STATIC_SCRATCH_BYTES).  Host-side planning only. */
size_t cb_gemm_noalloc_scratch_used(int M, int N, int K, int epilogue, cb_dtype dtype);

/* Status of the standalone GEMM calls (cb_gemm, cb_gemm_noalloc) on the current device:
 * waits up to timeout_ms (< 0: no limit) for the work enqueued on `stream`, then reads
 * and clears a device status word that those calls' kernels set when a bounded wait for
 * a stream-K partial tile gave up (their output is then not valid).  CB_OK, CB_ERR_DEVICE
 * (the word was set), CB_ERR_TIMEOUT (the stream did not finish in time; the word is not
 * read) or CB_ERR_CUDA.  The reason is in cb_gemm_noalloc_error().  One word per device
 * is shared by every caller: read it after the GEMMs that matter, on their stream. */
cb_status cb_gemm_get_status(void* stream, int timeout_ms);

/* Causal attention of sparse queries over one KV cache ([P3] "어떤 토큰을 다시 계산하는가":
 * selected queries attend under the causal mask to all available K/V).
 * q [m][n_heads][head_dim] dtype; q_pos int32 [m] (positions, < n_kv);
 * k, v [n_kv][n_kv_heads][head_dim] dtype; out [m][n_heads][head_dim] dtype.
 * Scale 1/sqrt(head_dim); head h reads KV head h / (n_heads / n_kv_heads). */
cb_status cb_attention(const void* q, const int32_t* q_pos, int m, const void* k, const void* v, int n_kv,
                       int n_heads, int n_kv_heads, int head_dim, void* out, cb_dtype dtype, void* stream);

/* --------------------------------------------------------------------- blended prefill */

/* Per-layer ratio of ALL cached tokens of a request to keep recomputed
 * (gradual filtering, [P1] 段階的フィルタリングスキーム; [P3] §4.3 narrowing of the
 * candidates).  layer_ratio is a HOST array [n_layers]; a negative entry means
 * "no check: keep the previous layer's set".  Layer 0 always runs on every token.
 * At a check layer k = ceil(r * Nc - 1e-9) cached tokens are kept (clamped to the
 * candidates that exist); query tokens are always kept.
 * dev_mode: 0 = squared L2 of K and V, 1 = K only, 2 = V only, 3 = 1 - cos of the
 * concatenated K and V rows (the cosine deviation of [P2] シーム修復戦略 /
 * CacheBlendRecompute; a zero row against a zero row gives 0, against a non-zero one 1).
 * forced_sel_host: NULL, or a host array [n_layers] of host int32 arrays: at a
 * check layer with a non-NULL entry the given sets replace the top-k (used to
 * separate numerics from selection).  Each entry lists, request after request,
 * a count c followed by c ascending cached token indices of that request.
 * select_mode: CB_SELECT_HKVD (deviation-guided, above) or CB_SELECT_SEAM: spatial
 * seam repair ([P2] シーム修復戦略 / SelectiveRecompute): the last seam_tokens tokens
 * of every cached chunk (each ends at a chunk boundary) and the query are recomputed
 * at every layer, layer 0 included; nothing else is recomputed and no deviation is
 * measured (layer_ratio_host, dev_mode and forced_sel_host are ignored; the ratio
 * array may be NULL). */
enum { CB_SELECT_HKVD = 0, CB_SELECT_SEAM = 1 };

/* The layer_ratio array of gradual filtering ([P1] 段階的フィルタリングスキーム: the
 * deviation is measured at an early layer over many tokens, and later layers keep a
 * narrower share of the earlier set).  out_host [n_layers] gets: layer 0 -1 (no check:
 * layer 0 runs on every token, which gives every cached token a layer-1 input); layer 1
 * r1; layers 2 .. 1 + n_narrow r1 + (r - r1) * j / n_narrow for j = 1 .. n_narrow (the
 * last of them is r); later layers -1 (the last checked set is kept).
 * CB_SCHEDULE_FIXED checks once, at layer 1, with r.  CB_SCHEDULE_GRADUAL takes r1 < 0
 * as min(1, 2 r).  Needs 0 <= r <= r1 <= 1 and n_narrow >= 0, else CB_ERR_INVALID_ARG.
 * Host-only. */
enum { CB_SCHEDULE_FIXED = 0, CB_SCHEDULE_GRADUAL = 1 };
cb_status cb_ratio_schedule(int n_layers, double r, int schedule, double r1, int n_narrow, double* out_host);

/* Cached tokens kept at a check layer of ratio r: ceil(r * n_cached - 1e-9) (0 when
 * r <= 0).  The 1e-9 keeps r * Nc that rounds just above an integer on that integer.
 * Host-only; the blend uses the same rule. */
int cb_k_for_ratio(double r, int n_cached);
typedef struct {
  int n_layers;
  const double* layer_ratio_host;
  int dev_mode;
  const int32_t* const* forced_sel_host;
  int select_mode;
  int seam_tokens;
} cb_blend_params;

/* One prompt: cached chunks (by registry id) in order, then the query tokens
 * (uncached, always recomputed).  A system prefix is simply the first chunk.
 *   query_ids: device int32 [n_query] (n_query >= 1)
 *   fused_k, fused_v: caller-owned [n_layers][kv_capacity][n_kv_heads][head_dim] (N = all
 *     prompt tokens <= kv_capacity): the blended cache, rows 0..N-1 written by the call
 *   out_hidden: NULL or fp32 [N][d_model]; rows of the final recomputed set are
 *     written (other rows untouched)
 *   out_sel: NULL or int32 [n_layers][N]: per layer the recomputed token indices,
 *     ascending; out_sel_count: NULL or int32 [n_layers] (device)
 *   out_first_token: NULL or int32 [1]: argmax of the LM head at the last token
 *   kv_capacity: rows per layer of fused_k / fused_v (0: exactly N); a capacity above N leaves
 *     room to decode after the blend (cb_decode_step) */
typedef struct {
  int n_chunks;
  const uint64_t* chunk_ids_host;
  const int32_t* query_ids;
  int n_query;
  void* fused_k;
  void* fused_v;
  float* out_hidden;
  int32_t* out_sel;
  int32_t* out_sel_count;
  int32_t* out_first_token;
  int kv_capacity;
} cb_request;

/* Whole blended prefill of n_req prompts (batched: the projections of all
 * requests share one GEMM per weight).  Equivalent to cb_blend_begin, then
 * cb_fetch_kv for every layer on copy_stream, cb_prefill_layer for every layer
 * on stream, cb_blend_finish.  copy_stream may be NULL when no chunk lives on the host. */
cb_status cb_blend_prefill(cb_ctx* ctx, const cb_request* reqs, int n_req, const cb_blend_params* params,
                           void* stream, void* copy_stream);

/* Full prefill of ids [n] from position 0 (the full-recompute baseline, [P1] 実験結果).
 * k_out, v_out: NULL or [n_layers][n][n_kv_heads][head_dim] (NULL: a one-layer
 * buffer inside the workspace is used); out_hidden: NULL or fp32 [n][d_model];
 * first_token: NULL or int32 [1]. */
cb_status cb_full_prefill(cb_ctx* ctx, const int32_t* ids, int n, void* k_out, void* v_out, float* out_hidden,
                          int32_t* first_token, void* stream);

/* --------------------------------------------------------------------- decode
 * Generation after the blend: the response is produced from the fused KV ([P3] flow: "융합한 KV로
 * 응답 생성"; [P1] 実験結果 reports the decoding throughput that follows).  One step feeds one token
 * per sequence at position n_past: per layer its q, k, v are computed (RoPE at n_past), its K/V
 * are written to row n_past of the sequence's cache, its query attends causally to rows
 * 0..n_past (split over the keys across the GPU, then merged), then output projection and MLP;
 * the LM head's argmax (ties to the lowest id) is the next token.
 *   fused_k, fused_v: [n_layers][kv_capacity][n_kv_heads][head_dim] (a blend's fused cache made
 *     with kv_capacity >= the prompt length + the tokens to generate); rows 0..n_past-1 hold
 *     the context; n_past + 1 <= kv_capacity.
 *   out_hidden: NULL or fp32 [d_model]: the token's final hidden state (before the last norm). */
typedef struct {
  void* fused_k;
  void* fused_v;
  int kv_capacity;
  int n_past;
  float* out_hidden;
} cb_decode_seq;
/* One decode step of n_seq sequences (n_seq <= the workspace's max_requests and max_tokens;
 * 1, 2, 4, 7, 8 or 16 query heads per KV head; head_dim 64 or 128).  tokens: device int32 [n_seq];
 * out_tokens: device int32 [n_seq] (may be the same array as tokens).  No batch may be active. */
cb_status cb_decode_step(cb_ctx* ctx, const cb_decode_seq* seqs_host, int n_seq, const int32_t* tokens,
                         int32_t* out_tokens, void* stream);

/* --------------------------------------------------------------------- per-layer API
 * The pages' three calls ([P1] vLLMとの統合): fetch_kv(text, layer_id) loads a layer's
 * cached KV, prefill_layer(input_dict, KVCache) runs the partial prefill of the
 * selected tokens, synchronize() waits for the load.  Loading of layer i+1 overlaps
 * the recompute of layer i ([P1] パイプライン化の設計; [P3] "로딩과 재계산의 시간을 겹친다":
 * T_layer ~ max(T_load, T_recompute)). */

/* Plans a batch (sizes of every layer's sets are fixed here), gathers embeddings,
 * re-rotates every device-resident chunk into the fused caches (all layers). */
cb_status cb_blend_begin(cb_ctx* ctx, const cb_request* reqs, int n_req, const cb_blend_params* params,
                         void* stream);
/* Enqueues on copy_stream the host->device copy of layer `layer` of every
 * host-resident chunk of the batch into the fused caches and records an event. */
cb_status cb_fetch_kv(cb_ctx* ctx, int layer, void* copy_stream);
/* Host wait, with a deadline, for the copy of `layer` (CB_ERR_TIMEOUT when it passes). */
cb_status cb_synchronize(cb_ctx* ctx, int layer, int timeout_ms);
/* Layer `layer` of the blend on stream: waits (on the device) for its fetch,
 * re-rotates its host-staged keys in place, then QKV for R_i, deviation and
 * selection at check layers, scatter, attention, output projection and MLP. */
cb_status cb_prefill_layer(cb_ctx* ctx, int layer, void* stream);
/* cb_prefill_layer, preceded by cb_fetch_kv of the same layer on the same stream
 * when that layer has host-resident chunks (no overlap; the simple form). */
cb_status cb_blend_layer(cb_ctx* ctx, int layer, void* stream);
/* Final norm, LM head and argmax of each request's last token; writes outputs. */
cb_status cb_blend_finish(cb_ctx* ctx, void* stream);

/* Waits (deadline timeout_ms) for the work enqueued so far on `stream` and reports
 * the device status word: CB_OK, CB_ERR_NAN or CB_ERR_DEVICE.  Clears it; when it was
 * not zero, also clears (on `stream`) the workspace counters that a kernel which gave up
 * may have left set, so that later calls start from a clean state. */
cb_status cb_get_status(cb_ctx* ctx, void* stream, int timeout_ms);

/* --------------------------------------------------------------------- profiling
 * Per-phase device time of the batches run since the last cb_get_profile, from CUDA
 * events recorded on the compute stream around each phase (only while profiling is
 * enabled), and the number of kernels each phase launched (always counted). */
enum {
  CB_PH_BEGIN = 0,      /* embedding gather + re-rotation of device-resident chunks */
  CB_PH_STAGED_ROT,     /* in-place re-rotation of host-staged chunks */
  CB_PH_NORM,           /* RMSNorm (attention and MLP inputs) */
  CB_PH_QKV,            /* q/k/v projection GEMM */
  CB_PH_ROPE,           /* (unused: RoPE of fresh q and k runs inside the deviation and scatter) */
  CB_PH_DEVIATION,      /* KV deviation with RoPE of the fresh k (check layers) */
  CB_PH_SELECT,         /* HKVD top-k (check layers) */
  CB_PH_SCATTER,        /* RoPE of q and k, compaction, q conversion, KV scatter into the fused cache */
  CB_PH_ATTENTION,      /* causal sparse-query attention */
  CB_PH_OPROJ,          /* output projection GEMM + residual */
  CB_PH_GATEUP,         /* gate/up GEMM + SiLU-mul */
  CB_PH_DOWN,           /* down projection GEMM + residual */
  CB_PH_FINISH,         /* final norm, LM head, argmax, outputs */
  CB_N_PHASES
};
typedef struct {
  float ms[CB_N_PHASES];     /* summed device time per phase (0 when profiling was off) */
  int launches[CB_N_PHASES]; /* kernels launched per phase */
  int calls[CB_N_PHASES];    /* timed phase instances */
} cb_profile;
/* enable: 0 off, 1 per-phase events, 2 per-layer events only (below), 3 both.  Events cost
 * a few microseconds each, so per-layer times are taken without the phase events. */
cb_status cb_set_profiling(cb_ctx* ctx, int enable);
/* Waits for the recorded events, fills *out and resets the counters. */
cb_status cb_get_profile(cb_ctx* ctx, cb_profile* out);
/* Per-layer device times of the batches run at profiling level 2 or 3 since the last call,
 * for the overlap of loading and recompute ([P1] パイプライン化の設計: per layer
 * T ~ max(T_load, T_recompute)).  load_ms_host[i]: the copy stream's staging of layer
 * i's host-resident chunk KV, from its first copy to its last (0 when nothing of layer i
 * was staged).  compute_ms_host[i]: layer i on the compute stream, from after its wait
 * for the staged KV to its last kernel (the begin and finish steps are not a layer).
 * Host arrays [n_layers]; waits for the recorded events and releases them. */
cb_status cb_get_layer_profile(cb_ctx* ctx, int n_layers, float* load_ms_host, float* compute_ms_host);

/* A context runs one batch at a time and reuses its workspace for the next one:
 * issue consecutive batches on one stream (or synchronize between them). */

/* Sizes of the current batch's sets (host values known at cb_blend_begin):
 * counts_host [n_layers] receives |S_i| of request `request`. */
cb_status cb_plan_counts(const cb_ctx* ctx, int request, int32_t* counts_host);

#ifdef __cplusplus
}
#endif
#endif /* CACHEBLEND_H */
