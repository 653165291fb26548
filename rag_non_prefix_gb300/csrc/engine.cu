// Runtime of the blended prefill and the C ABI (include/cacheblend.h).
//
// A batch of prompts is planned on the host once (cb_blend_begin): because k_i is a pure
// function of the ratio schedule and the chunk sizes, the size of every layer's recompute
// set is known before any kernel runs, so the layer loop enqueues everything without a
// device->host round trip.  Rows of all requests are batched into one GEMM per weight.
//
// Device rows: R = input rows of the current layer (positions pos_R, requests req_R,
// hidden states h_R, fp32).  At a check layer the selection writes S (a subsequence of
// R); otherwise S = R.  After the layer, S becomes the next R.
//
// Host-resident chunk KV is staged layer by layer on a caller-provided copy stream into
// the fused cache (cb_fetch_kv) and re-rotated in place just before the layer runs, so
// loading layer i+1 overlaps recomputing layer i.
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace cb {
cudaError_t launch_attention_direct(const void* q, const int32_t* q_pos, int m, const void* k, const void* v,
                                   int n_kv, int n_heads, int n_kv_heads, int head_dim, void* out, cb_dtype dt,
                                   cudaStream_t s);
}

using namespace cb;

namespace {

thread_local std::string g_last_error;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t dtype_bytes(cb_dtype d) { return d == CB_BF16 ? 2 : 4; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int k_for_ratio(double r, int n_cached) { return cb_k_for_ratio(r, n_cached); }

// ----------------------------------------------------------------------------- chunk registry
struct ChunkEntry {
  uint64_t id = 0;
  const int32_t* ids = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  int n = 0;
  int on_host = 0;
  int state = 0;  // 0 empty, 1 live, 2 deleted
  const uint8_t* blob = nullptr;  // quantised chunk (bits 8 or 4) instead of k / v
  int bits = 0;
  size_t layer_bytes = 0;  // bytes of one layer block of the blob
};

// Open addressing with linear probing, keyed by a 64-bit chunk id (e.g. a text hash).
class Registry {
 public:
  Registry() : slots_(64) {}
  ChunkEntry* find(uint64_t id) {
    const size_t mask = slots_.size() - 1;
    for (size_t i = hash(id) & mask, probes = 0; probes < slots_.size(); i = (i + 1) & mask, ++probes) {
      ChunkEntry& e = slots_[i];
      if (e.state == 0) return nullptr;
      if (e.state == 1 && e.id == id) return &e;
    }
    return nullptr;
  }
  void put(const ChunkEntry& c) {
    if (ChunkEntry* e = find(c.id)) {
      *e = c;
      e->state = 1;
      return;
    }
    if ((live_ + dead_ + 1) * 2 > slots_.size()) rehash(slots_.size() * ((live_ + 1) * 4 > slots_.size() ? 2 : 1));
    const size_t mask = slots_.size() - 1;
    for (size_t i = hash(c.id) & mask;; i = (i + 1) & mask) {
      if (slots_[i].state != 1) {
        if (slots_[i].state == 2) --dead_;
        slots_[i] = c;
        slots_[i].state = 1;
        ++live_;
        return;
      }
    }
  }
  bool erase(uint64_t id) {
    ChunkEntry* e = find(id);
    if (!e) return false;
    e->state = 2;
    --live_;
    ++dead_;
    return true;
  }
  int size() const { return static_cast<int>(live_); }

 private:
  static uint64_t hash(uint64_t x) {  // SplitMix64 finaliser as a mixing function
    x ^= x >> 30;
    x *= 0xBF58476D1CE4E5B9ull;
    x ^= x >> 27;
    x *= 0x94D049BB133111EBull;
    return x ^ (x >> 31);
  }
  void rehash(size_t cap) {
    std::vector<ChunkEntry> old;
    old.swap(slots_);
    slots_.assign(cap, ChunkEntry{});
    live_ = dead_ = 0;
    for (const ChunkEntry& e : old)
      if (e.state == 1) put(e);
  }
  std::vector<ChunkEntry> slots_;
  size_t live_ = 0, dead_ = 0;
};

// ----------------------------------------------------------------------------- batch plan
struct SegHost {
  const ChunkEntry* chunk;  // null for the query segment
  int off, n;
};

struct ReqHost {
  int N = 0, Nc = 0;
  std::vector<SegHost> segs;
  void* fused_k = nullptr;
  void* fused_v = nullptr;
  long long layer_stride = 0;
  float* out_hidden = nullptr;
  int32_t* out_sel = nullptr;
  int32_t* out_sel_count = nullptr;
  int32_t* out_first_token = nullptr;
  const int32_t* query_ids = nullptr;
  int n_query = 0;
};

struct Batch {
  bool active = false;
  int n_req = 0, T = 0, L = 0;
  std::vector<ReqHost> reqs;
  std::vector<PlanEntry> plan;                 // [L][n_req]
  std::vector<int> rows_R, rows_S;             // per layer totals
  std::vector<int> check;                      // per layer
  std::vector<int> tile_off, tile_n;           // per layer (bf16 attention tiles)
  std::vector<int> host_seg_off, host_seg_n;   // per layer: in-place re-rotation of staged chunks
  int resident_segs = 0, resident_max_rows = 0, host_max_rows = 0;
  std::vector<char> fetched;
  bool any_host = false;
  int cur = 0;  // which row-array set holds R of the next layer
  int next_layer = 0;
  bool has_forced = false;
  int dev_mode = 0;
  // quantised chunks: resident ones are decoded at begin (all layers); host ones are copied
  // layer by layer into a ring of staging slots and decoded from there
  int codec_res_segs = 0, codec_res_max = 0;
  std::vector<int> codec_host_off, codec_host_n;  // per layer: range of host codec segments
  int codec_host_max = 0;
  int n_slots = 0;
  size_t slot_bytes = 0;
  struct StageCopy {
    const uint8_t* src;  // host blob of the chunk (layer 0 block)
    size_t layer_bytes;
    size_t slot_off;     // offset of this occurrence inside a slot
  };
  std::vector<StageCopy> stage;
  std::vector<char> slot_freed;  // per layer: the slot this layer used was released (decode enqueued)
  // tcgen05 attention: per request K/V tensor maps, sizes, and per layer the tile range of each request
  std::vector<CUtensorMap> kmaps, vmaps;
  std::vector<int> n_kv, one_layer;
  std::vector<int> req_tile_off;  // [L][n_req + 1]
};

}  // namespace

// ----------------------------------------------------------------------------- context
struct cb_ctx {
  cb_model_cfg cfg{};
  const void* embed = nullptr;
  const void* lm = nullptr;
  std::vector<const void*> wq, wk, wv, wo, wg, wu, wd;
  Registry reg;
  std::string last_error;

  // workspace
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  int ws_tokens = 0, ws_reqs = 0;
  int32_t* status = nullptr;
  float2* rope = nullptr;
  int32_t* tok = nullptr;
  int32_t* pos[2] = {nullptr, nullptr};
  int32_t* req[2] = {nullptr, nullptr};
  int32_t* src = nullptr;
  float* dev = nullptr;
  float* h[2] = {nullptr, nullptr};
  void* x = nullptr;
  float* qkv = nullptr;
  void* q = nullptr;
  void* attn = nullptr;
  void* act = nullptr;
  void* tmp_k = nullptr;
  void* tmp_v = nullptr;
  float* logits = nullptr;
  float* xlast = nullptr;
  float* dec_o = nullptr;
  float* att_o = nullptr;     // attention key-range split partials (see launch_attention_bf16)
  float2* att_ml = nullptr;
  int* att_cnt = nullptr;
  float2* dec_ml = nullptr;
  void* gemm_scratch = nullptr;
  size_t gemm_scratch_bytes = 0;
  uint8_t* meta = nullptr;  // plan, requests, tiles, segments, row ids ... (uploaded per batch)
  size_t meta_bytes = 0;

  // pinned staging of the per-batch metadata
  uint8_t* pinned = nullptr;
  size_t pinned_bytes = 0;
  cudaEvent_t pinned_ev = nullptr;
  bool pinned_pending = false;

  int32_t* status_host = nullptr;
  cudaEvent_t status_ev = nullptr;
  std::vector<cudaEvent_t> fetch_ev;

  // device views of the uploaded metadata for the active batch
  PlanEntry* d_plan = nullptr;
  ReqDev* d_reqs = nullptr;
  AttnTile* d_tiles = nullptr;
  RerotSeg* d_segs = nullptr;  // resident segments first, then the host ones per layer
  CodecSeg* d_csegs = nullptr;  // quantised chunks: resident segments first, then host ones per layer
  uint8_t* staging = nullptr;   // caller's staging ring for host-resident quantised chunks
  size_t staging_bytes = 0;
  std::vector<cudaEvent_t> slot_ev;  // per slot: its last decode was enqueued after this event
  int32_t* d_forced = nullptr;
  int32_t* d_lastrows = nullptr;
  int32_t* d_counts = nullptr;
  int32_t** d_first_ptrs = nullptr;
  int32_t* d_first = nullptr;

  Batch b;

  // profiling: events around phases (bit 0 of the level), around each layer's staging copies
  // and compute (bit 1), and launch counts (always)
  int prof = 0;
  std::vector<cudaEvent_t> ev_pool;
  struct Mark {
    int phase;
    cudaEvent_t a, b;
  };
  std::vector<Mark> marks;
  struct LayerMark {
    int layer;
    int load;  // 1: staging copies (copy stream), 0: the layer's compute (compute stream)
    cudaEvent_t a, b;
  };
  std::vector<LayerMark> layer_marks;
  int launches[CB_N_PHASES] = {};
  cudaEvent_t get_event() {
    if (!ev_pool.empty()) {
      cudaEvent_t e = ev_pool.back();
      ev_pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};

// Records a phase: optional events around the enqueued work and the kernel count.
struct PhaseScope {
  cb_ctx* ctx;
  int phase;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  PhaseScope(cb_ctx* c, int ph, cudaStream_t st, int kernels) : ctx(c), phase(ph), s(st) {
    ctx->launches[ph] += kernels;
    if (ctx->prof & 1) {
      a = ctx->get_event();
      cudaEventRecord(a, s);
    }
  }
  ~PhaseScope() {
    if (a) {
      cudaEvent_t b = ctx->get_event();
      cudaEventRecord(b, s);
      ctx->marks.push_back(cb_ctx::Mark{phase, a, b});
    }
  }
};

namespace {

cb_status fail(cb_ctx* ctx, cb_status s, const std::string& msg) {
  if (ctx) ctx->last_error = msg;
  g_last_error = msg;
  return s;
}
cb_status cuda_fail(cb_ctx* ctx, cudaError_t e, const char* where) {
  return fail(ctx, CB_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}
#define CB_CUDA(ctx, expr)                                 \
  do {                                                     \
    cudaError_t e_ = (expr);                               \
    if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #expr); \
  } while (0)

bool valid_cfg(const cb_model_cfg& c, std::string* why) {
  if (c.n_layers < 1 || c.d_model < 8 || c.n_heads < 1 || c.n_kv_heads < 1 || c.ffn_dim < 8 || c.vocab < 1 ||
      c.max_positions < 2) {
    *why = "non-positive model size";
    return false;
  }
  if (c.n_heads % c.n_kv_heads) {
    *why = "n_heads must be a multiple of n_kv_heads";
    return false;
  }
  if (!(c.rope_theta > 0) || !(c.rms_eps >= 0)) {
    *why = "bad rope_theta / rms_eps";
    return false;
  }
  if (c.dtype == CB_BF16) {
    if (c.head_dim != 128 || c.d_model % 128 || c.ffn_dim % 64) {
      *why = "bf16 needs head_dim 128, d_model % 128 == 0, ffn_dim % 64 == 0";
      return false;
    }
  } else if (c.dtype == CB_F32) {
    if (c.head_dim % 32 || c.head_dim > 128 || c.d_model % 8 || c.ffn_dim % 8) {
      *why = "fp32 needs head_dim a multiple of 32 up to 128, d_model and ffn_dim multiples of 8";
      return false;
    }
  } else {
    *why = "unknown dtype";
    return false;
  }
  return true;
}

struct WsLayout {
  size_t status, rope, tok, pos0, pos1, req0, req1, src, dev, h0, h1, x, qkv, q, attn, act, tmpk, tmpv, logits,
      xlast, gemm, dec_o, dec_ml, att_o, att_ml, att_cnt, meta, total, meta_bytes;
};

WsLayout ws_layout(const cb_model_cfg& c, int T, int R) {
  WsLayout w{};
  const size_t es = dtype_bytes(c.dtype);
  const size_t qw = static_cast<size_t>(c.n_heads) * c.head_dim, kvw = static_cast<size_t>(c.n_kv_heads) * c.head_dim;
  const size_t Tz = static_cast<size_t>(T);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  w.status = take(256);
  w.rope = take(static_cast<size_t>(c.max_positions) * (c.head_dim / 2) * sizeof(float2));
  w.tok = take(Tz * 4);
  w.pos0 = take(Tz * 4);
  w.pos1 = take(Tz * 4);
  w.req0 = take(Tz * 4);
  w.req1 = take(Tz * 4);
  w.src = take(Tz * 4);
  w.dev = take(Tz * 4);
  w.h0 = take(Tz * c.d_model * 4);
  w.h1 = take(Tz * c.d_model * 4);
  w.x = take(Tz * std::max<size_t>(c.d_model, 1) * es);
  w.qkv = take(Tz * (qw + 2 * kvw) * 4);
  w.q = take(Tz * qw * es);
  w.attn = take(Tz * qw * es);
  w.act = take(Tz * c.ffn_dim * es);
  w.tmpk = take(Tz * kvw * es);
  w.tmpv = take(Tz * kvw * es);
  w.logits = take(static_cast<size_t>(R) * c.vocab * 4);
  w.xlast = take(static_cast<size_t>(R) * c.d_model * 4);
  w.gemm = take(gemm_scratch_bytes());
  // decode attention: per (sequence, head, key range) partial outputs and (max, sum)
  const size_t dec_rows = static_cast<size_t>(R) * c.n_heads * decode_splits(c.max_positions);
  w.dec_o = take(dec_rows * c.head_dim * 4);
  w.dec_ml = take(dec_rows * sizeof(float2));
  // attention key-range splits of the sparse layers: partial outputs, (max, sum), counters
  w.att_o = take(static_cast<size_t>(ATTN_SPLIT_UNITS) * 2 * 128 * 128 * 4);
  w.att_ml = take(static_cast<size_t>(ATTN_SPLIT_UNITS) * 2 * 128 * sizeof(float2));
  w.att_cnt = take(static_cast<size_t>(ATTN_SPLIT_UNITS) * 4);
  // metadata: plan, requests, tiles, segments, forced sets, last rows, counts, first-token pointers
  const size_t L = c.n_layers;
  size_t m = 0;
  m += align_up(L * R * sizeof(PlanEntry), 256);
  m += align_up(R * sizeof(ReqDev), 256);
  m += align_up(L * (Tz + R) * sizeof(AttnTile), 256);
  m += align_up(2 * L * (Tz / 1 + R) * sizeof(RerotSeg) / 1, 256);  // segments: at most one per chunk per layer
  m += 256;                                                          // (the codec segments' own alignment)
  m += align_up(L * Tz * 4, 256);                                  // forced sets
  m += align_up(R * 4 + L * R * 4 + R * sizeof(void*) + R * 4, 256);
  m += align_up(2 * Tz * 4, 256);  // layer-0 positions and requests
  w.meta_bytes = m;
  w.meta = take(m);
  w.total = o;
  return w;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

cb_status wait_event_deadline(cb_ctx* ctx, cudaEvent_t ev, int timeout_ms) {
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return CB_OK;
    if (e != cudaErrorNotReady) return cuda_fail(ctx, e, "cudaEventQuery");
    const auto ms =
        std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count();
    if (timeout_ms >= 0 && ms >= timeout_ms) return fail(ctx, CB_ERR_TIMEOUT, "wait passed its deadline");
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

// Internal request description shared by the blend and the full prefill.
struct InReq {
  std::vector<SegHost> segs;  // cached segments then one query segment
  const int32_t* query_ids = nullptr;
  int n_query = 0;
  void* fused_k = nullptr;
  void* fused_v = nullptr;
  long long layer_stride = 0;
  float* out_hidden = nullptr;
  int32_t* out_sel = nullptr;
  int32_t* out_sel_count = nullptr;
  int32_t* out_first_token = nullptr;
};

cb_status ensure_pinned(cb_ctx* ctx, size_t bytes) {
  if (ctx->pinned_pending) {
    cb_status st = wait_event_deadline(ctx, ctx->pinned_ev, 60000);
    if (st != CB_OK) return st;
    ctx->pinned_pending = false;
  }
  if (bytes <= ctx->pinned_bytes) return CB_OK;
  if (ctx->pinned) cudaFreeHost(ctx->pinned);
  ctx->pinned = nullptr;
  ctx->pinned_bytes = 0;
  void* p = nullptr;
  CB_CUDA(ctx, cudaMallocHost(&p, bytes));
  ctx->pinned = static_cast<uint8_t*>(p);
  ctx->pinned_bytes = bytes;
  return CB_OK;
}

// Plans the batch, uploads metadata, gathers embeddings, re-rotates resident chunks.
// seam_tokens < 0: deviation-guided selection (ratios per layer, layer 0 on every token);
// seam_tokens >= 0: spatial seam repair, one fixed set (the last seam_tokens tokens of every
// cached chunk, and the query) recomputed at every layer from layer 0 on, no check layers.
cb_status begin_impl(cb_ctx* ctx, std::vector<InReq>& in, const double* ratios, int dev_mode,
                     const int32_t* const* forced, int seam_tokens, cudaStream_t s) {
  const cb_model_cfg& c = ctx->cfg;
  Batch& b = ctx->b;
  if (b.active) return fail(ctx, CB_ERR_STATE, "a batch is already active (finish it first)");
  if (!ctx->ws) return fail(ctx, CB_ERR_WORKSPACE, "no workspace bound");
  const int n_req = static_cast<int>(in.size());
  const int L = c.n_layers;
  if (n_req < 1 || n_req > ctx->ws_reqs) return fail(ctx, CB_ERR_WORKSPACE, "too many requests for the workspace");
  const size_t kvw = static_cast<size_t>(c.n_kv_heads) * c.head_dim;
  const size_t es = dtype_bytes(c.dtype);

  b = Batch{};
  b.dev_mode = dev_mode;
  b.n_req = n_req;
  b.L = L;
  b.reqs.resize(n_req);
  int T = 0;
  for (int r = 0; r < n_req; ++r) {
    ReqHost& rh = b.reqs[r];
    int off = 0;
    for (SegHost sg : in[r].segs) {
      sg.off = off;
      off += sg.n;
      rh.segs.push_back(sg);
      if (sg.chunk && sg.chunk->on_host) b.any_host = true;
    }
    rh.Nc = off;
    rh.N = off + in[r].n_query;
    rh.query_ids = in[r].query_ids;
    rh.n_query = in[r].n_query;
    rh.fused_k = in[r].fused_k;
    rh.fused_v = in[r].fused_v;
    rh.layer_stride = in[r].layer_stride;
    rh.out_hidden = in[r].out_hidden;
    rh.out_sel = in[r].out_sel;
    rh.out_sel_count = in[r].out_sel_count;
    rh.out_first_token = in[r].out_first_token;
    if (rh.N > c.max_positions) return fail(ctx, CB_ERR_SHAPE, "prompt longer than max_positions");
    T += rh.N;
  }
  if (T > ctx->ws_tokens) return fail(ctx, CB_ERR_WORKSPACE, "prompt tokens exceed the workspace");
  b.T = T;
  const bool seam = seam_tokens >= 0;
  // layer-0 rows of each request: every token, or (seam repair) the seam tokens and the query
  std::vector<std::vector<int32_t>> rows0(n_req);
  int T0 = 0;
  for (int r = 0; r < n_req; ++r) {
    const ReqHost& rh = b.reqs[r];
    std::vector<int32_t>& v = rows0[r];
    if (seam) {
      for (const SegHost& sg : rh.segs) {
        const int keep = std::min(seam_tokens, sg.n);
        for (int j = sg.n - keep; j < sg.n; ++j) v.push_back(sg.off + j);
      }
      for (int j = rh.Nc; j < rh.N; ++j) v.push_back(j);
    } else {
      v.resize(rh.N);
      for (int j = 0; j < rh.N; ++j) v[j] = j;
    }
    T0 += static_cast<int>(v.size());
  }

  // ---- per-layer plan (sizes are host-known)
  b.plan.resize(static_cast<size_t>(L) * n_req);
  b.rows_R.assign(L, 0);
  b.rows_S.assign(L, 0);
  b.check.assign(L, 0);
  std::vector<int> rN(n_req), rC(n_req);  // rows of R, cached rows of R
  for (int r = 0; r < n_req; ++r) {
    rN[r] = static_cast<int>(rows0[r].size());
    rC[r] = rN[r] - b.reqs[r].n_query;
  }
  std::vector<int32_t> forced_all;
  for (int i = 0; i < L; ++i) {
    const bool chk = !seam && ratios && ratios[i] >= 0.0;
    b.check[i] = chk ? 1 : 0;
    int roff = 0, soff = 0;
    for (int r = 0; r < n_req; ++r) {
      PlanEntry& pe = b.plan[static_cast<size_t>(i) * n_req + r];
      pe.r_off = roff;
      pe.r_n = rN[r];
      pe.check = chk ? 1 : 0;
      pe.forced_off = -1;
      int kept_cached = rC[r];
      if (chk) {
        if (forced && forced[i]) {
          // forced lists hold, per request, the cached part of S_i; requests are laid out
          // one after the other, each list prefixed by its length
          const int32_t* fl = forced[i];
          int at = 0;
          for (int rr = 0; rr < r; ++rr) at += 1 + fl[at];
          const int cnt = fl[at];
          if (cnt < 0 || cnt > rC[r]) return fail(ctx, CB_ERR_INVALID_ARG, "forced set larger than the candidates");
          for (int j = 0; j < cnt; ++j) {
            const int v = fl[at + 1 + j];
            if (v < 0 || v >= b.reqs[r].Nc || (j && v <= fl[at + j]))
              return fail(ctx, CB_ERR_INVALID_ARG, "forced set must be sorted cached token indices");
          }
          pe.forced_off = static_cast<int>(forced_all.size());
          forced_all.insert(forced_all.end(), fl + at + 1, fl + at + 1 + cnt);
          kept_cached = cnt;
          b.has_forced = true;
        } else {
          kept_cached = std::min(k_for_ratio(ratios[i], b.reqs[r].Nc), rC[r]);
        }
        pe.k = kept_cached;
        pe.s_n = kept_cached + b.reqs[r].n_query;
      } else {
        pe.k = 0;
        pe.s_n = rN[r];
      }
      pe.s_off = soff;
      roff += pe.r_n;
      soff += pe.s_n;
      rN[r] = pe.s_n;
      rC[r] = kept_cached;
    }
    b.rows_R[i] = roff;
    b.rows_S[i] = soff;
  }

  // ---- attention tiles per layer (request by request), and the K/V tensor maps
  std::vector<AttnTile> tiles;
  b.tile_off.assign(L, 0);
  b.tile_n.assign(L, 0);
  b.req_tile_off.assign(static_cast<size_t>(L) * (n_req + 1), 0);
  const int QT = attention_tile_rows(c.n_heads, c.n_kv_heads, c.dtype);
  for (int i = 0; i < L; ++i) {
    b.tile_off[i] = static_cast<int>(tiles.size());
    if (c.dtype == CB_BF16) {
      for (int r = 0; r < n_req; ++r) {
        b.req_tile_off[static_cast<size_t>(i) * (n_req + 1) + r] = static_cast<int>(tiles.size()) - b.tile_off[i];
        const PlanEntry& pe = b.plan[static_cast<size_t>(i) * n_req + r];
        for (int q0 = 0; q0 < pe.s_n; q0 += QT) tiles.push_back(AttnTile{r, pe.s_off + q0, std::min(QT, pe.s_n - q0), 0});
      }
      b.req_tile_off[static_cast<size_t>(i) * (n_req + 1) + n_req] = static_cast<int>(tiles.size()) - b.tile_off[i];
    }
    b.tile_n[i] = static_cast<int>(tiles.size()) - b.tile_off[i];
  }
  if (c.dtype == CB_BF16) {
    b.kmaps.resize(n_req);
    b.vmaps.resize(n_req);
    b.n_kv.resize(n_req);
    b.one_layer.resize(n_req);
    for (int r = 0; r < n_req; ++r) {
      const ReqHost& rh = b.reqs[r];
      if (!encode_kv_map(&b.kmaps[r], rh.fused_k, L, rh.N, c.n_kv_heads, rh.layer_stride) ||
          !encode_kv_map(&b.vmaps[r], rh.fused_v, L, rh.N, c.n_kv_heads, rh.layer_stride))
        return fail(ctx, CB_ERR_INVALID_ARG, "cannot describe the fused cache to the tensor memory accelerator");
      b.n_kv[r] = rh.N;
      b.one_layer[r] = rh.layer_stride == 0 ? 1 : 0;
    }
  }

  // ---- re-rotation segments: resident chunks (all layers, once) then host chunks per layer
  std::vector<RerotSeg> segs;
  for (int i = 0; i < L; ++i)
    for (int r = 0; r < n_req; ++r) {
      const ReqHost& rh = b.reqs[r];
      for (const SegHost& sg : rh.segs) {
        if (!sg.chunk || sg.chunk->on_host || sg.chunk->bits) continue;
        const size_t so = static_cast<size_t>(i) * sg.n * kvw * es;
        const size_t dof = (static_cast<size_t>(i) * rh.layer_stride + static_cast<size_t>(sg.off) * kvw) * es;
        segs.push_back(RerotSeg{static_cast<const uint8_t*>(sg.chunk->k) + so,
                                static_cast<const uint8_t*>(sg.chunk->v) + so, static_cast<uint8_t*>(rh.fused_k) + dof,
                                static_cast<uint8_t*>(rh.fused_v) + dof, sg.n, sg.off});
        b.resident_max_rows = std::max(b.resident_max_rows, sg.n);
      }
    }
  b.resident_segs = static_cast<int>(segs.size());
  b.host_seg_off.assign(L, 0);
  b.host_seg_n.assign(L, 0);
  for (int i = 0; i < L; ++i) {
    b.host_seg_off[i] = static_cast<int>(segs.size());
    for (int r = 0; r < n_req; ++r) {
      const ReqHost& rh = b.reqs[r];
      for (const SegHost& sg : rh.segs) {
        if (!sg.chunk || !sg.chunk->on_host || sg.chunk->bits || sg.off == 0) continue;  // offset 0: R(0) = I
        const size_t dof = (static_cast<size_t>(i) * rh.layer_stride + static_cast<size_t>(sg.off) * kvw) * es;
        uint8_t* kd = static_cast<uint8_t*>(rh.fused_k) + dof;
        segs.push_back(RerotSeg{kd, nullptr, kd, nullptr, sg.n, sg.off});
        b.host_max_rows = std::max(b.host_max_rows, sg.n);
      }
    }
    b.host_seg_n[i] = static_cast<int>(segs.size()) - b.host_seg_off[i];
  }

  // ---- quantised chunks: resident blocks decoded at begin; host blocks staged per layer into
  //      slot (layer mod n_slots) of the staging ring, one region per chunk occurrence
  std::vector<CodecSeg> csegs;
  for (int i = 0; i < L; ++i)
    for (int r = 0; r < n_req; ++r) {
      const ReqHost& rh = b.reqs[r];
      for (const SegHost& sg : rh.segs) {
        if (!sg.chunk || !sg.chunk->bits || sg.chunk->on_host) continue;
        const size_t dof = (static_cast<size_t>(i) * rh.layer_stride + static_cast<size_t>(sg.off) * kvw) * es;
        csegs.push_back(CodecSeg{sg.chunk->blob + static_cast<size_t>(i) * sg.chunk->layer_bytes,
                                 static_cast<uint8_t*>(rh.fused_k) + dof, static_cast<uint8_t*>(rh.fused_v) + dof,
                                 sg.n, sg.off, sg.chunk->bits, 0});
        b.codec_res_max = std::max(b.codec_res_max, sg.n);
      }
    }
  b.codec_res_segs = static_cast<int>(csegs.size());
  std::vector<std::pair<int, const SegHost*>> staged_occ;  // (request, segment) of host codec chunks
  for (int r = 0; r < n_req; ++r)
    for (const SegHost& sg : b.reqs[r].segs)
      if (sg.chunk && sg.chunk->bits && sg.chunk->on_host) {
        b.stage.push_back(Batch::StageCopy{sg.chunk->blob, sg.chunk->layer_bytes, b.slot_bytes});
        b.slot_bytes += sg.chunk->layer_bytes;
        staged_occ.push_back({r, &sg});
      }
  b.codec_host_off.assign(L, 0);
  b.codec_host_n.assign(L, 0);
  b.slot_freed.assign(L, 0);
  if (!b.stage.empty()) {
    if (!ctx->staging || ctx->staging_bytes < b.slot_bytes)
      return fail(ctx, CB_ERR_WORKSPACE, "the staging buffer (cb_set_staging) holds less than one layer of the "
                                         "batch's host-resident quantised chunks");
    b.n_slots = static_cast<int>(std::min<size_t>(L, ctx->staging_bytes / b.slot_bytes));
    while (static_cast<int>(ctx->slot_ev.size()) < b.n_slots) {
      cudaEvent_t e = nullptr;
      CB_CUDA(ctx, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
      ctx->slot_ev.push_back(e);
    }
    for (int i = 0; i < L; ++i) {
      b.codec_host_off[i] = static_cast<int>(csegs.size());
      const uint8_t* slot = ctx->staging + static_cast<size_t>(i % b.n_slots) * b.slot_bytes;
      for (size_t k = 0; k < staged_occ.size(); ++k) {
        const ReqHost& rh = b.reqs[staged_occ[k].first];
        const SegHost& sg = *staged_occ[k].second;
        const size_t dof = (static_cast<size_t>(i) * rh.layer_stride + static_cast<size_t>(sg.off) * kvw) * es;
        csegs.push_back(CodecSeg{slot + b.stage[k].slot_off, static_cast<uint8_t*>(rh.fused_k) + dof,
                                 static_cast<uint8_t*>(rh.fused_v) + dof, sg.n, sg.off, sg.chunk->bits, 0});
        b.codec_host_max = std::max(b.codec_host_max, sg.n);
      }
      b.codec_host_n[i] = static_cast<int>(csegs.size()) - b.codec_host_off[i];
    }
  }

  // ---- request descriptors, layer-0 rows, last rows, counts, first-token pointers
  std::vector<ReqDev> rd(n_req);
  std::vector<int32_t> pos0(T0), req0(T0), lastrows(n_req), counts(static_cast<size_t>(L) * n_req);
  std::vector<int32_t*> firsts(n_req);
  {
    int at = 0;
    for (int r = 0; r < n_req; ++r) {
      const ReqHost& rh = b.reqs[r];
      rd[r] = ReqDev{rh.fused_k, rh.fused_v, rh.layer_stride, rh.N, rh.Nc};
      for (size_t j = 0; j < rows0[r].size(); ++j) {
        pos0[at + j] = rows0[r][j];
        req0[at + j] = r;
      }
      at += static_cast<int>(rows0[r].size());
      const PlanEntry& last = b.plan[static_cast<size_t>(L - 1) * n_req + r];
      lastrows[r] = last.s_off + last.s_n - 1;
      firsts[r] = rh.out_first_token;
      for (int i = 0; i < L; ++i) counts[static_cast<size_t>(i) * n_req + r] = b.plan[static_cast<size_t>(i) * n_req + r].s_n;
    }
  }

  // ---- pack into pinned staging, one async upload
  const size_t szPlan = align_up(b.plan.size() * sizeof(PlanEntry), 256);
  const size_t szReq = align_up(rd.size() * sizeof(ReqDev), 256);
  const size_t szTiles = align_up(std::max<size_t>(1, tiles.size()) * sizeof(AttnTile), 256);
  const size_t szSegs = align_up(std::max<size_t>(1, segs.size()) * sizeof(RerotSeg), 256);
  const size_t szCsegs = align_up(std::max<size_t>(1, csegs.size()) * sizeof(CodecSeg), 256);
  const size_t szForced = align_up(std::max<size_t>(1, forced_all.size()) * 4, 256);
  const size_t szSmall = align_up(lastrows.size() * 4, 256) + align_up(counts.size() * 4, 256) +
                         align_up(firsts.size() * sizeof(void*), 256) + align_up(n_req * 4, 256);
  const size_t szRows = align_up(T0 * 4, 256) * 2;
  const size_t total = szPlan + szReq + szTiles + szSegs + szCsegs + szForced + szSmall + szRows;
  if (total > ctx->meta_bytes) return fail(ctx, CB_ERR_WORKSPACE, "batch metadata exceeds the workspace");
  cb_status st = ensure_pinned(ctx, total);
  if (st != CB_OK) return st;
  uint8_t* hp = ctx->pinned;
  uint8_t* dp = ctx->meta;
  size_t o = 0;
  auto put = [&](const void* src, size_t bytes, size_t slot) -> uint8_t* {
    if (bytes) std::memcpy(hp + o, src, bytes);
    uint8_t* d = dp + o;
    o += slot;
    return d;
  };
  ctx->d_plan = reinterpret_cast<PlanEntry*>(put(b.plan.data(), b.plan.size() * sizeof(PlanEntry), szPlan));
  ctx->d_reqs = reinterpret_cast<ReqDev*>(put(rd.data(), rd.size() * sizeof(ReqDev), szReq));
  ctx->d_tiles = reinterpret_cast<AttnTile*>(put(tiles.data(), tiles.size() * sizeof(AttnTile), szTiles));
  ctx->d_segs = reinterpret_cast<RerotSeg*>(put(segs.data(), segs.size() * sizeof(RerotSeg), szSegs));
  ctx->d_csegs = reinterpret_cast<CodecSeg*>(put(csegs.data(), csegs.size() * sizeof(CodecSeg), szCsegs));
  ctx->d_forced = reinterpret_cast<int32_t*>(put(forced_all.data(), forced_all.size() * 4, szForced));
  ctx->d_lastrows = reinterpret_cast<int32_t*>(put(lastrows.data(), lastrows.size() * 4, align_up(lastrows.size() * 4, 256)));
  ctx->d_counts = reinterpret_cast<int32_t*>(put(counts.data(), counts.size() * 4, align_up(counts.size() * 4, 256)));
  ctx->d_first_ptrs = reinterpret_cast<int32_t**>(put(firsts.data(), firsts.size() * sizeof(void*), align_up(firsts.size() * sizeof(void*), 256)));
  ctx->d_first = reinterpret_cast<int32_t*>(put(nullptr, 0, align_up(n_req * 4, 256)));
  int32_t* d_pos0 = reinterpret_cast<int32_t*>(put(pos0.data(), T0 * 4, align_up(T0 * 4, 256)));
  int32_t* d_req0 = reinterpret_cast<int32_t*>(put(req0.data(), T0 * 4, align_up(T0 * 4, 256)));
  CB_CUDA(ctx, cudaMemcpyAsync(ctx->meta, ctx->pinned, o, cudaMemcpyHostToDevice, s));
  CB_CUDA(ctx, cudaEventRecord(ctx->pinned_ev, s));
  ctx->pinned_pending = true;
  CB_CUDA(ctx, cudaMemcpyAsync(ctx->pos[0], d_pos0, T0 * 4, cudaMemcpyDeviceToDevice, s));
  CB_CUDA(ctx, cudaMemcpyAsync(ctx->req[0], d_req0, T0 * 4, cudaMemcpyDeviceToDevice, s));

  // ---- token ids of every layer-0 row (chunk ids from the registry, then the query), embeddings
  {
    int at = 0;
    for (int r = 0; r < n_req; ++r) {
      const ReqHost& rh = b.reqs[r];
      for (const SegHost& sg : rh.segs) {
        const int keep = seam ? std::min(seam_tokens, sg.n) : sg.n;
        if (keep > 0)
          CB_CUDA(ctx, cudaMemcpyAsync(ctx->tok + at, sg.chunk->ids + (sg.n - keep), keep * 4,
                                       cudaMemcpyDeviceToDevice, s));
        at += keep;
      }
      CB_CUDA(ctx, cudaMemcpyAsync(ctx->tok + at, rh.query_ids, rh.n_query * 4, cudaMemcpyDeviceToDevice, s));
      at += rh.n_query;
    }
  }
  {
    PhaseScope ps(ctx, CB_PH_BEGIN, s, 1 + (b.resident_segs > 0 ? 1 : 0) + (b.codec_res_segs > 0 ? 1 : 0));
    CB_CUDA(ctx, launch_embed(ctx->embed, ctx->tok, T0, c.d_model, c.vocab, c.dtype, ctx->h[0], ctx->status, s));
    if (b.resident_segs > 0)
      CB_CUDA(ctx, launch_rerotate(ctx->d_segs, b.resident_segs, b.resident_max_rows, c.n_kv_heads, c.head_dim,
                                   ctx->rope, c.max_positions, c.dtype, ctx->status, s));
    if (b.codec_res_segs > 0)
      CB_CUDA(ctx, launch_codec_decode(ctx->d_csegs, b.codec_res_segs, b.codec_res_max, c.n_kv_heads, c.head_dim,
                                       ctx->rope, c.max_positions, c.dtype, ctx->status, s));
  }
  b.fetched.assign(L, 0);
  b.cur = 0;
  b.next_layer = 0;
  b.active = true;
  return CB_OK;
}

cb_status fetch_impl(cb_ctx* ctx, int layer, cudaStream_t cs) {
  Batch& b = ctx->b;
  const cb_model_cfg& c = ctx->cfg;
  if (!b.active) return fail(ctx, CB_ERR_STATE, "no active batch");
  if (layer < 0 || layer >= b.L) return fail(ctx, CB_ERR_INVALID_ARG, "layer out of range");
  const size_t kvw = static_cast<size_t>(c.n_kv_heads) * c.head_dim;
  const size_t es = dtype_bytes(c.dtype);
  cudaEvent_t load_a = nullptr;  // per-layer profiling: from the first copy of the layer
  if (!b.stage.empty()) {
    const int slot = layer % b.n_slots;
    if (layer >= b.n_slots) {
      if (!b.slot_freed[layer - b.n_slots])
        return fail(ctx, CB_ERR_STATE, "staging slot still in use: enqueue cb_prefill_layer of layer - n_slots first");
      CB_CUDA(ctx, cudaStreamWaitEvent(cs, ctx->slot_ev[slot], 0));
    }
    uint8_t* dst = ctx->staging + static_cast<size_t>(slot) * b.slot_bytes;
    if ((ctx->prof & 2) && !load_a) {
      load_a = ctx->get_event();
      CB_CUDA(ctx, cudaEventRecord(load_a, cs));
    }
    for (const Batch::StageCopy& sc : b.stage)
      CB_CUDA(ctx, cudaMemcpyAsync(dst + sc.slot_off, sc.src + static_cast<size_t>(layer) * sc.layer_bytes,
                                   sc.layer_bytes, cudaMemcpyHostToDevice, cs));
  }
  for (const ReqHost& rh : b.reqs)
    for (const SegHost& sg : rh.segs) {
      if (!sg.chunk || !sg.chunk->on_host || sg.chunk->bits) continue;
      const size_t bytes = static_cast<size_t>(sg.n) * kvw * es;
      const size_t so = static_cast<size_t>(layer) * bytes;
      const size_t dof = (static_cast<size_t>(layer) * rh.layer_stride + static_cast<size_t>(sg.off) * kvw) * es;
      if ((ctx->prof & 2) && !load_a) {
        load_a = ctx->get_event();
        CB_CUDA(ctx, cudaEventRecord(load_a, cs));
      }
      CB_CUDA(ctx, cudaMemcpyAsync(static_cast<uint8_t*>(rh.fused_k) + dof,
                                   static_cast<const uint8_t*>(sg.chunk->k) + so, bytes, cudaMemcpyHostToDevice, cs));
      CB_CUDA(ctx, cudaMemcpyAsync(static_cast<uint8_t*>(rh.fused_v) + dof,
                                   static_cast<const uint8_t*>(sg.chunk->v) + so, bytes, cudaMemcpyHostToDevice, cs));
    }
  if (load_a) {
    cudaEvent_t load_b = ctx->get_event();
    CB_CUDA(ctx, cudaEventRecord(load_b, cs));
    ctx->layer_marks.push_back(cb_ctx::LayerMark{layer, 1, load_a, load_b});
  }
  CB_CUDA(ctx, cudaEventRecord(ctx->fetch_ev[layer], cs));
  b.fetched[layer] = 1;
  return CB_OK;
}

// Per-layer profiling (bit 1 of the level): events around one layer's work on the compute stream,
// from after its wait for staged KV to its last kernel.
struct LayerScope {
  cb_ctx* ctx;
  int layer;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  LayerScope(cb_ctx* c, int i, cudaStream_t st) : ctx(c), layer(i), s(st) {
    if (ctx->prof & 2) {
      a = ctx->get_event();
      cudaEventRecord(a, s);
    }
  }
  ~LayerScope() {
    if (a) {
      cudaEvent_t b = ctx->get_event();
      cudaEventRecord(b, s);
      ctx->layer_marks.push_back(cb_ctx::LayerMark{layer, 0, a, b});
    }
  }
};

cb_status layer_impl(cb_ctx* ctx, int i, cudaStream_t s) {
  Batch& b = ctx->b;
  const cb_model_cfg& c = ctx->cfg;
  if (!b.active) return fail(ctx, CB_ERR_STATE, "no active batch");
  if (i != b.next_layer) return fail(ctx, CB_ERR_STATE, "layers must run in order");
  if (b.any_host) {
    if (!b.fetched[i]) return fail(ctx, CB_ERR_STATE, "cb_fetch_kv was not called for this layer");
    CB_CUDA(ctx, cudaStreamWaitEvent(s, ctx->fetch_ev[i], 0));
  }
  LayerScope layer_scope(ctx, i, s);
  if (b.any_host) {
    if (b.host_seg_n[i] > 0) {
      PhaseScope ps(ctx, CB_PH_STAGED_ROT, s, 1);
      CB_CUDA(ctx, launch_rerotate(ctx->d_segs + b.host_seg_off[i], b.host_seg_n[i], b.host_max_rows, c.n_kv_heads,
                                   c.head_dim, ctx->rope, c.max_positions, c.dtype, ctx->status, s));
    }
    if (b.codec_host_n[i] > 0) {
      PhaseScope ps(ctx, CB_PH_STAGED_ROT, s, 1);
      CB_CUDA(ctx, launch_codec_decode(ctx->d_csegs + b.codec_host_off[i], b.codec_host_n[i], b.codec_host_max,
                                       c.n_kv_heads, c.head_dim, ctx->rope, c.max_positions, c.dtype, ctx->status, s));
      CB_CUDA(ctx, cudaEventRecord(ctx->slot_ev[i % b.n_slots], s));  // the slot may be refilled after this
      b.slot_freed[i] = 1;
    }
  }
  const int H = c.n_heads, Hkv = c.n_kv_heads, dh = c.head_dim, d = c.d_model;
  const int qw = H * dh, kvw = Hkv * dh;
  const int Rn = b.rows_R[i], Sn = b.rows_S[i];
  const int cur = b.cur;
  int32_t* posR = ctx->pos[cur];
  int32_t* reqR = ctx->req[cur];
  float* hR = ctx->h[cur];
  // 1. QKV of R: x = RMSNorm(h_R); [q | k | v] = x W^T (RoPE of q and k is applied where
  //    they are consumed: the deviation and the scatter).  A layer without a check keeps its
  //    set, so the scatter needs no compaction: RoPE and the scatter run in the GEMM's
  //    epilogue where the projection runs on CTA pairs.
  {
    PhaseScope ps(ctx, CB_PH_NORM, s, 1);
    CB_CUDA(ctx, launch_rmsnorm(hR, Rn, d, c.rms_eps, ctx->x, c.dtype, s));
  }
  bool fused = false;
  if (!b.check[i] && c.dtype == CB_BF16 && dh == 128 && qkv_fusion()) {
    PhaseScope ps(ctx, CB_PH_QKV, s, 1);
    const QkvRope qr{posR, reqR, ctx->d_reqs, ctx->rope, i, c.max_positions, ctx->q, qw, kvw};
    const cudaError_t e = launch_qkv_rope_gemm(ctx->x, ctx->wq[i], ctx->wk[i], ctx->wv[i], Rn, d, qr, ctx->status,
                                               ctx->gemm_scratch, ctx->gemm_scratch_bytes, s);
    if (e != cudaErrorNotSupported) CB_CUDA(ctx, e);
    fused = e == cudaSuccess;
  }
  if (!fused) {
    PhaseScope ps(ctx, CB_PH_QKV, s, 1);
    CB_CUDA(ctx, launch_gemm(ctx->x, ctx->wq[i], ctx->wk[i], ctx->wv[i], qw, qw + kvw, ctx->qkv, Rn, qw + 2 * kvw, d,
                             qw + 2 * kvw, 0, c.dtype, ctx->status, ctx->gemm_scratch, ctx->gemm_scratch_bytes, s));
  }
  int32_t* posS = posR;
  int32_t* reqS = reqR;
  float* hS = hR;
  const PlanEntry* plan_i = ctx->d_plan + static_cast<size_t>(i) * b.n_req;
  if (b.check[i]) {
    // 2. deviation of the cached rows of R against the fused cache, then top-k per request
    {
      PhaseScope ps(ctx, CB_PH_DEVIATION, s, 1);
      CB_CUDA(ctx, launch_deviation_rows(ctx->qkv, Rn, posR, reqR, ctx->d_reqs, i, H, Hkv, dh, b.dev_mode, ctx->rope,
                                         c.max_positions, c.dtype, ctx->dev, ctx->status, s));
    }
    posS = ctx->pos[cur ^ 1];
    reqS = ctx->req[cur ^ 1];
    hS = ctx->h[cur ^ 1];
    {
      PhaseScope ps(ctx, CB_PH_SELECT, s, 1);
      CB_CUDA(ctx, launch_select_batched(ctx->dev, posR, plan_i, ctx->d_reqs, ctx->d_forced, b.n_req, ctx->src, posS,
                                         reqS, ctx->status, s));
    }
    // 3. compact S, scatter fresh K/V of S into the fused cache, q of S in the model dtype
    {
      PhaseScope ps(ctx, CB_PH_SCATTER, s, 1);
      CB_CUDA(ctx, launch_post_qkv(ctx->qkv, Sn, ctx->src, posS, reqS, ctx->d_reqs, i, H, Hkv, dh, ctx->rope,
                                   c.max_positions, c.dtype, ctx->q, hR, hS, d, ctx->status, s));
    }
    b.cur ^= 1;
  } else if (!fused) {
    PhaseScope ps(ctx, CB_PH_SCATTER, s, 1);
    CB_CUDA(ctx, launch_post_qkv(ctx->qkv, Sn, nullptr, posS, reqS, ctx->d_reqs, i, H, Hkv, dh, ctx->rope,
                                 c.max_positions, c.dtype, ctx->q, hR, hR, d, ctx->status, s));
  }
  // 4. causal attention of S over the fused cache
  {
    PhaseScope ps(ctx, CB_PH_ATTENTION, s, 1);
    if (c.dtype == CB_BF16)
      CB_CUDA(ctx, launch_attention_bf16(ctx->q, posS, ctx->d_tiles + b.tile_off[i],
                                         b.req_tile_off.data() + static_cast<size_t>(i) * (b.n_req + 1),
                                         b.kmaps.data(), b.vmaps.data(), b.n_kv.data(), b.one_layer.data(), b.n_req,
                                         i, H, Hkv, ctx->attn, ctx->status, ctx->att_o, ctx->att_ml, ctx->att_cnt,
                                         s));
    else
      CB_CUDA(ctx, launch_attention(ctx->q, posS, reqS, ctx->d_reqs, nullptr, Sn, i, H, Hkv, dh, ctx->attn, c.dtype,
                                    s));
  }
  // 5. h_S += attn W_o^T;  h_S += W_down(SiLU(x W_gate^T) * x W_up^T), x = RMSNorm(h_S)
  {
    PhaseScope ps(ctx, CB_PH_OPROJ, s, 1);
    CB_CUDA(ctx, launch_gemm(ctx->attn, ctx->wo[i], nullptr, nullptr, d, d, hS, Sn, d, qw, d, 1, c.dtype, ctx->status,
                             ctx->gemm_scratch, ctx->gemm_scratch_bytes, s));
  }
  {
    PhaseScope ps(ctx, CB_PH_NORM, s, 1);
    CB_CUDA(ctx, launch_rmsnorm(hS, Sn, d, c.rms_eps, ctx->x, c.dtype, s));
  }
  {
    PhaseScope ps(ctx, CB_PH_GATEUP, s, 1);
    CB_CUDA(ctx, launch_gemm(ctx->x, ctx->wg[i], ctx->wu[i], nullptr, 0, 0, ctx->act, Sn, 2 * c.ffn_dim, d,
                             c.ffn_dim, 2, c.dtype, ctx->status, ctx->gemm_scratch, ctx->gemm_scratch_bytes, s));
  }
  {
    PhaseScope ps(ctx, CB_PH_DOWN, s, 1);
    CB_CUDA(ctx, launch_gemm(ctx->act, ctx->wd[i], nullptr, nullptr, d, d, hS, Sn, d, c.ffn_dim, d, 1, c.dtype,
                             ctx->status, ctx->gemm_scratch, ctx->gemm_scratch_bytes, s));
  }
  // 6. optional per-layer sets
  for (int r = 0; r < b.n_req; ++r) {
    const ReqHost& rh = b.reqs[r];
    if (!rh.out_sel) continue;
    const PlanEntry& pe = b.plan[static_cast<size_t>(i) * b.n_req + r];
    CB_CUDA(ctx, cudaMemcpyAsync(rh.out_sel + static_cast<size_t>(i) * rh.N, posS + pe.s_off, pe.s_n * 4,
                                 cudaMemcpyDeviceToDevice, s));
  }
  b.next_layer = i + 1;
  return CB_OK;
}

cb_status finish_impl(cb_ctx* ctx, cudaStream_t s) {
  Batch& b = ctx->b;
  const cb_model_cfg& c = ctx->cfg;
  if (!b.active) return fail(ctx, CB_ERR_STATE, "no active batch");
  if (b.next_layer != b.L) return fail(ctx, CB_ERR_STATE, "not every layer has run");
  const int cur = b.cur;
  float* hS = ctx->h[cur];
  int32_t* posS = ctx->pos[cur];
  int n_hidden = 0;
  for (const ReqHost& rh : b.reqs) n_hidden += rh.out_hidden ? 1 : 0;
  PhaseScope ps(ctx, CB_PH_FINISH, s, 2 + (b.n_req + 15) / 16 + n_hidden);
  CB_CUDA(ctx, launch_last_rows_norm(hS, ctx->d_lastrows, b.n_req, c.d_model, c.rms_eps, ctx->xlast, s));
  CB_CUDA(ctx, launch_lm_head(ctx->xlast, b.n_req, c.d_model, ctx->lm, c.vocab, c.dtype, ctx->logits, s));
  CB_CUDA(ctx, launch_argmax(ctx->logits, b.n_req, c.vocab, ctx->d_first_ptrs, ctx->d_first, s));
  for (int r = 0; r < b.n_req; ++r) {
    const ReqHost& rh = b.reqs[r];
    const PlanEntry& pe = b.plan[static_cast<size_t>(b.L - 1) * b.n_req + r];
    if (rh.out_hidden) CB_CUDA(ctx, launch_write_hidden(hS, posS, pe.s_off, pe.s_n, c.d_model, rh.out_hidden, s));
    if (rh.out_sel_count) {
      // counts of request r are strided by n_req in d_counts: copy one by one
      for (int i = 0; i < b.L; ++i)
        CB_CUDA(ctx, cudaMemcpyAsync(rh.out_sel_count + i, ctx->d_counts + static_cast<size_t>(i) * b.n_req + r, 4,
                                     cudaMemcpyDeviceToDevice, s));
    }
  }
  b.active = false;
  return CB_OK;
}

}  // namespace

namespace cb {
static std::atomic<bool> g_launch_overlap{true};
bool launch_overlap_enabled() { return g_launch_overlap.load(std::memory_order_relaxed); }
void set_launch_overlap(bool on) { g_launch_overlap.store(on); }
}  // namespace cb

// ============================================================================= C ABI
extern "C" {

const char* cb_status_string(cb_status s) {
  switch (s) {
    case CB_OK: return "ok";
    case CB_ERR_INVALID_ARG: return "invalid argument";
    case CB_ERR_SHAPE: return "shape not supported";
    case CB_ERR_DTYPE: return "dtype not supported";
    case CB_ERR_NOT_FOUND: return "chunk id not registered";
    case CB_ERR_WORKSPACE: return "workspace missing or too small";
    case CB_ERR_CUDA: return "CUDA error";
    case CB_ERR_TIMEOUT: return "deadline passed";
    case CB_ERR_NAN: return "NaN deviation";
    case CB_ERR_DEVICE: return "device-side check failed";
    case CB_ERR_STATE: return "call out of order";
  }
  return "unknown status";
}

const char* cb_last_error(const cb_ctx* ctx) { return ctx ? ctx->last_error.c_str() : g_last_error.c_str(); }

cb_status cb_create(const cb_model_cfg* cfg, const cb_weights* w, cb_ctx** out) {
  if (!cfg || !w || !out) return fail(nullptr, CB_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  std::string why;
  if (!valid_cfg(*cfg, &why)) return fail(nullptr, CB_ERR_SHAPE, why);
  if (!w->embed || !w->lm_head || !w->wq || !w->wk || !w->wv || !w->wo || !w->wgate || !w->wup || !w->wdown)
    return fail(nullptr, CB_ERR_INVALID_ARG, "null weight pointer");
  cb_ctx* c = new cb_ctx();
  c->cfg = *cfg;
  c->embed = w->embed;
  c->lm = w->lm_head;
  const int L = cfg->n_layers;
  for (int i = 0; i < L; ++i) {
    const void* ps[7] = {w->wq[i], w->wk[i], w->wv[i], w->wo[i], w->wgate[i], w->wup[i], w->wdown[i]};
    for (const void* p : ps)
      if (!p || !aligned16(p)) {
        delete c;
        return fail(nullptr, CB_ERR_INVALID_ARG, "null or misaligned layer weight");
      }
    c->wq.push_back(ps[0]);
    c->wk.push_back(ps[1]);
    c->wv.push_back(ps[2]);
    c->wo.push_back(ps[3]);
    c->wg.push_back(ps[4]);
    c->wu.push_back(ps[5]);
    c->wd.push_back(ps[6]);
  }
  c->fetch_ev.resize(L, nullptr);
  bool ok = cudaEventCreateWithFlags(&c->pinned_ev, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&c->status_ev, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < L; ++i) ok = cudaEventCreateWithFlags(&c->fetch_ev[i], cudaEventDisableTiming) == cudaSuccess;
  void* sh = nullptr;
  ok = ok && cudaMallocHost(&sh, 64) == cudaSuccess;
  if (!ok) {
    cb_destroy(c);
    return fail(nullptr, CB_ERR_CUDA, "event or pinned-buffer creation failed");
  }
  c->status_host = static_cast<int32_t*>(sh);
  *out = c;
  return CB_OK;
}

cb_status cb_destroy(cb_ctx* ctx) {
  if (!ctx) return CB_OK;
  if (ctx->pinned_pending) cudaEventSynchronize(ctx->pinned_ev);
  for (cudaEvent_t e : ctx->fetch_ev)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : ctx->slot_ev)
    if (e) cudaEventDestroy(e);
  if (ctx->pinned_ev) cudaEventDestroy(ctx->pinned_ev);
  if (ctx->status_ev) cudaEventDestroy(ctx->status_ev);
  if (ctx->pinned) cudaFreeHost(ctx->pinned);
  if (ctx->status_host) cudaFreeHost(ctx->status_host);
  for (const cb_ctx::Mark& m : ctx->marks) {
    cudaEventDestroy(m.a);
    cudaEventDestroy(m.b);
  }
  for (cudaEvent_t e : ctx->ev_pool) cudaEventDestroy(e);
  delete ctx;
  return CB_OK;
}

size_t cb_workspace_size(const cb_ctx* ctx, int max_tokens, int max_requests) {
  if (!ctx || max_tokens < 1 || max_requests < 1) return 0;
  return ws_layout(ctx->cfg, max_tokens, max_requests).total;
}

cb_status cb_set_workspace(cb_ctx* ctx, void* ws, size_t bytes, int max_tokens, int max_requests) {
  if (!ctx || !ws || max_tokens < 1 || max_requests < 1) return fail(ctx, CB_ERR_INVALID_ARG, "bad workspace arguments");
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(ctx, CB_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ctx->b.active) return fail(ctx, CB_ERR_STATE, "cannot rebind the workspace during a batch");
  const cb_model_cfg& c = ctx->cfg;
  const WsLayout w = ws_layout(c, max_tokens, max_requests);
  if (bytes < w.total) return fail(ctx, CB_ERR_WORKSPACE, "workspace too small");
  uint8_t* base = static_cast<uint8_t*>(ws);
  ctx->ws = base;
  ctx->ws_bytes = bytes;
  ctx->ws_tokens = max_tokens;
  ctx->ws_reqs = max_requests;
  ctx->status = reinterpret_cast<int32_t*>(base + w.status);
  ctx->rope = reinterpret_cast<float2*>(base + w.rope);
  ctx->tok = reinterpret_cast<int32_t*>(base + w.tok);
  ctx->pos[0] = reinterpret_cast<int32_t*>(base + w.pos0);
  ctx->pos[1] = reinterpret_cast<int32_t*>(base + w.pos1);
  ctx->req[0] = reinterpret_cast<int32_t*>(base + w.req0);
  ctx->req[1] = reinterpret_cast<int32_t*>(base + w.req1);
  ctx->src = reinterpret_cast<int32_t*>(base + w.src);
  ctx->dev = reinterpret_cast<float*>(base + w.dev);
  ctx->h[0] = reinterpret_cast<float*>(base + w.h0);
  ctx->h[1] = reinterpret_cast<float*>(base + w.h1);
  ctx->x = base + w.x;
  ctx->qkv = reinterpret_cast<float*>(base + w.qkv);
  ctx->q = base + w.q;
  ctx->attn = base + w.attn;
  ctx->act = base + w.act;
  ctx->tmp_k = base + w.tmpk;
  ctx->tmp_v = base + w.tmpv;
  ctx->logits = reinterpret_cast<float*>(base + w.logits);
  ctx->xlast = reinterpret_cast<float*>(base + w.xlast);
  ctx->gemm_scratch = base + w.gemm;
  ctx->gemm_scratch_bytes = gemm_scratch_bytes();
  ctx->dec_o = reinterpret_cast<float*>(base + w.dec_o);
  ctx->dec_ml = reinterpret_cast<float2*>(base + w.dec_ml);
  ctx->att_o = reinterpret_cast<float*>(base + w.att_o);
  ctx->att_ml = reinterpret_cast<float2*>(base + w.att_ml);
  ctx->att_cnt = reinterpret_cast<int*>(base + w.att_cnt);
  ctx->meta = base + w.meta;
  ctx->meta_bytes = w.meta_bytes;
  // rotary table: (cos, sin) of p * theta^(-2i/dh), evaluated in double on the host
  const int half = c.head_dim / 2;
  std::vector<float2> tab(static_cast<size_t>(c.max_positions) * half);
  for (int i = 0; i < half; ++i) {
    const double inv = std::pow(c.rope_theta, -2.0 * i / c.head_dim);
    for (int p = 0; p < c.max_positions; ++p) {
      const double a = static_cast<double>(p) * inv;
      tab[static_cast<size_t>(p) * half + i] = make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
    }
  }
  CB_CUDA(ctx, cudaMemcpy(ctx->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice));
  CB_CUDA(ctx, cudaMemset(ctx->status, 0, 256));
  CB_CUDA(ctx, cudaMemset(ctx->gemm_scratch, 0, ctx->gemm_scratch_bytes));
  CB_CUDA(ctx, cudaMemset(ctx->att_cnt, 0, static_cast<size_t>(ATTN_SPLIT_UNITS) * 4));
  return CB_OK;
}

cb_status cb_register_chunk(cb_ctx* ctx, uint64_t chunk_id, const int32_t* ids, const void* k, const void* v, int n,
                            int on_host) {
  if (!ctx || !ids || !k || !v || n < 1) return fail(ctx, CB_ERR_INVALID_ARG, "bad chunk arguments");
  if (!aligned16(k) || !aligned16(v)) return fail(ctx, CB_ERR_INVALID_ARG, "chunk KV must be 16-byte aligned");
  if (n >= ctx->cfg.max_positions) return fail(ctx, CB_ERR_SHAPE, "chunk longer than max_positions");
  if (ctx->b.active) return fail(ctx, CB_ERR_STATE, "cannot change the registry during a batch");
  ChunkEntry e;
  e.id = chunk_id;
  e.ids = ids;
  e.k = k;
  e.v = v;
  e.n = n;
  e.on_host = on_host ? 1 : 0;
  ctx->reg.put(e);
  return CB_OK;
}

cb_status cb_register_chunk_codec(cb_ctx* ctx, uint64_t chunk_id, const int32_t* ids, const void* blob, int n,
                                  int bits, int on_host) {
  if (!ctx || !ids || !blob || n < 1) return fail(ctx, CB_ERR_INVALID_ARG, "bad chunk arguments");
  if (bits != 8 && bits != 4) return fail(ctx, CB_ERR_INVALID_ARG, "bits must be 8 or 4");
  if (!aligned16(blob)) return fail(ctx, CB_ERR_INVALID_ARG, "the quantised chunk must be 16-byte aligned");
  if (ctx->cfg.head_dim != 64 && ctx->cfg.head_dim != 128)
    return fail(ctx, CB_ERR_SHAPE, "the KV codec needs head_dim 64 or 128");
  if (n >= ctx->cfg.max_positions) return fail(ctx, CB_ERR_SHAPE, "chunk longer than max_positions");
  if (ctx->b.active) return fail(ctx, CB_ERR_STATE, "cannot change the registry during a batch");
  ChunkEntry e;
  e.id = chunk_id;
  e.ids = ids;
  e.n = n;
  e.on_host = on_host ? 1 : 0;
  e.blob = static_cast<const uint8_t*>(blob);
  e.bits = bits;
  e.layer_bytes = codec_layout(n, ctx->cfg.n_kv_heads, ctx->cfg.head_dim, bits).bytes;
  ctx->reg.put(e);
  return CB_OK;
}

cb_status cb_chunk_info_of(const cb_ctx* ctx, uint64_t chunk_id, cb_chunk_info* out) {
  if (!ctx || !out) return fail(nullptr, CB_ERR_INVALID_ARG, "null argument");
  *out = cb_chunk_info{0, CB_TIER_MISSING, 0.0};
  const ChunkEntry* e = const_cast<cb_ctx*>(ctx)->reg.find(chunk_id);
  if (!e) return CB_OK;
  const cb_model_cfg& c = ctx->cfg;
  out->n_tokens = e->n;
  out->tier = e->on_host ? CB_TIER_HOST : CB_TIER_DEVICE;
  out->bytes = e->bits ? static_cast<double>(e->layer_bytes) * c.n_layers
                       : 2.0 * c.n_layers * e->n * c.n_kv_heads * c.head_dim * dtype_bytes(c.dtype);
  return CB_OK;
}

cb_status cb_set_staging(cb_ctx* ctx, void* buf, size_t bytes) {
  if (!ctx || (bytes && !buf)) return fail(ctx, CB_ERR_INVALID_ARG, "bad staging buffer");
  if (buf && !aligned16(buf)) return fail(ctx, CB_ERR_INVALID_ARG, "the staging buffer must be 16-byte aligned");
  if (ctx->b.active) return fail(ctx, CB_ERR_STATE, "cannot change the staging buffer during a batch");
  ctx->staging = static_cast<uint8_t*>(buf);
  ctx->staging_bytes = buf ? bytes : 0;
  return CB_OK;
}

size_t cb_codec_layer_bytes(int n_tok, int n_kv_heads, int head_dim, int bits) {
  if (n_tok < 1 || n_kv_heads < 1 || (head_dim != 64 && head_dim != 128) || (bits != 8 && bits != 4)) return 0;
  return codec_layout(n_tok, n_kv_heads, head_dim, bits).bytes;
}

cb_status cb_kv_encode(const void* k, const void* v, int n_layers, int n_tok, int n_kv_heads, int head_dim,
                       cb_dtype dtype, int bits, void* blob, void* stream) {
  if (!k || !v || !blob) return fail(nullptr, CB_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(blob)) return fail(nullptr, CB_ERR_INVALID_ARG, "blob must be 16-byte aligned");
  if (n_layers < 1 || n_tok < 1 || n_kv_heads < 1 || (head_dim != 64 && head_dim != 128))
    return fail(nullptr, CB_ERR_SHAPE, "bad codec sizes (head_dim 64 or 128)");
  if (bits != 8 && bits != 4) return fail(nullptr, CB_ERR_INVALID_ARG, "bits must be 8 or 4");
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(nullptr, CB_ERR_DTYPE, "unknown dtype");
  cudaError_t e = launch_kv_encode(k, v, n_layers, n_tok, n_kv_heads, head_dim, bits, dtype, blob, as_stream(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(nullptr, e, "cb_kv_encode");
}

cb_status cb_kv_decode(const void* blob, int n_layers, int n_tok, int n_kv_heads, int head_dim, int bits,
                       int delta_pos, double theta, cb_dtype dtype, void* k_out, void* v_out, void* stream) {
  if (!blob || !k_out || !v_out) return fail(nullptr, CB_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(blob) || !aligned16(k_out) || !aligned16(v_out))
    return fail(nullptr, CB_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (n_layers < 1 || n_tok < 1 || n_kv_heads < 1 || (head_dim != 64 && head_dim != 128) || delta_pos < 0 ||
      !(theta > 0))
    return fail(nullptr, CB_ERR_SHAPE, "bad codec sizes (head_dim 64 or 128)");
  if (bits != 8 && bits != 4) return fail(nullptr, CB_ERR_INVALID_ARG, "bits must be 8 or 4");
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(nullptr, CB_ERR_DTYPE, "unknown dtype");
  float cs[128];
  for (int i = 0; i < head_dim / 2; ++i) {
    const double a = static_cast<double>(delta_pos) * std::pow(theta, -2.0 * i / head_dim);
    cs[2 * i] = static_cast<float>(std::cos(a));
    cs[2 * i + 1] = static_cast<float>(std::sin(a));
  }
  cudaError_t e = launch_codec_decode_blob(blob, n_layers, n_tok, n_kv_heads, head_dim, bits, cs, dtype, k_out, v_out,
                                           as_stream(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(nullptr, e, "cb_kv_decode");
}

cb_status cb_unregister_chunk(cb_ctx* ctx, uint64_t chunk_id) {
  if (!ctx) return fail(ctx, CB_ERR_INVALID_ARG, "null context");
  if (ctx->b.active) return fail(ctx, CB_ERR_STATE, "cannot change the registry during a batch");
  return ctx->reg.erase(chunk_id) ? CB_OK : fail(ctx, CB_ERR_NOT_FOUND, "chunk id not registered");
}

int cb_registered_chunks(const cb_ctx* ctx) { return ctx ? const_cast<cb_ctx*>(ctx)->reg.size() : 0; }

// ----------------------------------------------------------------------------- standalone kernels
cb_status cb_rope_rerotate(const void* k_src, void* k_dst, const void* v_src, void* v_dst, int n_tok, int n_kv_heads,
                           int head_dim, int delta_pos, double theta, cb_dtype dtype, void* stream) {
  if (!k_src || !k_dst || (v_src == nullptr) != (v_dst == nullptr)) return fail(nullptr, CB_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_src) || !aligned16(k_dst) || (v_src && (!aligned16(v_src) || !aligned16(v_dst))))
    return fail(nullptr, CB_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (n_tok < 0 || n_kv_heads < 1 || head_dim < 16 || head_dim > 128 || head_dim % 16 || delta_pos < 0 || !(theta > 0))
    return fail(nullptr, CB_ERR_SHAPE, "bad rerotate sizes");
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(nullptr, CB_ERR_DTYPE, "unknown dtype");
  float cs[128];
  for (int i = 0; i < head_dim / 2; ++i) {
    const double a = static_cast<double>(delta_pos) * std::pow(theta, -2.0 * i / head_dim);
    cs[2 * i] = static_cast<float>(std::cos(a));
    cs[2 * i + 1] = static_cast<float>(std::sin(a));
  }
  cudaError_t e = launch_rerotate_single(k_src, k_dst, v_src, v_dst, n_tok, n_kv_heads, head_dim, cs, dtype,
                                         as_stream(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(nullptr, e, "cb_rope_rerotate");
}

cb_status cb_kv_deviation(const float* k_new, const float* v_new, const void* k_fus, const void* v_fus,
                          const int32_t* idx, int n, int kv_width, int mode, cb_dtype dtype, float* dev_out,
                          void* stream) {
  if (!k_new || !v_new || !k_fus || !v_fus || !dev_out) return fail(nullptr, CB_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_fus) || !aligned16(v_fus))
    return fail(nullptr, CB_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (n < 0 || kv_width < 8 || kv_width % 8 || mode < 0 || mode > 3) return fail(nullptr, CB_ERR_SHAPE, "bad sizes");
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(nullptr, CB_ERR_DTYPE, "unknown dtype");
  cudaError_t e = launch_deviation_plain(k_new, v_new, k_fus, v_fus, idx, n, kv_width, mode, dtype, dev_out,
                                         as_stream(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(nullptr, e, "cb_kv_deviation");
}

cb_status cb_select_hkvd(const float* dev, const int32_t* cand, int n, int k, int32_t* sel_out, int32_t* status,
                         void* stream) {
  if (n < 0 || n > 65536 || k < 0 || k > n) return fail(nullptr, CB_ERR_SHAPE, "need 0 <= k <= n <= 65536");
  if (k > 0 && (!dev || !sel_out)) return fail(nullptr, CB_ERR_INVALID_ARG, "null pointer");
  cudaError_t e = launch_select_plain(dev, cand, n, k, sel_out, status, as_stream(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(nullptr, e, "cb_select_hkvd");
}

cb_status cb_gemm(const void* A, const void* B, const void* B2, void* C, int M, int N, int K, int ldc, int epilogue,
                  cb_dtype dtype, void* scratch, size_t scratch_bytes, void* stream) {
  if (!A || !B || !C || (epilogue == 2 && !B2)) return fail(nullptr, CB_ERR_INVALID_ARG, "null pointer");
  if (epilogue < 0 || epilogue > 2) return fail(nullptr, CB_ERR_INVALID_ARG, "bad epilogue");
  if (M < 0 || N < 1 || K < 1) return fail(nullptr, CB_ERR_SHAPE, "bad sizes");
  if (dtype == CB_BF16) {
    if (K % 64 || N % 128 || (reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        (B2 && (reinterpret_cast<uintptr_t>(B2) & 15)))
      return fail(nullptr, CB_ERR_SHAPE, "bf16 GEMM needs K % 64 == 0, N % 128 == 0 and 16-byte aligned operands");
    if (ldc % 8 || (reinterpret_cast<uintptr_t>(C) & 15)) return fail(nullptr, CB_ERR_SHAPE, "ldc % 8 and aligned C");
    if (scratch && (reinterpret_cast<uintptr_t>(scratch) & 15))
      return fail(nullptr, CB_ERR_INVALID_ARG, "scratch must be 16-byte aligned");
  } else if (dtype != CB_F32) {
    return fail(nullptr, CB_ERR_DTYPE, "unknown dtype");
  }
  if (epilogue == 2 ? ldc < N / 2 : ldc < N) return fail(nullptr, CB_ERR_SHAPE, "ldc too small");
  int32_t* status = nullptr;  // device-side problems go to the standalone GEMM status word
  cudaError_t e = standalone_gemm_status(&status);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cb_gemm");
  e = launch_gemm(A, B, epilogue == 2 ? B2 : nullptr, nullptr, N, N, C, M, N, K, ldc, epilogue, dtype, status, scratch,
                  scratch ? scratch_bytes : 0, as_stream(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(nullptr, e, "cb_gemm");
}

size_t cb_gemm_scratch_size(void) { return gemm_scratch_bytes(); }

cb_status cb_set_launch_overlap(int enabled) {
  cb::set_launch_overlap(enabled != 0);
  return CB_OK;
}

cb_status cb_set_qkv_fusion(int enabled) {
  if (enabled != 0 && enabled != 1) return fail(nullptr, CB_ERR_INVALID_ARG, "enabled must be 0 or 1");
  set_qkv_fusion(enabled != 0);
  return CB_OK;
}

cb_status cb_attention_set_tiles(int tiles) {
  if (tiles < 0 || tiles > 2) return fail(nullptr, CB_ERR_INVALID_ARG, "tiles must be 0, 1 or 2");
  attention_set_tiles(tiles);
  return CB_OK;
}

cb_status cb_gemm_set_orientation(int orientation) {
  const bool tile = orientation >= 16 && orientation <= 256 && orientation % 16 == 0;
  if ((orientation < 0 || orientation > 2) && !tile)
    return fail(nullptr, CB_ERR_INVALID_ARG, "orientation must be 0, 1, 2 or a token tile 16..256 (multiple of 16)");
  gemm_set_orientation(orientation);
  return CB_OK;
}

cb_status cb_gemm_describe(int M, int N, int K, int epilogue, size_t scratch_bytes, char* buf, size_t len) {
  if (!buf || len == 0) return fail(nullptr, CB_ERR_INVALID_ARG, "null buffer");
  if (M < 0 || N < 0 || K < 0 || epilogue < 0 || epilogue > 2)
    return fail(nullptr, CB_ERR_INVALID_ARG, "negative size or unknown epilogue");
  gemm_describe(M, N, K, epilogue, scratch_bytes, buf, len);
  return CB_OK;
}

cb_status cb_gemm_set_pairing(int pairing) {
  if (pairing != 0 && pairing != 1 && pairing != 2 && pairing != 4)
    return fail(nullptr, CB_ERR_INVALID_ARG, "pairing must be 0, 1, 2 or 4");
  gemm_set_pairing(pairing);
  return CB_OK;
}

cb_status cb_attention(const void* q, const int32_t* q_pos, int m, const void* k, const void* v, int n_kv, int n_heads,
                       int n_kv_heads, int head_dim, void* out, cb_dtype dtype, void* stream) {
  if (!q || !q_pos || !k || !v || !out) return fail(nullptr, CB_ERR_INVALID_ARG, "null pointer");
  if (m < 0 || n_kv < 1 || n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads)
    return fail(nullptr, CB_ERR_SHAPE, "bad sizes");
  if (dtype == CB_BF16 ? head_dim != 128 : (head_dim % 32 || head_dim > 128))
    return fail(nullptr, CB_ERR_SHAPE, "head_dim must be 128 (bf16) or a multiple of 32 up to 128 (fp32)");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return fail(nullptr, CB_ERR_INVALID_ARG, "unaligned operand");
  cudaError_t e = launch_attention_direct(q, q_pos, m, k, v, n_kv, n_heads, n_kv_heads, head_dim, out, dtype,
                                          as_stream(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(nullptr, e, "cb_attention");
}

// ----------------------------------------------------------------------------- blended prefill
static cb_status build_blend_requests(cb_ctx* ctx, const cb_request* reqs, int n_req, std::vector<InReq>& in) {
  const cb_model_cfg& c = ctx->cfg;
  in.assign(n_req, InReq{});
  for (int r = 0; r < n_req; ++r) {
    const cb_request& q = reqs[r];
    if (q.n_query < 1 || !q.query_ids || !q.fused_k || !q.fused_v || q.n_chunks < 0 || (q.n_chunks && !q.chunk_ids_host))
      return fail(ctx, CB_ERR_INVALID_ARG, "bad request (query, fused cache or chunk list)");
    if (!aligned16(q.fused_k) || !aligned16(q.fused_v)) return fail(ctx, CB_ERR_INVALID_ARG, "unaligned fused cache");
    int N = 0;
    for (int j = 0; j < q.n_chunks; ++j) {
      ChunkEntry* e = ctx->reg.find(q.chunk_ids_host[j]);
      if (!e) return fail(ctx, CB_ERR_NOT_FOUND, "chunk id not registered");
      in[r].segs.push_back(SegHost{e, N, e->n});
      N += e->n;
    }
    N += q.n_query;
    if (N > c.max_positions) return fail(ctx, CB_ERR_SHAPE, "prompt longer than max_positions");
    if (q.kv_capacity != 0 && q.kv_capacity < N) return fail(ctx, CB_ERR_SHAPE, "kv_capacity below the prompt length");
    const int cap = q.kv_capacity ? q.kv_capacity : N;
    in[r].query_ids = q.query_ids;
    in[r].n_query = q.n_query;
    in[r].fused_k = q.fused_k;
    in[r].fused_v = q.fused_v;
    in[r].layer_stride = static_cast<long long>(cap) * c.n_kv_heads * c.head_dim;
    in[r].out_hidden = q.out_hidden;
    in[r].out_sel = q.out_sel;
    in[r].out_sel_count = q.out_sel_count;
    in[r].out_first_token = q.out_first_token;
  }
  return CB_OK;
}

cb_status cb_blend_begin(cb_ctx* ctx, const cb_request* reqs, int n_req, const cb_blend_params* params, void* stream) {
  if (!ctx || !reqs || !params) return fail(ctx, CB_ERR_INVALID_ARG, "null argument");
  if (params->select_mode != CB_SELECT_HKVD && params->select_mode != CB_SELECT_SEAM)
    return fail(ctx, CB_ERR_INVALID_ARG, "bad select_mode");
  const bool seam = params->select_mode == CB_SELECT_SEAM;
  if (params->n_layers != ctx->cfg.n_layers || (!seam && !params->layer_ratio_host))
    return fail(ctx, CB_ERR_INVALID_ARG, "layer_ratio_host must have n_layers entries");
  if (params->dev_mode < 0 || params->dev_mode > 3) return fail(ctx, CB_ERR_INVALID_ARG, "bad dev_mode");
  if (seam && params->seam_tokens < 0) return fail(ctx, CB_ERR_INVALID_ARG, "seam_tokens must be >= 0");
  std::vector<InReq> in;
  cb_status st = build_blend_requests(ctx, reqs, n_req, in);
  if (st != CB_OK) return st;
  return begin_impl(ctx, in, seam ? nullptr : params->layer_ratio_host, params->dev_mode,
                    seam ? nullptr : params->forced_sel_host, seam ? params->seam_tokens : -1, as_stream(stream));
}

cb_status cb_fetch_kv(cb_ctx* ctx, int layer, void* copy_stream) {
  if (!ctx) return fail(ctx, CB_ERR_INVALID_ARG, "null context");
  return fetch_impl(ctx, layer, as_stream(copy_stream));
}

cb_status cb_synchronize(cb_ctx* ctx, int layer, int timeout_ms) {
  if (!ctx) return fail(ctx, CB_ERR_INVALID_ARG, "null context");
  if (!ctx->b.active && ctx->b.fetched.empty()) return fail(ctx, CB_ERR_STATE, "no batch");
  if (layer < 0 || layer >= ctx->cfg.n_layers) return fail(ctx, CB_ERR_INVALID_ARG, "layer out of range");
  if (!ctx->b.any_host) return CB_OK;
  if (ctx->b.fetched.empty() || !ctx->b.fetched[layer]) return fail(ctx, CB_ERR_STATE, "layer was not fetched");
  return wait_event_deadline(ctx, ctx->fetch_ev[layer], timeout_ms);
}

cb_status cb_prefill_layer(cb_ctx* ctx, int layer, void* stream) {
  if (!ctx) return fail(ctx, CB_ERR_INVALID_ARG, "null context");
  return layer_impl(ctx, layer, as_stream(stream));
}

cb_status cb_blend_layer(cb_ctx* ctx, int layer, void* stream) {
  if (!ctx) return fail(ctx, CB_ERR_INVALID_ARG, "null context");
  if (ctx->b.active && ctx->b.any_host && layer >= 0 && layer < ctx->b.L && !ctx->b.fetched[layer]) {
    cb_status st = fetch_impl(ctx, layer, as_stream(stream));
    if (st != CB_OK) return st;
  }
  return layer_impl(ctx, layer, as_stream(stream));
}

cb_status cb_blend_finish(cb_ctx* ctx, void* stream) {
  if (!ctx) return fail(ctx, CB_ERR_INVALID_ARG, "null context");
  return finish_impl(ctx, as_stream(stream));
}

cb_status cb_blend_prefill(cb_ctx* ctx, const cb_request* reqs, int n_req, const cb_blend_params* params, void* stream,
                           void* copy_stream) {
  cb_status st = cb_blend_begin(ctx, reqs, n_req, params, stream);
  if (st != CB_OK) return st;
  Batch& b = ctx->b;
  // fetches run ahead of the layers by `window` layers: all of them for plain host chunks
  // (each layer has its own destination), the staging ring's slot count for quantised ones
  const int window = b.any_host ? (b.stage.empty() ? b.L : b.n_slots) : 0;
  if (b.any_host && !copy_stream) {
    b.active = false;
    return fail(ctx, CB_ERR_INVALID_ARG, "host-resident chunks need a copy stream");
  }
  for (int i = 0; i < std::min(window, b.L); ++i) {
    st = fetch_impl(ctx, i, as_stream(copy_stream));
    if (st != CB_OK) {
      b.active = false;
      return st;
    }
  }
  for (int i = 0; i < b.L; ++i) {
    st = layer_impl(ctx, i, as_stream(stream));
    if (st == CB_OK && window > 0 && i + window < b.L) st = fetch_impl(ctx, i + window, as_stream(copy_stream));
    if (st != CB_OK) {
      b.active = false;
      return st;
    }
  }
  return finish_impl(ctx, as_stream(stream));
}

// ----------------------------------------------------------------------------- decode
cb_status cb_decode_step(cb_ctx* ctx, const cb_decode_seq* seqs, int n_seq, const int32_t* tokens,
                         int32_t* out_tokens, void* stream) {
  if (!ctx || !seqs || !tokens || !out_tokens || n_seq < 1) return fail(ctx, CB_ERR_INVALID_ARG, "bad decode arguments");
  if (!ctx->ws) return fail(ctx, CB_ERR_WORKSPACE, "no workspace bound");
  if (ctx->b.active) return fail(ctx, CB_ERR_STATE, "a blend batch is active (finish it first)");
  if (n_seq > ctx->ws_reqs || n_seq > ctx->ws_tokens)
    return fail(ctx, CB_ERR_WORKSPACE, "more sequences than the workspace's max_requests / max_tokens");
  const cb_model_cfg& c = ctx->cfg;
  {
    const int g = c.n_heads / c.n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 7 && g != 8 && g != 16)
      return fail(ctx, CB_ERR_SHAPE, "decode supports 1, 2, 4, 7, 8 or 16 query heads per KV head");
  }
  if (c.head_dim != 64 && c.head_dim != 128) return fail(ctx, CB_ERR_SHAPE, "decode needs head_dim 64 or 128");
  const int H = c.n_heads, Hkv = c.n_kv_heads, dh = c.head_dim, d = c.d_model;
  const int qw = H * dh, kvw = Hkv * dh;
  cudaStream_t s = as_stream(stream);
  std::vector<ReqDev> rd(n_seq);
  std::vector<int32_t> pos(n_seq), req(n_seq);
  int max_keys = 1;
  for (int i = 0; i < n_seq; ++i) {
    const cb_decode_seq& q = seqs[i];
    if (!q.fused_k || !q.fused_v || !aligned16(q.fused_k) || !aligned16(q.fused_v))
      return fail(ctx, CB_ERR_INVALID_ARG, "bad fused cache of a decode sequence");
    if (q.n_past < 0 || q.kv_capacity < q.n_past + 1) return fail(ctx, CB_ERR_SHAPE, "no room in the cache for the new token");
    if (q.n_past + 1 > c.max_positions) return fail(ctx, CB_ERR_SHAPE, "position beyond max_positions");
    rd[i] = ReqDev{q.fused_k, q.fused_v, static_cast<long long>(q.kv_capacity) * kvw, q.n_past + 1, q.n_past};
    pos[i] = q.n_past;
    req[i] = i;
    max_keys = std::max(max_keys, q.n_past + 1);
  }
  const int n_splits = decode_splits(max_keys);
  // metadata: request descriptors, positions, request indices, last rows (= 0..n-1)
  const size_t szReq = align_up(n_seq * sizeof(ReqDev), 256), szI = align_up(n_seq * 4, 256);
  const size_t total = szReq + 3 * szI;
  if (total > ctx->meta_bytes) return fail(ctx, CB_ERR_WORKSPACE, "decode metadata exceeds the workspace");
  cb_status st = ensure_pinned(ctx, total);
  if (st != CB_OK) return st;
  std::memcpy(ctx->pinned, rd.data(), n_seq * sizeof(ReqDev));
  std::memcpy(ctx->pinned + szReq, pos.data(), n_seq * 4);
  std::memcpy(ctx->pinned + szReq + szI, req.data(), n_seq * 4);
  std::memcpy(ctx->pinned + szReq + 2 * szI, req.data(), n_seq * 4);  // last rows: row i of sequence i
  CB_CUDA(ctx, cudaMemcpyAsync(ctx->meta, ctx->pinned, total, cudaMemcpyHostToDevice, s));
  CB_CUDA(ctx, cudaEventRecord(ctx->pinned_ev, s));
  ctx->pinned_pending = true;
  const ReqDev* d_rd = reinterpret_cast<const ReqDev*>(ctx->meta);
  const int32_t* d_pos = reinterpret_cast<const int32_t*>(ctx->meta + szReq);
  const int32_t* d_req = reinterpret_cast<const int32_t*>(ctx->meta + szReq + szI);
  const int32_t* d_rows = reinterpret_cast<const int32_t*>(ctx->meta + szReq + 2 * szI);
  float* h = ctx->h[0];
  {
    PhaseScope ps(ctx, CB_PH_BEGIN, s, 1);
    CB_CUDA(ctx, launch_embed(ctx->embed, tokens, n_seq, d, c.vocab, c.dtype, h, ctx->status, s));
  }
  for (int i = 0; i < c.n_layers; ++i) {
    {
      PhaseScope ps(ctx, CB_PH_NORM, s, 1);
      CB_CUDA(ctx, launch_rmsnorm(h, n_seq, d, c.rms_eps, ctx->x, c.dtype, s));
    }
    {
      PhaseScope ps(ctx, CB_PH_QKV, s, 1);
      CB_CUDA(ctx, launch_gemm(ctx->x, ctx->wq[i], ctx->wk[i], ctx->wv[i], qw, qw + kvw, ctx->qkv, n_seq, qw + 2 * kvw,
                               d, qw + 2 * kvw, 0, c.dtype, ctx->status, ctx->gemm_scratch, ctx->gemm_scratch_bytes, s));
    }
    {
      PhaseScope ps(ctx, CB_PH_SCATTER, s, 1);  // RoPE of q and k, the new K/V row appended to the cache
      CB_CUDA(ctx, launch_post_qkv(ctx->qkv, n_seq, nullptr, d_pos, d_req, d_rd, i, H, Hkv, dh, ctx->rope,
                                   c.max_positions, c.dtype, ctx->q, h, h, d, ctx->status, s));
    }
    {
      PhaseScope ps(ctx, CB_PH_ATTENTION, s, n_splits > 1 ? 2 : 1);
      CB_CUDA(ctx, launch_decode_attention(ctx->q, d_pos, d_rd, n_seq, i, H, Hkv, dh, n_splits, ctx->dec_o, ctx->dec_ml,
                                           ctx->attn, c.dtype, ctx->status, s));
    }
    {
      PhaseScope ps(ctx, CB_PH_OPROJ, s, 1);
      CB_CUDA(ctx, launch_gemm(ctx->attn, ctx->wo[i], nullptr, nullptr, d, d, h, n_seq, d, qw, d, 1, c.dtype,
                               ctx->status, ctx->gemm_scratch, ctx->gemm_scratch_bytes, s));
    }
    {
      PhaseScope ps(ctx, CB_PH_NORM, s, 1);
      CB_CUDA(ctx, launch_rmsnorm(h, n_seq, d, c.rms_eps, ctx->x, c.dtype, s));
    }
    {
      PhaseScope ps(ctx, CB_PH_GATEUP, s, 1);
      CB_CUDA(ctx, launch_gemm(ctx->x, ctx->wg[i], ctx->wu[i], nullptr, 0, 0, ctx->act, n_seq, 2 * c.ffn_dim, d,
                               c.ffn_dim, 2, c.dtype, ctx->status, ctx->gemm_scratch, ctx->gemm_scratch_bytes, s));
    }
    {
      PhaseScope ps(ctx, CB_PH_DOWN, s, 1);
      CB_CUDA(ctx, launch_gemm(ctx->act, ctx->wd[i], nullptr, nullptr, d, d, h, n_seq, d, c.ffn_dim, d, 1, c.dtype,
                               ctx->status, ctx->gemm_scratch, ctx->gemm_scratch_bytes, s));
    }
  }
  {
    PhaseScope ps(ctx, CB_PH_FINISH, s, 2 + (n_seq + 15) / 16);
    CB_CUDA(ctx, launch_last_rows_norm(h, d_rows, n_seq, d, c.rms_eps, ctx->xlast, s));
    CB_CUDA(ctx, launch_lm_head(ctx->xlast, n_seq, d, ctx->lm, c.vocab, c.dtype, ctx->logits, s));
    CB_CUDA(ctx, launch_argmax(ctx->logits, n_seq, c.vocab, nullptr, out_tokens, s));
  }
  for (int i = 0; i < n_seq; ++i)
    if (seqs[i].out_hidden)
      CB_CUDA(ctx, cudaMemcpyAsync(seqs[i].out_hidden, h + static_cast<size_t>(i) * d, d * 4, cudaMemcpyDeviceToDevice, s));
  return CB_OK;
}

cb_status cb_full_prefill(cb_ctx* ctx, const int32_t* ids, int n, void* k_out, void* v_out, float* out_hidden,
                          int32_t* first_token, void* stream) {
  if (!ctx || !ids || n < 1) return fail(ctx, CB_ERR_INVALID_ARG, "bad full-prefill arguments");
  if ((k_out == nullptr) != (v_out == nullptr)) return fail(ctx, CB_ERR_INVALID_ARG, "give both k_out and v_out or neither");
  if (k_out && (!aligned16(k_out) || !aligned16(v_out))) return fail(ctx, CB_ERR_INVALID_ARG, "unaligned KV output");
  if (n > ctx->cfg.max_positions) return fail(ctx, CB_ERR_SHAPE, "prompt longer than max_positions");
  if (!ctx->ws) return fail(ctx, CB_ERR_WORKSPACE, "no workspace bound");
  std::vector<InReq> in(1);
  in[0].query_ids = ids;
  in[0].n_query = n;
  if (k_out) {
    in[0].fused_k = k_out;
    in[0].fused_v = v_out;
    in[0].layer_stride = static_cast<long long>(n) * ctx->cfg.n_kv_heads * ctx->cfg.head_dim;
  } else {
    in[0].fused_k = ctx->tmp_k;
    in[0].fused_v = ctx->tmp_v;
    in[0].layer_stride = 0;
  }
  in[0].out_hidden = out_hidden;
  in[0].out_first_token = first_token;
  cudaStream_t s = as_stream(stream);
  cb_status st = begin_impl(ctx, in, nullptr, 0, nullptr, -1, s);
  if (st != CB_OK) return st;
  for (int i = 0; i < ctx->b.L; ++i) {
    st = layer_impl(ctx, i, s);
    if (st != CB_OK) {
      ctx->b.active = false;
      return st;
    }
  }
  return finish_impl(ctx, s);
}

cb_status cb_precompute_chunk(cb_ctx* ctx, const int32_t* ids, int n, void* k_out, void* v_out, void* stream) {
  if (!k_out || !v_out) return fail(ctx, CB_ERR_INVALID_ARG, "k_out and v_out are required");
  return cb_full_prefill(ctx, ids, n, k_out, v_out, nullptr, nullptr, stream);
}

cb_status cb_get_status(cb_ctx* ctx, void* stream, int timeout_ms) {
  if (!ctx || !ctx->ws) return fail(ctx, CB_ERR_WORKSPACE, "no workspace bound");
  cudaStream_t s = as_stream(stream);
  CB_CUDA(ctx, cudaMemcpyAsync(ctx->status_host, ctx->status, 4, cudaMemcpyDeviceToHost, s));
  CB_CUDA(ctx, cudaMemsetAsync(ctx->status, 0, 4, s));
  CB_CUDA(ctx, cudaEventRecord(ctx->status_ev, s));
  cb_status st = wait_event_deadline(ctx, ctx->status_ev, timeout_ms);
  if (st != CB_OK) return st;
  const int32_t v = *ctx->status_host;
  if (v) {
    // A kernel that gave up (a bounded wait ran out) may have left the counters that later
    // launches expect at zero -- the stream-K flags of the GEMM scratch, the attention's
    // key-range tickets: clear them before anything else runs on the stream.
    CB_CUDA(ctx, cudaMemsetAsync(ctx->gemm_scratch, 0, ctx->gemm_scratch_bytes, s));
    CB_CUDA(ctx, cudaMemsetAsync(ctx->att_cnt, 0, static_cast<size_t>(ATTN_SPLIT_UNITS) * 4, s));
  }
  if (v & ST_NAN) return fail(ctx, CB_ERR_NAN, "a deviation was NaN");
  if (v) return fail(ctx, CB_ERR_DEVICE, "device status word " + std::to_string(v));
  return CB_OK;
}

cb_status cb_set_profiling(cb_ctx* ctx, int enable) {
  if (!ctx) return fail(ctx, CB_ERR_INVALID_ARG, "null context");
  ctx->prof = enable < 0 ? 0 : (enable > 3 ? 3 : enable);
  return CB_OK;
}

cb_status cb_get_layer_profile(cb_ctx* ctx, int n_layers, float* load_ms_host, float* compute_ms_host) {
  if (!ctx || n_layers < 0 || (n_layers > 0 && (!load_ms_host || !compute_ms_host)))
    return fail(ctx, CB_ERR_INVALID_ARG, "bad arguments");
  for (int i = 0; i < n_layers; ++i) load_ms_host[i] = compute_ms_host[i] = 0.f;
  cb_status st = CB_OK;
  for (const cb_ctx::LayerMark& m : ctx->layer_marks) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(m.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, m.a, m.b);
    if (e != cudaSuccess && st == CB_OK) st = cuda_fail(ctx, e, "cb_get_layer_profile");
    if (m.layer >= 0 && m.layer < n_layers) (m.load ? load_ms_host : compute_ms_host)[m.layer] += ms;
    ctx->ev_pool.push_back(m.a);
    ctx->ev_pool.push_back(m.b);
  }
  ctx->layer_marks.clear();
  return st;
}

cb_status cb_get_profile(cb_ctx* ctx, cb_profile* out) {
  if (!ctx || !out) return fail(ctx, CB_ERR_INVALID_ARG, "null argument");
  std::memset(out, 0, sizeof(*out));
  for (const cb_ctx::Mark& m : ctx->marks) {
    CB_CUDA(ctx, cudaEventSynchronize(m.b));
    float ms = 0.f;
    CB_CUDA(ctx, cudaEventElapsedTime(&ms, m.a, m.b));
    out->ms[m.phase] += ms;
    out->calls[m.phase] += 1;
    ctx->ev_pool.push_back(m.a);
    ctx->ev_pool.push_back(m.b);
  }
  ctx->marks.clear();
  for (int p = 0; p < CB_N_PHASES; ++p) {
    out->launches[p] = ctx->launches[p];
    ctx->launches[p] = 0;
  }
  return CB_OK;
}

cb_status cb_plan_counts(const cb_ctx* ctx, int request, int32_t* counts_host) {
  if (!ctx || !counts_host) return fail(nullptr, CB_ERR_INVALID_ARG, "null argument");
  const Batch& b = ctx->b;
  if (b.plan.empty() || request < 0 || request >= b.n_req) return fail(nullptr, CB_ERR_STATE, "no planned batch");
  for (int i = 0; i < b.L; ++i) counts_host[i] = b.plan[static_cast<size_t>(i) * b.n_req + request].s_n;
  return CB_OK;
}

}  // extern "C"
