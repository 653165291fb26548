// Loading controller (host code): the content key of a chunk and the plan that decides, per
// chunk of a prompt, whether its cached KV is used, loaded or recomputed, and which recompute
// ratio hides under the loading.
//   [P3] loading controller: checks whether the selected chunks' caches exist and where they
//        are stored, and coordinates loading and recompute; the cache manager finds a cache by
//        a hash of its text.
//   [P1] パイプライン化の設計 (T_recompute = r% x T_prefill, T_load = KV bytes / throughput, both
//        overlapped) and 閾値チューニングのガイドライン (raise r on slow storage, lower it on fast).
//   [P4] §5 損益分岐: load only when the transfer costs less than recomputing the same tokens.
#include <cmath>
#include <cstdint>

#include "cacheblend.h"

extern "C" {

int cb_k_for_ratio(double r, int n_cached) {
  // k = ceil(r * Nc), guarded against the rounding of r * Nc just above an integer
  if (!(r > 0) || n_cached <= 0) return 0;
  return static_cast<int>(std::ceil(r * n_cached - 1e-9));
}

cb_status cb_ratio_schedule(int n_layers, double r, int schedule, double r1, int n_narrow, double* out_host) {
  // Gradual filtering ([P1] 段階的フィルタリングスキーム): layer 0 runs on every token (no
  // check), layer 1 measures the deviation of all cached tokens and keeps r1 of them, the
  // next n_narrow layers narrow linearly from r1 down to r, later layers keep the set.
  if (n_layers < 0 || !(r >= 0) || r > 1 || (n_layers > 0 && !out_host) || n_narrow < 0)
    return CB_ERR_INVALID_ARG;
  if (schedule != CB_SCHEDULE_FIXED && schedule != CB_SCHEDULE_GRADUAL) return CB_ERR_INVALID_ARG;
  for (int i = 0; i < n_layers; ++i) out_host[i] = -1.0;
  if (n_layers < 2) return CB_OK;
  if (schedule == CB_SCHEDULE_FIXED) {
    out_host[1] = r;
    return CB_OK;
  }
  if (r1 < 0) r1 = std::fmin(1.0, 2.0 * r);
  if (r1 > 1 || r1 < r) return CB_ERR_INVALID_ARG;
  out_host[1] = r1;
  for (int j = 1; j <= n_narrow && 1 + j < n_layers; ++j) out_host[1 + j] = r1 + (r - r1) * j / n_narrow;
  return CB_OK;
}

uint64_t cb_chunk_hash(const int32_t* ids_host, int n) {
  // FNV-1a, 64 bit (Fowler, Noll, Vo) over the ids as little-endian 32-bit integers
  uint64_t h = 0xCBF29CE484222325ull;
  if (!ids_host || n <= 0) return h;
  for (int i = 0; i < n; ++i) {
    const uint32_t u = static_cast<uint32_t>(ids_host[i]);
    for (int b = 0; b < 4; ++b) {
      h ^= (u >> (8 * b)) & 0xFFu;
      h *= 0x100000001B3ull;
    }
  }
  return h;
}

cb_status cb_plan_loading(const cb_cost_model* m, const cb_chunk_info* chunks, int n_chunks, int n_query,
                          int32_t* actions_host, double* ratio_out, double* t_load_out, double* t_recompute_out) {
  if (!m || n_chunks < 0 || n_query < 0 || (n_chunks && (!chunks || !actions_host)) || !ratio_out)
    return CB_ERR_INVALID_ARG;
  if (!(m->link_bytes_per_s > 0) || !(m->prefill_s_per_token > 0) || m->link_latency_s < 0 ||
      m->recompute_fixed_s < 0 || !(m->r_min >= 0) || !(m->r_max >= m->r_min) || m->r_max > 1)
    return CB_ERR_INVALID_ARG;
  double t_load = 0.0;
  long long n_total = n_query;
  for (int i = 0; i < n_chunks; ++i) {
    const cb_chunk_info& c = chunks[i];
    if (c.n_tokens < 0 || c.bytes < 0) return CB_ERR_INVALID_ARG;
    n_total += c.n_tokens;
    int act;
    if (c.tier == CB_TIER_DEVICE) {
      act = CB_ACT_USE;
    } else if (c.tier == CB_TIER_HOST) {
      const double tl = c.bytes / m->link_bytes_per_s + m->link_latency_s;
      act = tl < c.n_tokens * m->prefill_s_per_token ? CB_ACT_LOAD : CB_ACT_RECOMPUTE;
      if (act == CB_ACT_LOAD) t_load += tl;
    } else if (c.tier == CB_TIER_MISSING) {
      act = CB_ACT_RECOMPUTE;
    } else {
      return CB_ERR_INVALID_ARG;
    }
    actions_host[i] = act;
  }
  const double t_prefill = static_cast<double>(n_total) * m->prefill_s_per_token;
  double r = m->r_min;
  if (t_load > 0 && t_prefill > 0) r = std::fmin(m->r_max, std::fmax(m->r_min, (t_load - m->recompute_fixed_s) / t_prefill));
  *ratio_out = r;
  if (t_load_out) *t_load_out = t_load;
  if (t_recompute_out) *t_recompute_out = m->recompute_fixed_s + r * t_prefill;
  return CB_OK;
}

}  // extern "C"
