// HKVD selection: block-wide top-k by (deviation descending, token index ascending),
// emitted as an ascending index list.  One thread block per request.
//
// Each candidate gets a unique 64-bit key: the order-preserving bit pattern of its fp32
// deviation in the high word and the complement of its token index in the low word, so
// "larger key" means "ranks higher" and no two keys are equal.  An 8-pass radix select
// (8 bits per pass, 256-bin shared histogram) finds the k-th largest key T exactly; the
// selected set is {key >= T}.  An ordered compaction (block prefix scan over contiguous
// per-thread ranges) then writes the selected rows in their original ascending order.
#include "common.cuh"
#include "internal.h"

namespace cb {

constexpr int SEL_THREADS = 1024;

__device__ __forceinline__ uint32_t ord_f32(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Key of one candidate; NaN ranks below every number and raises ST_NAN.
__device__ __forceinline__ uint64_t sel_key(float dev, int32_t idx, int32_t* status) {
  uint32_t hi;
  if (isnan(dev)) {
    set_status(status, ST_NAN);
    hi = 0u;
  } else {
    hi = ord_f32(dev);
  }
  return (static_cast<uint64_t>(hi) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

struct SelShared {
  unsigned int hist[256];
  unsigned long long prefix;
  unsigned long long mask;
  unsigned int rem;
  int warp_tot[32];
  int total;
};

// k-th largest key among the items for which Item::cand(j) is true (k >= 1, k <= count).
template <typename Item>
__device__ uint64_t radix_select_kth(const Item& it, int n, int k, SelShared& sh) {
  if (threadIdx.x == 0) {
    sh.prefix = 0ull;
    sh.mask = 0ull;
    sh.rem = static_cast<unsigned int>(k);
  }
  __syncthreads();
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) sh.hist[b] = 0u;
    __syncthreads();
    const uint64_t prefix = sh.prefix, mask = sh.mask;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      if (!it.cand(j)) continue;
      const uint64_t key = it.key(j);
      if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned int rem = sh.rem, cum = 0u;
      int digit = 0;
      for (int dgt = 255; dgt >= 0; --dgt) {
        const unsigned int c = sh.hist[dgt];
        if (cum + c >= rem) {
          digit = dgt;
          break;
        }
        cum += c;
      }
      sh.rem = rem - cum;
      sh.prefix = prefix | (static_cast<uint64_t>(digit) << shift);
      sh.mask = mask | (255ull << shift);
    }
    __syncthreads();
  }
  return sh.prefix;
}

// Writes out[pos] for every j with take(j), in increasing j; returns the count.
template <typename Take, typename Emit>
__device__ int ordered_compact(int n, const Take& take, const Emit& emit, SelShared& sh) {
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int j0 = threadIdx.x * per;
  const int j1 = min(n, j0 + per);
  int cnt = 0;
  for (int j = j0; j < j1; ++j) cnt += take(j) ? 1 : 0;
  // exclusive block scan of cnt
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh.warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    int v = lane < nw ? sh.warp_tot[lane] : 0;
    int iv = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, iv, o);
      if (lane >= o) iv += t;
    }
    if (lane < nw) sh.warp_tot[lane] = iv - v;  // exclusive warp offsets
    if (lane == nw - 1) sh.total = iv;
  }
  __syncthreads();
  int pos = sh.warp_tot[w] + incl - cnt;
  for (int j = j0; j < j1; ++j)
    if (take(j)) emit(j, pos++);
  __syncthreads();
  return sh.total;
}

// ----------------------------------------------------------------------------- standalone
struct PlainItem {
  const float* dev;
  const int32_t* cand_idx;
  int32_t* status;
  __device__ bool cand(int) const { return true; }
  __device__ int32_t idx(int j) const { return cand_idx ? cand_idx[j] : j; }
  __device__ uint64_t key(int j) const { return sel_key(dev[j], idx(j), status); }
};

__global__ void __launch_bounds__(SEL_THREADS) select_plain_kernel(const float* __restrict__ dev,
                                                                   const int32_t* __restrict__ cand, int n, int k,
                                                                   int32_t* __restrict__ out, int32_t* status) {
  __shared__ SelShared sh;
  PlainItem it{dev, cand, status};
  if (k <= 0) return;
  uint64_t thr = 0ull;
  if (k < n) thr = radix_select_kth(it, n, k, sh);
  // NaN check also for k >= n (every item is taken)
  if (k >= n)
    for (int j = threadIdx.x; j < n; j += blockDim.x)
      if (isnan(dev[j])) set_status(status, ST_NAN);
  auto take = [&](int j) { return k >= n || it.key(j) >= thr; };
  auto emit = [&](int j, int p) { out[p] = it.idx(j); };
  ordered_compact(n, take, emit, sh);
}

cudaError_t launch_select_plain(const float* dev, const int32_t* cand, int n, int k, int32_t* sel_out,
                                int32_t* status, cudaStream_t s) {
  if (n <= 0 || k <= 0) return cudaSuccess;
  select_plain_kernel<<<1, SEL_THREADS, 0, s>>>(dev, cand, n, k, sel_out, status);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- batched (one block per request)
// Rows of R for request r are r_off..r_off+r_n-1 with ascending positions r_pos.  Cached
// rows (position < Nc) are candidates; query rows are always kept.  Output: the rows of S
// (ascending): s_src = row of R, s_pos = token position, s_req = r, written at s_off.
struct BatchItem {
  const float* dev;
  const int32_t* pos;
  int n_cached;
  int32_t* status;
  __device__ bool cand(int j) const { return pos[j] < n_cached; }
  __device__ uint64_t key(int j) const { return sel_key(dev[j], pos[j], status); }
};

__device__ __forceinline__ bool in_sorted(const int32_t* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < x)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo < n && a[lo] == x;
}

__global__ void __launch_bounds__(SEL_THREADS) select_batched_kernel(const float* __restrict__ dev,
                                                                     const int32_t* __restrict__ r_pos,
                                                                     const PlanEntry* __restrict__ plan,
                                                                     const ReqDev* __restrict__ reqs,
                                                                     const int32_t* __restrict__ forced,
                                                                     int32_t* __restrict__ s_src,
                                                                     int32_t* __restrict__ s_pos,
                                                                     int32_t* __restrict__ s_req, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ SelShared sh;
  const int r = blockIdx.x;
  const PlanEntry pe = plan[r];
  const int nc = reqs[r].n_cached;
  const float* d = dev + pe.r_off;
  const int32_t* pos = r_pos + pe.r_off;
  BatchItem it{d, pos, nc, status};
  const int n = pe.r_n;
  const int k = pe.k;
  int n_cand = 0;  // number of cached rows (all cached rows precede the query rows)
  {
    // count candidates: positions ascend, so the cached rows form a prefix
    int lo = 0, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (pos[mid] < nc)
        lo = mid + 1;
      else
        hi = mid;
    }
    n_cand = lo;
  }
  uint64_t thr = 0ull;
  const bool use_forced = pe.forced_off >= 0;
  if (!use_forced && k > 0 && k < n_cand) thr = radix_select_kth(it, n_cand, k, sh);
  if (!use_forced && k >= n_cand)
    for (int j = threadIdx.x; j < n_cand; j += blockDim.x)
      if (isnan(d[j])) set_status(status, ST_NAN);
  const int32_t* fs = use_forced ? forced + pe.forced_off : nullptr;
  auto take = [&](int j) {
    if (j >= n_cand) return true;  // query rows
    if (use_forced) return in_sorted(fs, k, pos[j]);
    if (k <= 0) return false;
    if (k >= n_cand) return true;
    return it.key(j) >= thr;
  };
  auto emit = [&](int j, int p) {
    if (p < pe.s_n) {
      s_src[pe.s_off + p] = pe.r_off + j;
      s_pos[pe.s_off + p] = pos[j];
      s_req[pe.s_off + p] = r;
    }
  };
  const int total = ordered_compact(n, take, emit, sh);
  if (total != pe.s_n) {
    // a forced set that is not a subset of R: flag it and fill the planned rows with the
    // last row of R (a query row) so that every later kernel reads valid positions
    if (threadIdx.x == 0) set_status(status, ST_RANGE);
    for (int p = total + static_cast<int>(threadIdx.x); p < pe.s_n; p += blockDim.x) {
      s_src[pe.s_off + p] = pe.r_off + n - 1;
      s_pos[pe.s_off + p] = pos[n - 1];
      s_req[pe.s_off + p] = r;
    }
  }
}

cudaError_t launch_select_batched(const float* dev, const int32_t* r_pos, const PlanEntry* plan, const ReqDev* reqs,
                                  const int32_t* forced, int n_req, int32_t* s_src, int32_t* s_pos, int32_t* s_req,
                                  int32_t* status, cudaStream_t s) {
  if (n_req <= 0) return cudaSuccess;
  launch_chain(select_batched_kernel, dim3(n_req), dim3(SEL_THREADS), 0, s, dev, r_pos, plan, reqs, forced, s_src, s_pos, s_req, status);
  return cudaGetLastError();
}

}  // namespace cb
