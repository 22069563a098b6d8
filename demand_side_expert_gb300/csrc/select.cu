// Per-expert top-q selection of routed pairs by LRM score.
//
// LRMoE Alg. 1 (TopK inside each expert's pair set with its fixed quota)
// and Sec. 7.2 Prop. 7.1: for fixed per-expert drop counts, keeping the
// largest scores inside each expert minimises the summed isolated
// perturbation; solutions differ only among tied boundary scores, which are
// broken here by the lower pair index (= lower dispatch position inside a
// segment, the dispatch permutation being stable).
//
// One CTA per expert segment. Scores are non-negative floats, so their bit
// patterns order like the values: a 4-pass 8-bit radix select over the
// segment (staged once in shared memory) finds the q-th largest key tau and
// how many keys equal to tau must be kept; an ordered pass over warp-
// contiguous ranges (ballot ranks + a scan over warps) then writes the keep
// flags and the retained positions in ascending order.
#include <algorithm>

#include "common.cuh"

namespace lrm {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelSmemKeysMax = 40960;  // 160 KB of staged keys

// Exclusive scan of one value per warp (lane 0 holds it), returned to all lanes.
__device__ __forceinline__ int warp_values_exclusive_scan(int v, int* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    const int x = sh[lane];
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    sh[lane] = inc - x;
  }
  __syncthreads();
  const int r = sh[w];
  __syncthreads();
  return r;
}

__device__ __forceinline__ int block_sum(int v, int* sh) {
  v = __reduce_add_sync(0xffffffffu, v);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) sh[w] = v;
  __syncthreads();
  int r = 0;
  for (int i = 0; i < kSelWarps; ++i) r += sh[i];
  __syncthreads();
  return r;
}

// Quota of an expert with n routed pairs under RATE: min(ceil(num/den * n),
// cap), in exact integers (cap <= 0: none); otherwise the given quota.
template <bool RATE>
__device__ __forceinline__ int quota_of(const int32_t* quota, int j, int n, int num, int den,
                                        int cap) {
  if constexpr (RATE) {
    int q = (int)(((int64_t)num * n + den - 1) / den);
    return cap > 0 ? min(q, cap) : q;
  } else {
    return quota[j];
  }
}

// RATE: the quotas are computed from the rate num/den and the cap (and
// written to quota[e]) instead of read from quota.
template <bool RATE>
__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float* __restrict__ score, const int32_t* __restrict__ off,
              int32_t* __restrict__ quota, int num, int den, int cap, int E, int keys_cap,
              uint8_t* __restrict__ keep, int32_t* __restrict__ sel_off,
              int32_t* __restrict__ sel_pos, int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[256];
  __shared__ int scratch[kSelWarps];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

  // clamped quotas of all earlier experts -> this expert's output offset
  int part = 0;
  for (int j = tid; j < e; j += kSelThreads) {
    const int nj = max(off[j + 1] - off[j], 0);
    part += min(max(quota_of<RATE>(quota, j, nj, num, den, cap), 0), nj);
  }
  const int sel_base = block_sum(part, scratch);

  const int lo = off[e];
  int n = off[e + 1] - lo;
  if (n < 0) {
    if (tid == 0) flag_error(err, LRM_DEVERR_INDEX);
    n = 0;
  }
  int q = quota_of<RATE>(quota, e, n, num, den, cap);
  if constexpr (RATE) {
    if (tid == 0) quota[e] = q;
  }
  if (q < 0 || q > n) {
    if (tid == 0) flag_error(err, LRM_DEVERR_QUOTA);
    q = min(max(q, 0), n);
  }
  if (tid == 0) {
    sel_off[e] = sel_base;
    if (e == E - 1) sel_off[E] = sel_base + q;
  }
  if (q == n) {  // keep the whole segment (full retention)
    for (int i = tid; i < n; i += kSelThreads) {
      keep[lo + i] = 1;
      sel_pos[sel_base + i] = lo + i;
    }
    return;
  }
  if (q == 0) {
    for (int i = tid; i < n; i += kSelThreads) keep[lo + i] = 0;
    return;
  }

  const uint32_t* src = reinterpret_cast<const uint32_t*>(score + lo);
  if (n <= keys_cap) {
    for (int i = tid; i < n; i += kSelThreads) keys[i] = src[i];
    src = keys;
  }
  __syncthreads();

  // radix select of the q-th largest key, most significant digit first
  uint32_t prefix = 0, mask = 0;
  int remaining = q;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += kSelThreads) hist[b] = 0;
    __syncthreads();
    for (int base = w * 32; base < n; base += kSelThreads) {
      const int i = base + lane;
      uint32_t d = 0xffffffffu;
      if (i < n) {
        const uint32_t k = src[i];
        if ((k & mask) == prefix) d = (k >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (d != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
    }
    __syncthreads();
    if (w == 0) {  // lane l owns bins 255-8l .. 255-8l-7 (descending)
      uint32_t c[8];
      int sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sum += (int)c[j];
      }
      int inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      const int exc = inc - sum;
      const uint32_t hit = __ballot_sync(0xffffffffu, exc < remaining && remaining <= inc);
      if (lane == __ffs(hit) - 1) {
        int acc = exc;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + (int)c[j] >= remaining) {
            s_prefix = prefix | ((uint32_t)(255 - 8 * lane - j) << shift);
            s_remaining = remaining - acc;
            break;
          }
          acc += (int)c[j];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t tau = prefix;
  const int need_eq = remaining;  // keys equal to tau to keep, lowest positions first

  // ordered keep pass over warp-contiguous ranges
  const int per_warp = (((n + kSelWarps - 1) / kSelWarps) + 31) & ~31;
  const int w_lo = min(w * per_warp, n), w_hi = min(w_lo + per_warp, n);
  int cnt_eq = 0;
  for (int b = w_lo; b < w_hi; b += 32) {
    const int i = b + lane;
    cnt_eq += __popc(__ballot_sync(0xffffffffu, i < w_hi && src[i] == tau));
  }
  const int eq_base = warp_values_exclusive_scan(cnt_eq, scratch);
  int eq_run = eq_base, cnt_kept = 0;
  for (int b = w_lo; b < w_hi; b += 32) {
    const int i = b + lane;
    const uint32_t k = i < w_hi ? src[i] : 0u;
    const bool eq = i < w_hi && k == tau;
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const bool kept = i < w_hi && (k > tau || (eq && eq_run + __popc(beq & lanemask_lt()) < need_eq));
    cnt_kept += __popc(__ballot_sync(0xffffffffu, kept));
    eq_run += __popc(beq);
  }
  const int kept_base = warp_values_exclusive_scan(cnt_kept, scratch);
  eq_run = eq_base;
  int kept_run = kept_base;
  for (int b = w_lo; b < w_hi; b += 32) {
    const int i = b + lane;
    const uint32_t k = i < w_hi ? src[i] : 0u;
    const bool eq = i < w_hi && k == tau;
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const bool kept = i < w_hi && (k > tau || (eq && eq_run + __popc(beq & lanemask_lt()) < need_eq));
    const uint32_t bk = __ballot_sync(0xffffffffu, kept);
    if (i < w_hi) {
      keep[lo + i] = kept ? 1 : 0;
      if (kept) sel_pos[sel_base + kept_run + __popc(bk & lanemask_lt())] = lo + i;
    }
    kept_run += __popc(bk);
    eq_run += __popc(beq);
  }
}

}  // namespace lrm

using namespace lrm;

template <bool RATE>
static lrm_status select_entry(const lrm_shape* s, const float* score, const int32_t* off,
                               int32_t* quota, int num, int den, int cap, uint8_t* keep,
                               int32_t* sel_off, int32_t* sel_pos, void* ws, size_t ws_bytes,
                               void* stream) {
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes)) != LRM_OK) return st;
  const int64_t N = (int64_t)s->T * s->K;
  if (!off || !quota || !sel_off) return LRM_ERR_INVALID_ARG;
  if (N > 0 && (!score || !keep || !sel_pos)) return LRM_ERR_INVALID_ARG;
  if (RATE && (den <= 0 || num < 0 || num > den)) return LRM_ERR_INVALID_ARG;
  const int keys_cap = (int)std::min<int64_t>(std::max(s->T, 1), kSelSmemKeysMax);
  const size_t smem = (size_t)keys_cap * 4;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(select_kernel<RATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
  launch_k(select_kernel<RATE>, dim3(s->E), dim3(kSelThreads), smem, (cudaStream_t)stream,
           score, off, quota, num, den, cap, s->E, keys_cap, keep, sel_off, sel_pos,
           error_word(ws));
  return launch_status();
}

extern "C" lrm_status lrm_select_quota(const lrm_shape* s, const float* score,
                                       const int32_t* off, const int32_t* quota,
                                       uint8_t* keep, int32_t* sel_off, int32_t* sel_pos,
                                       void* ws, size_t ws_bytes, void* stream) {
  return select_entry<false>(s, score, off, const_cast<int32_t*>(quota), 0, 1, 0, keep,
                             sel_off, sel_pos, ws, ws_bytes, stream);
}

extern "C" lrm_status lrm_select_rate(const lrm_shape* s, const float* score,
                                      const int32_t* off, int32_t num, int32_t den, int32_t cap,
                                      int32_t* quota, uint8_t* keep, int32_t* sel_off,
                                      int32_t* sel_pos, void* ws, size_t ws_bytes,
                                      void* stream) {
  return select_entry<true>(s, score, off, quota, num, den, cap, keep, sel_off, sel_pos, ws,
                            ws_bytes, stream);
}
