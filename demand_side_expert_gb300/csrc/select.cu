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
// patterns order like the values: an 8-bit radix select (at most four
// passes, most significant byte first, per-warp digit counts) finds the q-th
// largest key tau and how many keys equal to tau must be kept. The first
// pass runs while the segment is staged in shared memory; the later ones scan
// only the keys of the first pass's bucket (copied to a candidate buffer when
// they fit), and the passes stop once the bucket holding the q-th key is kept
// whole. An ordered pass over warp-contiguous ranges (ballot ranks and two
// scans over warps) then writes the keep flags and the retained positions in
// ascending order.
#include <algorithm>

#include "common.cuh"

namespace lrm {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelSmemKeysMax = 40960;  // 160 KB of staged keys
// dynamic shared memory for the staged keys and the candidates (the static
// per-warp histograms take another 32 KB of the 227 KB)
constexpr size_t kSelSmemDynBytes = 190 * 1024;

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

// Per-warp digit counts, so warps never contend for a bin (a segment's keys
// share only a few top bytes, and one shared histogram serialised every warp
// on them). Every lane adds its own key with a shared-memory atomic:
// aggregating equal digits first with match_any measured 2.4x (top byte) to
// 5.7x (lower bytes) slower on a 32,708-key segment.
__device__ __forceinline__ void count_digit(uint32_t* wh, bool valid, uint32_t k, uint32_t mask,
                                            uint32_t prefix, int shift) {
  if (valid && (k & mask) == prefix) atomicAdd(&wh[(k >> shift) & 255u], 1u);
}

// RATE: the quotas are computed from the rate num/den and the cap (and
// written to quota[e]) instead of read from quota.
//
// Radix select of the q-th largest key, most significant byte first. Each
// warp owns a contiguous range of the segment; the first pass runs while the
// keys are staged in shared memory. If the bucket holding the q-th key after
// the first pass fits in the candidate buffer, its keys are copied there (in
// segment order, at offsets from the warps' own counts) and the later passes
// scan only them. The passes stop as soon as the bucket holding the q-th key
// is kept whole; the keep pass then compares keys on the bits decided so far.
template <bool RATE>
__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float* __restrict__ score, const int32_t* __restrict__ off,
              int32_t* __restrict__ quota, int num, int den, int cap, int E, int keys_cap,
              int cand_cap, uint8_t* __restrict__ keep, int32_t* __restrict__ sel_off,
              int32_t* __restrict__ sel_pos, int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  extern __shared__ uint32_t keys[];  // [keys_cap] the segment, then [cand_cap] candidates
  uint32_t* cand = keys + keys_cap;
  __shared__ uint32_t whist[kSelWarps * 256];  // per-warp digit counts
  __shared__ uint32_t hist[256];
  __shared__ int scratch[kSelWarps];
  __shared__ int cand_base[kSelWarps];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining, s_bucket;
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

  // warp-contiguous ranges (multiples of 32) of a set of m keys
  auto range = [&](int m, int& r_lo, int& r_hi) {
    const int per = (((m + kSelWarps - 1) / kSelWarps) + 31) & ~31;
    r_lo = min(w * per, m);
    r_hi = min(r_lo + per, m);
  };
  // per-warp counts -> hist; warp 0 then finds the bin holding the
  // remaining-th largest key among those matching the prefix
  auto find_digit = [&](uint32_t prefix, int remaining, int shift) {
    __syncthreads();
    if (tid < 256) {
      uint32_t t = 0;
#pragma unroll 8
      for (int v = 0; v < kSelWarps; ++v) t += whist[v * 256 + tid];
      hist[tid] = t;
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
            s_bucket = (int)c[j];
            break;
          }
          acc += (int)c[j];
        }
      }
    }
    __syncthreads();
  };

  // pass 1 (top byte), fused with staging the keys in shared memory
  const uint32_t* gsrc = reinterpret_cast<const uint32_t*>(score + lo);
  const bool staged = n <= keys_cap;
  int r_lo, r_hi;
  range(n, r_lo, r_hi);
  for (int i = tid; i < kSelWarps * 256; i += kSelThreads) whist[i] = 0;
  __syncthreads();
  {
    constexpr int U = 8;  // keys per lane in flight
    for (int b0 = r_lo; b0 < r_hi; b0 += 32 * U) {
      uint32_t kk[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b0 + 32 * u + lane;
        kk[u] = i < r_hi ? gsrc[i] : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b0 + 32 * u + lane;
        if (staged && i < r_hi) keys[i] = kk[u];
        count_digit(whist + w * 256, i < r_hi, kk[u], 0u, 0u, 24);
      }
    }
  }
  const uint32_t* src = staged ? keys : gsrc;
  find_digit(0u, q, 24);
  uint32_t prefix = s_prefix, mask = 0xff000000u;
  int remaining = s_remaining;
  bool done = s_bucket == remaining;  // the bucket is kept whole

  // the later passes scan the first pass's bucket only, if it fits
  const uint32_t* cur = src;
  int cur_n = n;
  if (!done && s_bucket <= cand_cap) {
    const uint32_t d1 = prefix >> 24;
    if (w == 0) {
      const int v = (int)whist[lane * 256 + d1];
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      cand_base[lane] = inc - v;
    }
    __syncthreads();
    int run = cand_base[w];
    for (int b = r_lo; b < r_hi; b += 32) {
      const int i = b + lane;
      const uint32_t k = i < r_hi ? src[i] : 0u;
      const bool m = i < r_hi && (k >> 24) == d1;
      const uint32_t bm = __ballot_sync(0xffffffffu, m);
      if (m) cand[run + __popc(bm & lanemask_lt())] = k;
      run += __popc(bm);
    }
    cur = cand;
    cur_n = s_bucket;
  }

  for (int shift = 16; shift >= 0 && !done; shift -= 8) {
    for (int i = tid; i < kSelWarps * 256; i += kSelThreads) whist[i] = 0;
    __syncthreads();  // also: candidates written before they are read
    int c_lo, c_hi;
    range(cur_n, c_lo, c_hi);
    for (int b = c_lo; b < c_hi; b += 32) {
      const int i = b + lane;
      count_digit(whist + w * 256, i < c_hi, i < c_hi ? cur[i] : 0u, mask, prefix, shift);
    }
    find_digit(prefix, remaining, shift);
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
    done = s_bucket == remaining;
  }
  // keep the keys whose decided bits exceed tau, and the first need_eq keys
  // (lowest positions) whose decided bits equal it
  const uint32_t tau = prefix;
  const int need_eq = remaining;

  // ordered keep pass over the warp-contiguous ranges of the segment
  // (ballot ranks inside a warp, a scan over warps for each warp's base)
  int cnt_eq = 0, cnt_gt = 0;
  for (int b = r_lo; b < r_hi; b += 32) {
    const int i = b + lane;
    const uint32_t k = i < r_hi ? (src[i] & mask) : 0u;
    cnt_eq += __popc(__ballot_sync(0xffffffffu, i < r_hi && k == tau));
    cnt_gt += __popc(__ballot_sync(0xffffffffu, i < r_hi && k > tau));
  }
  const int eq_base = warp_values_exclusive_scan(cnt_eq, scratch);
  const int kept_w = cnt_gt + min(max(need_eq - eq_base, 0), cnt_eq);
  const int kept_base = warp_values_exclusive_scan(kept_w, scratch);
  int eq_run = eq_base, kept_run = kept_base;
  for (int b = r_lo; b < r_hi; b += 32) {
    const int i = b + lane;
    const uint32_t k = i < r_hi ? (src[i] & mask) : 0u;
    const bool eq = i < r_hi && k == tau;
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const bool kept = i < r_hi && (k > tau || (eq && eq_run + __popc(beq & lanemask_lt()) < need_eq));
    const uint32_t bk = __ballot_sync(0xffffffffu, kept);
    if (i < r_hi) {
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
  const int cand_cap =
      std::min(keys_cap, (int)((kSelSmemDynBytes - (size_t)keys_cap * 4) / 4));
  const size_t smem = (size_t)(keys_cap + cand_cap) * 4;
  // the static 34 KB count against the default 48 KB too
  if (smem > 8 * 1024)
    cudaFuncSetAttribute(select_kernel<RATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
  launch_k(select_kernel<RATE>, dim3(s->E), dim3(kSelThreads), smem, (cudaStream_t)stream,
           score, off, quota, num, den, cap, s->E, keys_cap, cand_cap, keep, sel_off, sel_pos,
           error_word(ws));
  return launch_status();
}

extern "C" lrm_status lrm_select_quota(const lrm_shape* s, const float* score,
                                       const int32_t* off, const int32_t* quota,
                                       uint8_t* keep, int32_t* sel_off, int32_t* sel_pos,
                                       void* ws, size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_select_quota");
  return select_entry<false>(s, score, off, const_cast<int32_t*>(quota), 0, 1, 0, keep,
                             sel_off, sel_pos, ws, ws_bytes, stream);
}

extern "C" lrm_status lrm_select_rate(const lrm_shape* s, const float* score,
                                      const int32_t* off, int32_t num, int32_t den, int32_t cap,
                                      int32_t* quota, uint8_t* keep, int32_t* sel_off,
                                      int32_t* sel_pos, void* ws, size_t ws_bytes,
                                      void* stream) {
  LRM_NVTX("lrm_select_rate");
  return select_entry<true>(s, score, off, quota, num, den, cap, keep, sel_off, sel_pos, ws,
                            ws_bytes, stream);
}
