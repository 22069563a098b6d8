// Load Recalibration Metric of every routed pair.
//
// LRMoE Sec. 3.2 Prop. 3.1 Eq. 3 / Sec. 7.1 Eq. 12:
//   R_u = alpha_u^2 * ||g_t||^2 * ||phi_u||^2,
// the squared Frobenius norm of the rank-one contribution (alpha_u g_t) phi_u^T
// to the protected FC2 weight gradient, computed without forming it.
//
// One warp per token. HBM-bound: every byte of g and phi is read exactly once
// with 128-bit streaming loads. The time is set by how many bytes each SM
// keeps in flight: for BF16 layers with up to 8 routed experts per token the
// kernel is instantiated with compile-time counts of 16-byte chunks per lane
// (GV for the cotangent row g_t, HV for each saved FC2-input row phi_u), so
// every load of the token is issued before any reduction (one memory round
// trip per token); other shapes take a generic kernel that sweeps the rows
// with runtime bounds.
#include <algorithm>

#include "common.cuh"

namespace lrm {

constexpr int kScoreThreads = 256;
constexpr int kRowsInFlight = 8;

template <typename T>
__device__ __forceinline__ float row_sq_partial(const T* row, int n_vec, int lane) {
  constexpr int V = Vec16<T>::kElems;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  const uint4* r = reinterpret_cast<const uint4*>(row);
#pragma unroll 4
  for (int c = lane; c < n_vec; c += 32) {
    float f[V];
    Vec16<T>::unpack(ld_stream(r + c), f);
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = fmaf(f[i], f[i], acc[i]);
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) s += acc[i];
  return s;
}

// Sum of squares of one 16-byte vector of activations.
template <typename T>
__device__ __forceinline__ float sum_sq(const uint4& v) {
  constexpr int V = Vec16<T>::kElems;
  float f[V];
  Vec16<T>::unpack(v, f);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) s = fmaf(f[i], f[i], s);
  return s;
}

template <typename T>
__device__ __forceinline__ float row_abs_partial(const T* row, int n_vec, int lane) {
  constexpr int V = Vec16<T>::kElems;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  const uint4* r = reinterpret_cast<const uint4*>(row);
#pragma unroll 4
  for (int c = lane; c < n_vec; c += 32) {
    float f[V];
    Vec16<T>::unpack(ld_stream(r + c), f);
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] += fabsf(f[i]);
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) s += acc[i];
  return s;
}

// SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): mix of the state after
// its increment; the random criterion of pair p is output p+1 for `seed`.
__device__ __forceinline__ float random_score(uint64_t seed, uint64_t p) {
  uint64_t z = seed + (p + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return (float)(z >> 40) * (1.0f / 16777216.0f);
}

// Up to kRowsInFlight of the token's pairs are reduced per pass; the loads of
// g_t and of all those phi rows are issued before any reduction. The other
// criteria of LRMoE Sec. 4.7 read g_t only (or nothing, for the random one).
template <typename T, int METRIC>
__global__ void __launch_bounds__(kScoreThreads)
score_kernel(const T* __restrict__ g, const T* __restrict__ phi,
             const float* __restrict__ alpha, const int32_t* __restrict__ inv,
             float* __restrict__ score, int ntok, int D, int H, int K, uint64_t seed,
             int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  constexpr int V = Vec16<T>::kElems;
  const int lane = threadIdx.x & 31;
  const int64_t N = (int64_t)ntok * K;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int gv = D / V, hv = H / V;
  for (int64_t t = warp; t < ntok; t += nwarps) {
    // the token's dispatch positions, lane k holding slot k
    int my_pos = -1;
    if (lane < K) {
      const int q = inv[t * K + lane];
      if (q >= 0 && q < N) my_pos = q;
      else flag_error(err, LRM_DEVERR_INDEX);
    }
    if constexpr (METRIC != LRM_METRIC_LRM) {
      float tok = 0.f;
      if constexpr (METRIC == LRM_METRIC_GRAD_SQ)
        tok = warp_sum(row_sq_partial(g + t * D, gv, lane));
      if constexpr (METRIC == LRM_METRIC_GRAD_ABS)
        tok = warp_sum(row_abs_partial(g + t * D, gv, lane));
      if (lane < K && my_pos >= 0) {
        if constexpr (METRIC == LRM_METRIC_RANDOM)
          tok = random_score(seed, (uint64_t)t * K + lane);
        score[my_pos] = tok;
      }
      continue;
    }
    float gpart = 0.f;
    for (int k0 = 0; k0 < K; k0 += kRowsInFlight) {
      int pos[kRowsInFlight];
#pragma unroll
      for (int r = 0; r < kRowsInFlight; ++r) {
        pos[r] = __shfl_sync(0xffffffffu, my_pos, (k0 + r) & 31);
        if (k0 + r >= K) pos[r] = -1;
      }
      float part[kRowsInFlight];
      if (k0 == 0) gpart = row_sq_partial(g + t * D, gv, lane);  // issued with the rows
#pragma unroll
      for (int r = 0; r < kRowsInFlight; ++r)
        part[r] = pos[r] >= 0 ? row_sq_partial(phi + (int64_t)pos[r] * H, hv, lane) : 0.f;
      const float gsq = warp_sum(gpart);
#pragma unroll
      for (int r = 0; r < kRowsInFlight; ++r) {
        const float psq = warp_sum(part[r]);
        if (lane == 0 && pos[r] >= 0) {
          const float a = alpha[t * K + k0 + r];
          score[pos[r]] = (a * a) * gsq * psq;
        }
      }
    }
  }
}

// LRM score with every load of the token issued up front: GV 16-byte chunks
// of g_t and HV of each of the token's (at most 8) phi rows per lane,
// predicated on the actual row lengths (D / 8 and H / 8 chunks).
constexpr int kUpfrontThreads = 128;

template <int GV, int HV>
__global__ void __launch_bounds__(kUpfrontThreads)
score_upfront_kernel(const __nv_bfloat16* __restrict__ g, const __nv_bfloat16* __restrict__ phi,
                     const float* __restrict__ alpha, const int32_t* __restrict__ inv,
                     float* __restrict__ score, int ntok, int D, int H, int K, int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  const int lane = threadIdx.x & 31;
  const int64_t N = (int64_t)ntok * K;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int gv = D / 8, hv = H / 8;
  for (int64_t t = warp; t < ntok; t += nwarps) {
    // lane k: dispatch position of slot k; a bad entry is flagged, its row
    // read at position 0 and its score not written
    int my_pos = 0, my_dst = -1;
    if (lane < K) {
      const int q = inv[t * K + lane];
      if (q >= 0 && q < N) my_pos = my_dst = q;
      else flag_error(err, LRM_DEVERR_INDEX);
    }
    const uint4* grow = reinterpret_cast<const uint4*>(g + t * D);
    uint4 vg[GV], vp[kRowsInFlight][HV];
#pragma unroll
    for (int i = 0; i < GV; ++i) {
      const int c = lane + 32 * i;
      vg[i] = c < gv ? ld_stream(grow + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int r = 0; r < kRowsInFlight; ++r) {
      const int pos = __shfl_sync(0xffffffffu, my_pos, r);
      const uint4* prow = reinterpret_cast<const uint4*>(phi + (int64_t)pos * H);
#pragma unroll
      for (int i = 0; i < HV; ++i) {
        const int c = lane + 32 * i;
        vp[r][i] = (r < K && c < hv) ? ld_stream(prow + c) : make_uint4(0, 0, 0, 0);
      }
    }
    float gpart = 0.f;
#pragma unroll
    for (int i = 0; i < GV; ++i) gpart += sum_sq<__nv_bfloat16>(vg[i]);
    const float gsq = warp_sum(gpart);
#pragma unroll
    for (int r = 0; r < kRowsInFlight; ++r) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < HV; ++i) part += sum_sq<__nv_bfloat16>(vp[r][i]);
      const float psq = warp_sum(part);
      const int dst = __shfl_sync(0xffffffffu, my_dst, r);
      if (lane == 0 && dst >= 0) {
        const float a = alpha[t * K + r];
        score[dst] = (a * a) * gsq * psq;
      }
    }
  }
}

// The smallest instantiation that covers the layer (chunks per lane), or
// nullptr when none does (then the generic kernel runs).
using UpfrontKernel = void (*)(const __nv_bfloat16*, const __nv_bfloat16*, const float*,
                               const int32_t*, float*, int, int, int, int, int32_t*);

static UpfrontKernel pick_upfront(int D, int H, int K) {
  if (K > kRowsInFlight) return nullptr;
  const int gl = (D / 8 + 31) / 32, hl = (H / 8 + 31) / 32;
#define LRM_UPFRONT(GVv, HVv) \
  if (gl <= GVv && hl <= HVv) return score_upfront_kernel<GVv, HVv>;
  if (gl <= 8) {
    LRM_UPFRONT(8, 1) LRM_UPFRONT(8, 2) LRM_UPFRONT(8, 3) LRM_UPFRONT(8, 4) LRM_UPFRONT(8, 6)
  }
  if (gl <= 16) {
    LRM_UPFRONT(16, 1) LRM_UPFRONT(16, 2) LRM_UPFRONT(16, 3) LRM_UPFRONT(16, 4)
    LRM_UPFRONT(16, 6)
  }
#undef LRM_UPFRONT
  return nullptr;
}

template <typename T>
static void launch_score(const lrm_shape* s, int metric, uint64_t seed, const void* g,
                         const void* phi, const float* alpha, const int32_t* inv, float* score,
                         int32_t* err, int blocks, cudaStream_t cs) {
  const T* gt = (const T*)g;
  const T* pt = (const T*)phi;
  switch (metric) {
    case LRM_METRIC_GRAD_SQ:
      launch_k(score_kernel<T, LRM_METRIC_GRAD_SQ>, dim3(blocks), dim3(kScoreThreads), 0, cs, 
          gt, pt, alpha, inv, score, s->T, s->D, s->H, s->K, seed, err);
      break;
    case LRM_METRIC_GRAD_ABS:
      launch_k(score_kernel<T, LRM_METRIC_GRAD_ABS>, dim3(blocks), dim3(kScoreThreads), 0, cs, 
          gt, pt, alpha, inv, score, s->T, s->D, s->H, s->K, seed, err);
      break;
    case LRM_METRIC_RANDOM:
      launch_k(score_kernel<T, LRM_METRIC_RANDOM>, dim3(blocks), dim3(kScoreThreads), 0, cs, 
          gt, pt, alpha, inv, score, s->T, s->D, s->H, s->K, seed, err);
      break;
    default:
      launch_k(score_kernel<T, LRM_METRIC_LRM>, dim3(blocks), dim3(kScoreThreads), 0, cs, 
          gt, pt, alpha, inv, score, s->T, s->D, s->H, s->K, seed, err);
  }
}

}  // namespace lrm

using namespace lrm;

static lrm_status score_entry(const lrm_shape* s, int metric, uint64_t seed, const void* g,
                              const void* phi, const float* alpha, const int32_t* inv,
                              float* score, void* ws, size_t ws_bytes, void* stream) {
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes)) != LRM_OK) return st;
  if (metric < LRM_METRIC_LRM || metric > LRM_METRIC_RANDOM) return LRM_ERR_INVALID_ARG;
  if (s->T == 0) return LRM_OK;
  const bool needs_g = metric != LRM_METRIC_RANDOM;
  const bool needs_phi = metric == LRM_METRIC_LRM;
  if (!inv || !score || (needs_g && !g) || (needs_phi && (!phi || !alpha)))
    return LRM_ERR_INVALID_ARG;
  if ((needs_g && !aligned16(g)) || (needs_phi && !aligned16(phi))) return LRM_ERR_UNSUPPORTED;
  const int64_t warps = s->T;
  cudaStream_t cs = (cudaStream_t)stream;
  if (s->dtype == LRM_BF16 && metric == LRM_METRIC_LRM) {
    if (UpfrontKernel kern = pick_upfront(s->D, s->H, s->K)) {
      // a warp per token, all of them at once where the grid allows
      const int64_t per_cta = kUpfrontThreads / 32;
      const int64_t cap = (int64_t)num_sms() * 64;
      const int blocks = (int)std::min((warps + per_cta - 1) / per_cta, cap);
      launch_k(kern, dim3(blocks), dim3(kUpfrontThreads), 0, cs, (const __nv_bfloat16*)g,
               (const __nv_bfloat16*)phi, alpha, inv, score, s->T, s->D, s->H, s->K,
               error_word(ws));
      return launch_status();
    }
  }
  const int64_t cap = (int64_t)num_sms() * (2048 / kScoreThreads) * (kScoreThreads / 32);
  const int blocks = (int)((std::min(warps, cap) + 7) / 8);
  if (s->dtype == LRM_BF16)
    launch_score<__nv_bfloat16>(s, metric, seed, g, phi, alpha, inv, score, error_word(ws),
                                blocks, cs);
  else
    launch_score<float>(s, metric, seed, g, phi, alpha, inv, score, error_word(ws), blocks, cs);
  return launch_status();
}

extern "C" lrm_status lrm_score(const lrm_shape* s, const void* g, const void* phi,
                                const float* alpha, const int32_t* inv, float* score,
                                void* ws, size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_score");
  return score_entry(s, LRM_METRIC_LRM, 0, g, phi, alpha, inv, score, ws, ws_bytes, stream);
}

extern "C" lrm_status lrm_score_variant(const lrm_shape* s, int32_t metric, uint64_t seed,
                                        const void* g, const void* phi, const float* alpha,
                                        const int32_t* inv, float* score, void* ws,
                                        size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_score_variant");
  return score_entry(s, metric, seed, g, phi, alpha, inv, score, ws, ws_bytes, stream);
}
