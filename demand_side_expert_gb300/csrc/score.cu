// Load Recalibration Metric of every routed pair.
//
// LRMoE Sec. 3.2 Prop. 3.1 Eq. 3 / Sec. 7.1 Eq. 12:
//   R_u = alpha_u^2 * ||g_t||^2 * ||phi_u||^2,
// the squared Frobenius norm of the rank-one contribution (alpha_u g_t) phi_u^T
// to the protected FC2 weight gradient, computed without forming it.
//
// One warp per token: the loads of the token's cotangent row g_t and of its
// K saved FC2-input rows phi_u (found through inv, up to 8 at a time) are all
// issued before any reduction, so some thirty 16-byte loads per lane are in
// flight. HBM-bound: every byte of g and phi is read exactly once with
// 128-bit streaming loads.
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

// Up to kRowsInFlight of the token's pairs are reduced per pass; the loads of
// g_t and of all those phi rows are issued before any reduction.
template <typename T>
__global__ void __launch_bounds__(kScoreThreads)
score_kernel(const T* __restrict__ g, const T* __restrict__ phi,
             const float* __restrict__ alpha, const int32_t* __restrict__ inv,
             float* __restrict__ score, int ntok, int D, int H, int K, int32_t* err) {
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

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_score(const lrm_shape* s, const void* g, const void* phi,
                                const float* alpha, const int32_t* inv, float* score,
                                void* ws, size_t ws_bytes, void* stream) {
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes)) != LRM_OK) return st;
  if (s->T == 0) return LRM_OK;
  if (!g || !phi || !alpha || !inv || !score) return LRM_ERR_INVALID_ARG;
  if (!aligned16(g) || !aligned16(phi)) return LRM_ERR_UNSUPPORTED;
  const int64_t warps = s->T;
  const int64_t cap = (int64_t)num_sms() * (2048 / kScoreThreads) * (kScoreThreads / 32);
  const int blocks = (int)((std::min(warps, cap) + 7) / 8);
  cudaStream_t cs = (cudaStream_t)stream;
  if (s->dtype == LRM_BF16)
    score_kernel<__nv_bfloat16><<<blocks, kScoreThreads, 0, cs>>>(
        (const __nv_bfloat16*)g, (const __nv_bfloat16*)phi, alpha, inv, score, s->T, s->D,
        s->H, s->K, error_word(ws));
  else
    score_kernel<float><<<blocks, kScoreThreads, 0, cs>>>(
        (const float*)g, (const float*)phi, alpha, inv, score, s->T, s->D, s->H, s->K,
        error_word(ws));
  return launch_status();
}
