// Forward expert pass that produces the saved state: token gather into
// dispatch order, the two grouped expert products, and the weighted combine.
//
// LRMoE Sec. 3.1 (design overview) and Alg. 1 (FullForwardAndSaveContext):
// the full forward dispatches every routed pair, runs its expert and combines
// the outputs, keeping the intermediates the backward reads ([a | b] and
// phi, in dispatch order). LLEP Sec. 2.1: the token rows are re-indexed into
// per-expert groups, each group runs one product per expert, and the MoE
// output is the routing-weighted sum of the selected experts' outputs.
// The gate/up product also serves the retained-only recompute of the
// backward (RelayMoE Sec. 3.3): run over the compacted rows, it rebuilds
// [a | b] of the retained pairs without saved state.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace lrm {

// x_disp[pos] = x[perm[pos] / K]: one warp per dispatch row, 16-byte copies.
__global__ void __launch_bounds__(256)
gather_tokens_kernel(const int32_t* __restrict__ perm, const uint4* __restrict__ x,
                     uint4* __restrict__ x_disp, int64_t N, int K, int64_t ntok, int vec_per_row,
                     int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t pos = warp; pos < N; pos += nwarps) {
    const int p = perm[pos];
    if (p < 0 || p >= N) {
      if (lane == 0) flag_error(err, LRM_DEVERR_INDEX);
      continue;
    }
    const int64_t t = p / K;
    const uint4* src = x + t * vec_per_row;
    uint4* dst = x_disp + pos * vec_per_row;
    for (int c = lane; c < vec_per_row; c += 32) dst[c] = src[c];
  }
}

// out[t] = sum_k alpha[t,k] * y[inv[t*K+k]], slots in ascending k, FP32.
// A CTA per token: its warps split the D columns, and in every warp lane k
// holds slot k's position and weight (so a token's rows are read by 256
// threads at once, and 8 tokens per SM are in flight instead of one warp's
// worth). Each output element sums its slots in slot order.
constexpr int kCombineWarps = 8;

template <typename T>
__global__ void __launch_bounds__(32 * kCombineWarps)
combine_kernel(const T* __restrict__ y, const float* __restrict__ alpha,
               const int32_t* __restrict__ inv, float* __restrict__ out, int ntok, int D, int K,
               int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  constexpr int V = Vec16<T>::kElems;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t N = (int64_t)ntok * K;
  for (int64_t t = blockIdx.x; t < ntok; t += gridDim.x) {
    int pos = -1;
    float wt = 0.f;
    if (lane < K) {
      const int q = inv[t * K + lane];
      if (q >= 0 && q < N) {
        pos = q;
        wt = alpha[t * K + lane];
      } else if (w == 0) {
        flag_error(err, LRM_DEVERR_INDEX);
      }
    }
    for (int c = (w * 32 + lane) * V; c < D; c += 32 * kCombineWarps * V) {
      float acc[V];
#pragma unroll
      for (int u = 0; u < V; ++u) acc[u] = 0.f;
      for (int k = 0; k < K; ++k) {
        const int r = __shfl_sync(0xffffffffu, pos, k);
        const float a = __shfl_sync(0xffffffffu, wt, k);
        if (r >= 0) {
          float f[V];
          Vec16<T>::unpack(ld_stream(y + (int64_t)r * D + c), f);
#pragma unroll
          for (int u = 0; u < V; ++u) acc[u] = fmaf(a, f[u], acc[u]);
        }
      }
      float4* o = reinterpret_cast<float4*>(out + t * D + c);
#pragma unroll
      for (int u = 0; u < V; u += 4) o[u / 4] = make_float4(acc[u], acc[u + 1], acc[u + 2], acc[u + 3]);
    }
  }
}

static int warp_grid(int64_t rows) {
  const int64_t cap = (int64_t)num_sms() * 64;  // 8 blocks of 8 warps per SM
  return (int)std::max<int64_t>(1, (std::min<int64_t>(rows, cap) + 7) / 8);
}

static lrm_status launch_gather(const lrm_shape* s, const int32_t* perm, const void* x,
                                void* x_disp, int32_t* err, cudaStream_t cs) {
  const int64_t N = (int64_t)s->T * s->K;
  if (N == 0) return LRM_OK;
  const int vec = s->D * elem_bytes(s->dtype) / 16;
  launch_k(gather_tokens_kernel, dim3(warp_grid(N)), dim3(256), 0, cs, perm, (const uint4*)x, (uint4*)x_disp, N,
                                                     s->K, s->T, vec, err);
  return launch_status();
}

static lrm_status launch_combine(const lrm_shape* s, const void* y, const float* alpha,
                                 const int32_t* inv, float* out, int32_t* err, cudaStream_t cs) {
  if (s->T == 0) return LRM_OK;
  const int blocks = (int)std::min<int64_t>(s->T, (int64_t)num_sms() * 64);
  if (s->dtype == LRM_BF16)
    launch_k(combine_kernel<__nv_bfloat16>, dim3(blocks), dim3(32 * kCombineWarps), 0, cs,
             (const __nv_bfloat16*)y, alpha, inv, out, s->T, s->D, s->K, err);
  else
    launch_k(combine_kernel<float>, dim3(blocks), dim3(32 * kCombineWarps), 0, cs,
             (const float*)y, alpha, inv, out, s->T, s->D, s->K, err);
  return launch_status();
}

static lrm_status run_fwd(const FwdArgs& a, unsigned parts) {
  return a.s->dtype == LRM_BF16 ? launch_fwd_tc(a, parts) : launch_fwd_f32(a, parts);
}

static lrm_status check_base(const lrm_shape* s, const void* ws, size_t ws_bytes) {
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  return check_ws(s, ws, ws_bytes);
}

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_gather_tokens(const lrm_shape* s, const int32_t* perm, const void* x,
                                        void* x_disp, void* ws, size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_gather_tokens");
  lrm_status st = check_base(s, ws, ws_bytes);
  if (st != LRM_OK) return st;
  if ((st = check_ptrs(s, {}, {perm, x, x_disp})) != LRM_OK) return st;
  return launch_gather(s, perm, x, x_disp, error_word(ws), (cudaStream_t)stream);
}

extern "C" lrm_status lrm_expert_fc1_fwd(const lrm_shape* s, const int32_t* off,
                                         const void* x_disp, const void* w_gate,
                                         const void* w_up, void* ab, void* phi, void* ws,
                                         size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_fc1_fwd");
  lrm_status st = check_base(s, ws, ws_bytes);
  if (st != LRM_OK) return st;
  if ((st = check_ptrs(s, {off, w_gate, w_up}, {x_disp, ab, phi})) != LRM_OK) return st;
  if ((int64_t)s->T * s->K == 0) return LRM_OK;
  FwdArgs a{s, off, w_gate, w_up, nullptr, x_disp, ab, phi, nullptr, error_word(ws),
            (cudaStream_t)stream};
  return run_fwd(a, kPartFc1Fwd);
}

extern "C" lrm_status lrm_expert_fc2_fwd(const lrm_shape* s, const int32_t* off,
                                         const void* phi, const void* w_down, void* y, void* ws,
                                         size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_fc2_fwd");
  lrm_status st = check_base(s, ws, ws_bytes);
  if (st != LRM_OK) return st;
  if ((st = check_ptrs(s, {off, w_down}, {phi, y})) != LRM_OK) return st;
  if ((int64_t)s->T * s->K == 0) return LRM_OK;
  FwdArgs a{s, off, nullptr, nullptr, w_down, nullptr, nullptr, const_cast<void*>(phi), y,
            error_word(ws), (cudaStream_t)stream};
  return run_fwd(a, kPartFc2Fwd);
}

extern "C" lrm_status lrm_combine(const lrm_shape* s, const void* y, const float* alpha,
                                  const int32_t* inv, float* out, void* ws, size_t ws_bytes,
                                  void* stream) {
  LRM_NVTX("lrm_combine");
  lrm_status st = check_base(s, ws, ws_bytes);
  if (st != LRM_OK) return st;
  if (s->K > 32) return LRM_ERR_UNSUPPORTED;
  if ((st = check_ptrs(s, {}, {y, alpha, inv, out})) != LRM_OK) return st;
  return launch_combine(s, y, alpha, inv, out, error_word(ws), (cudaStream_t)stream);
}

extern "C" lrm_status lrm_expert_fwd_grouped(const lrm_shape* s, const int32_t* perm,
                                             const int32_t* inv, const int32_t* off,
                                             const float* alpha, const void* x,
                                             const void* w_gate, const void* w_up,
                                             const void* w_down, void* x_disp, void* ab,
                                             void* phi, void* y, float* out, void* ws,
                                             size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_fwd_grouped");
  lrm_status st = check_base(s, ws, ws_bytes);
  if (st != LRM_OK) return st;
  if (s->K > 32) return LRM_ERR_UNSUPPORTED;
  if ((st = check_ptrs(s, {off, w_gate, w_up, w_down},
                       {perm, inv, alpha, x, x_disp, ab, phi, y, out})) != LRM_OK)
    return st;
  if (s->T == 0) return LRM_OK;
  cudaStream_t cs = (cudaStream_t)stream;
  if ((st = launch_gather(s, perm, x, x_disp, error_word(ws), cs)) != LRM_OK) return st;
  FwdArgs a{s, off, w_gate, w_up, w_down, x_disp, ab, phi, y, error_word(ws), cs};
  if ((st = run_fwd(a, kPartFwdAll)) != LRM_OK) return st;
  return launch_combine(s, y, alpha, inv, out, error_word(ws), cs);
}

extern "C" lrm_status lrm_expert_fc1_recompute(const lrm_shape* s, const int32_t* sel_off,
                                               const void* x_c, const void* w_gate,
                                               const void* w_up, void* ab_c, void* ws,
                                               size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_fc1_recompute");
  lrm_status st = check_base(s, ws, ws_bytes);
  if (st != LRM_OK) return st;
  if ((st = check_ptrs(s, {sel_off, w_gate, w_up}, {x_c, ab_c})) != LRM_OK) return st;
  if ((int64_t)s->T * s->K == 0) return LRM_OK;
  FwdArgs a{s, sel_off, w_gate, w_up, nullptr, x_c, ab_c, nullptr, nullptr, error_word(ws),
            (cudaStream_t)stream};
  return run_fwd(a, kPartFc1Fwd);
}
