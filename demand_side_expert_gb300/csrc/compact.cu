// Physical compaction of the retained rows and the scatter of input
// gradients back to tokens.
//
// LRMoE Sec. 3.1 (compact runtime) and Sec. 3.4 / Fig. 4: retained gradient
// rows and their matching saved state are packed into contiguous expert
// segments (counts and offsets come from the selection), so the expert
// products run over the retained rows only, with no zero-masked rows. The
// gradient row is delta_u = alpha_u * g_t (LRMoE Sec. 7.1 Eq. 5), formed here
// once and rounded to the layer dtype.
//
// One warp per retained row, 16-byte vector copies; the retained row count
// M = sel_off[E] is read on the device, so the grid is sized from the upper
// bound and walks rows with a grid stride.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace lrm {

template <typename T>
__global__ void __launch_bounds__(256)
compact_kernel(const int32_t* __restrict__ perm, const uint8_t* __restrict__ keep,
               const int32_t* __restrict__ sel_off, const int32_t* __restrict__ sel_pos,
               const float* __restrict__ alpha, const T* __restrict__ x,
               const T* __restrict__ g, const T* __restrict__ ab, const T* __restrict__ phi,
               T* __restrict__ dy_c, T* __restrict__ x_c, T* __restrict__ ab_c,
               T* __restrict__ phi_c, int32_t* __restrict__ tok_c,
               int32_t* __restrict__ row_of_pos, int ntok, int D, int H, int K, int E,
               int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  constexpr int V = Vec16<T>::kElems;
  const int64_t N = (int64_t)ntok * K;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = gtid; i < N; i += nthr)
    if (!keep[i]) row_of_pos[i] = -1;

  const int lane = threadIdx.x & 31;
  // M = sel_off[E] comes from the caller's buffer: a value outside [0, N]
  // (sel_off not written by the selection) is clamped and flagged, so no
  // row past the N-row buffers is ever addressed
  int64_t M = sel_off[E];
  if (M < 0 || M > N) {
    if (gtid == 0) flag_error(err, LRM_DEVERR_INDEX);
    M = M < 0 ? 0 : N;
  }
  const int dv = D / V, abv = 2 * H / V, hv = H / V;
  {  // 64 zero rows of dy_c after the retained ones: the padding the FC2
     // weight-gradient product reads as B past the last group
    const int64_t zrows = M < N ? min((int64_t)64, N - M) : 0;
    uint4* z = reinterpret_cast<uint4*>(dy_c + M * D);
    for (int64_t i = gtid; i < zrows * dv; i += nthr) z[i] = make_uint4(0, 0, 0, 0);
  }
  for (int64_t j = gtid >> 5; j < M; j += nthr >> 5) {
    const int i = sel_pos[j];
    const int p = (i >= 0 && i < N) ? perm[i] : -1;
    if (p < 0 || p >= N) {
      if (lane == 0) flag_error(err, LRM_DEVERR_INDEX);
      continue;
    }
    const int64_t t = p / K;
    const float a = alpha[p];
    const uint4* gs = reinterpret_cast<const uint4*>(g + t * D);
    const uint4* xs = reinterpret_cast<const uint4*>(x + t * D);
    uint4* dyd = reinterpret_cast<uint4*>(dy_c + j * D);
    uint4* xd = reinterpret_cast<uint4*>(x_c + j * D);
    // up to 8 of the lane's 16-byte chunks loaded before any is written
    for (int c0 = lane; c0 < dv; c0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + 32 * u < dv) v[u] = gs[c0 + 32 * u];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + 32 * u < dv) {
          float f[V];
          Vec16<T>::unpack(v[u], f);
#pragma unroll
          for (int e = 0; e < V; ++e) f[e] *= a;
          dyd[c0 + 32 * u] = Vec16<T>::pack(f);
        }
      }
    }
    if (x_c)
      for (int c = lane; c < dv; c += 32) xd[c] = xs[c];
    // the saved-state copies are skipped when their destination is absent:
    // [a | b] recomputed, or rows gathered by the products themselves
    if (ab_c) {
      const uint4* abs_ = reinterpret_cast<const uint4*>(ab + (int64_t)i * 2 * H);
      uint4* abd = reinterpret_cast<uint4*>(ab_c + j * 2 * H);
      for (int c = lane; c < abv; c += 32) abd[c] = ld_stream(abs_ + c);
    }
    if (phi_c) {
      const uint4* ps = reinterpret_cast<const uint4*>(phi + (int64_t)i * H);
      uint4* pd = reinterpret_cast<uint4*>(phi_c + j * H);
      for (int c = lane; c < hv; c += 32) pd[c] = ld_stream(ps + c);
    }
    if (lane == 0) {
      tok_c[j] = (int32_t)t;
      row_of_pos[i] = (int32_t)j;
    }
  }
}

// dx[t] = sum over the token's kept slots k (ascending) of dx_c[row].
// One CTA per token, its warps splitting the D columns: each lane keeps the
// K loads of a column group in flight, and every output element is summed in
// slot order (the same order for every split, so the result is exact and
// deterministic).
constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(32 * kGatherWarps)
dx_gather_kernel(const float* __restrict__ dx_c, const int32_t* __restrict__ inv,
                 const int32_t* __restrict__ row_of_pos, float* __restrict__ dx, int ntok,
                 int D, int K, int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t N = (int64_t)ntok * K;
  for (int64_t t = blockIdx.x; t < ntok; t += gridDim.x) {
    int row = -1;
    if (lane < K) {
      const int pos = inv[t * K + lane];
      if (pos >= 0 && pos < N) {
        row = row_of_pos[pos];
        if (row >= N) {
          if (w == 0) flag_error(err, LRM_DEVERR_INDEX);
          row = -1;
        }
      } else if (w == 0) {
        flag_error(err, LRM_DEVERR_INDEX);
      }
    }
    for (int c = (w * 32 + lane) * 4; c < D; c += 32 * kGatherWarps * 4) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < K; ++k) {
        const int r = __shfl_sync(0xffffffffu, row, k);
        if (r >= 0) {
          const float4 v = __ldcs(reinterpret_cast<const float4*>(dx_c + (int64_t)r * D + c));
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
      }
      *reinterpret_cast<float4*>(dx + t * D + c) = acc;
    }
  }
}

lrm_status launch_dx_gather(const lrm_shape* s, const float* dx_c, const int32_t* inv,
                            const int32_t* row_of_pos, float* dx, int32_t* err,
                            cudaStream_t cs) {
  if (s->T == 0) return LRM_OK;
  const int blocks = (int)std::min<int64_t>(s->T, (int64_t)num_sms() * 64);
  launch_k(dx_gather_kernel, dim3(blocks), dim3(32 * kGatherWarps), 0, cs, dx_c, inv, row_of_pos,
           dx, s->T, s->D, s->K, err);
  return launch_status();
}

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_compact(const lrm_shape* s, const int32_t* perm,
                                  const uint8_t* keep, const int32_t* sel_off,
                                  const int32_t* sel_pos, const float* alpha, const void* x,
                                  const void* g, const void* ab, const void* phi, void* dy_c,
                                  void* x_c, void* ab_c, void* phi_c, int32_t* tok_c,
                                  int32_t* row_of_pos, void* ws, size_t ws_bytes,
                                  void* stream) {
  LRM_NVTX("lrm_compact");
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes)) != LRM_OK) return st;
  const int64_t N = (int64_t)s->T * s->K;
  if (N == 0) return LRM_OK;
  const void* ptrs[] = {perm, keep, sel_off, sel_pos, alpha, g, dy_c, tok_c, row_of_pos};
  for (const void* p : ptrs)
    if (!p) return LRM_ERR_INVALID_ARG;
  // a copied row needs its source; absent destinations are skipped
  if ((x_c && !x) || (ab_c && !ab) || (phi_c && !phi)) return LRM_ERR_INVALID_ARG;
  const void* vec[] = {x, g, ab, phi, dy_c, x_c, ab_c, phi_c};
  for (const void* p : vec)
    if (!aligned16(p)) return LRM_ERR_UNSUPPORTED;
  const int blocks = num_sms() * 8;
  cudaStream_t cs = (cudaStream_t)stream;
  if (s->dtype == LRM_BF16) {
    using T = __nv_bfloat16;
    launch_k(compact_kernel<T>, dim3(blocks), dim3(256), 0, cs, 
        perm, keep, sel_off, sel_pos, alpha, (const T*)x, (const T*)g, (const T*)ab,
        (const T*)phi, (T*)dy_c, (T*)x_c, (T*)ab_c, (T*)phi_c, tok_c, row_of_pos, s->T, s->D,
        s->H, s->K, s->E, error_word(ws));
  } else {
    using T = float;
    launch_k(compact_kernel<T>, dim3(blocks), dim3(256), 0, cs, 
        perm, keep, sel_off, sel_pos, alpha, (const T*)x, (const T*)g, (const T*)ab,
        (const T*)phi, (T*)dy_c, (T*)x_c, (T*)ab_c, (T*)phi_c, tok_c, row_of_pos, s->T, s->D,
        s->H, s->K, s->E, error_word(ws));
  }
  return launch_status();
}
