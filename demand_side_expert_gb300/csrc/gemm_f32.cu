// FP32 variant of the four expert-backward products and of the two forward
// expert products on CUDA cores.
//
// Same arithmetic as the tensor-core path (LRMoE Alg. 1 PackedExpertBackward
// over each expert's retained rows, m_e read from sel_off on the device; the
// forward over each expert's routed rows, groups from the dispatch offsets),
// one thread per output element with a sequential FP32 dot product. It
// serves FP32 layers, whose sizes are small; the BF16 path is the fast one.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace lrm {

constexpr int kF32Threads = 256;

__device__ __forceinline__ int expert_of_row(const int32_t* sel_off, int E, int j) {
  int lo = 0, hi = E;  // largest e with sel_off[e] <= j
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sel_off[mid] <= j) lo = mid; else hi = mid;
  }
  return lo;
}

// G1 + SwiGLU gradient: dab_c[j] = [da | db]
// ab_rows (optional): the row of ab_c (then the uncompacted saved state)
// read for compacted row j.
__global__ void f32_g1_kernel(const int32_t* __restrict__ sel_off, int E, int D, int H,
                              const float* __restrict__ dy_c, const float* __restrict__ w_down,
                              const float* __restrict__ ab_c, const int32_t* __restrict__ ab_rows,
                              float* __restrict__ dab_c) {
  const int64_t M = sel_off[E];
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < M * H;
       o += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(o / H), h = (int)(o % H);
    const int e = expert_of_row(sel_off, E, j);
    const float* wd = w_down + ((int64_t)e * H + h) * D;
    const float* dy = dy_c + (int64_t)j * D;
    float dphi = 0.f;
    for (int d = 0; d < D; ++d) dphi = fmaf(dy[d], wd[d], dphi);
    const int64_t r = ab_rows ? ab_rows[j] : j;
    const float a = ab_c[r * 2 * H + h];
    const float b = ab_c[r * 2 * H + H + h];
    const float s = 1.0f / (1.0f + expf(-a));
    dab_c[(int64_t)j * 2 * H + h] = dphi * b * s * (1.0f + a * (1.0f - s));
    dab_c[(int64_t)j * 2 * H + H + h] = dphi * a * s;
  }
}

// G4: dx_c[j, d] = sum_h da[j,h] W_gate[e][d,h] + db[j,h] W_up[e][d,h]
__global__ void f32_g4_kernel(const int32_t* __restrict__ sel_off, int E, int D, int H,
                              const float* __restrict__ dab_c, const float* __restrict__ w_gate,
                              const float* __restrict__ w_up, float* __restrict__ dx_c) {
  const int64_t M = sel_off[E];
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < M * D;
       o += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(o / D), d = (int)(o % D);
    const int e = expert_of_row(sel_off, E, j);
    const float* wg = w_gate + ((int64_t)e * D + d) * H;
    const float* wu = w_up + ((int64_t)e * D + d) * H;
    const float* da = dab_c + (int64_t)j * 2 * H;
    float acc = 0.f;
    for (int h = 0; h < H; ++h) acc = fmaf(da[h], wg[h], acc);
    for (int h = 0; h < H; ++h) acc = fmaf(da[H + h], wu[h], acc);
    dx_c[(int64_t)j * D + d] = acc;
  }
}

// G2: dW_down[e][h, d] = sum_{j in e} phi_c[j,h] dy_c[j,d]
__global__ void f32_g2_kernel(const int32_t* __restrict__ sel_off, int E, int D, int H,
                              const float* __restrict__ phi_c, const int32_t* __restrict__ rows,
                              const float* __restrict__ dy_c, float* __restrict__ dw_down) {
  const int64_t total = (int64_t)E * H * D;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < total;
       o += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(o / ((int64_t)H * D));
    const int h = (int)((o / D) % H), d = (int)(o % D);
    float acc = 0.f;
    for (int j = sel_off[e]; j < sel_off[e + 1]; ++j)
      acc = fmaf(phi_c[(rows ? (int64_t)rows[j] : j) * H + h], dy_c[(int64_t)j * D + d], acc);
    dw_down[o] = acc;
  }
}

// G3: dW_gate[e][d, n] / dW_up[e][d, n - H] = sum_{j in e} x_c[j,d] dab_c[j,n]
__global__ void f32_g3_kernel(const int32_t* __restrict__ sel_off, int E, int D, int H,
                              const float* __restrict__ x_c, const int32_t* __restrict__ rows,
                              const float* __restrict__ dab_c, float* __restrict__ dw_gate,
                              float* __restrict__ dw_up) {
  const int64_t total = (int64_t)E * D * 2 * H;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < total;
       o += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(o / ((int64_t)D * 2 * H));
    const int d = (int)((o / (2 * H)) % D), n = (int)(o % (2 * H));
    float acc = 0.f;
    for (int j = sel_off[e]; j < sel_off[e + 1]; ++j)
      acc = fmaf(x_c[(rows ? (int64_t)rows[j] : j) * D + d], dab_c[(int64_t)j * 2 * H + n], acc);
    float* out = n < H ? dw_gate : dw_up;
    out[((int64_t)e * D + d) * H + (n < H ? n : n - H)] = acc;
  }
}

// F1: ab[j] = [x_j W_gate[e] | x_j W_up[e]], phi[j] = SiLU(a) * b
__global__ void f32_f1_kernel(const int32_t* __restrict__ off, int64_t n_rows, int E, int D,
                              int H,
                              const float* __restrict__ x_disp, const float* __restrict__ w_gate,
                              const float* __restrict__ w_up, float* __restrict__ ab,
                              float* __restrict__ phi) {
  const int64_t N = min((int64_t)off[E], n_rows);
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < N * H;
       o += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(o / H), h = (int)(o % H);
    const int e = expert_of_row(off, E, j);
    const float* xr = x_disp + (int64_t)j * D;
    const float* wg = w_gate + (int64_t)e * D * H + h;
    const float* wu = w_up + (int64_t)e * D * H + h;
    float a = 0.f, b = 0.f;
    for (int d = 0; d < D; ++d) {
      a = fmaf(xr[d], wg[(int64_t)d * H], a);
      b = fmaf(xr[d], wu[(int64_t)d * H], b);
    }
    ab[(int64_t)j * 2 * H + h] = a;
    ab[(int64_t)j * 2 * H + H + h] = b;
    if (phi) phi[(int64_t)j * H + h] = a / (1.0f + expf(-a)) * b;
  }
}

// F2: y[j, d] = sum_h phi[j,h] W_down[e][h,d]
__global__ void f32_f2_kernel(const int32_t* __restrict__ off, int64_t n_rows, int E, int D,
                              int H,
                              const float* __restrict__ phi, const float* __restrict__ w_down,
                              float* __restrict__ y) {
  const int64_t N = min((int64_t)off[E], n_rows);
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < N * D;
       o += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(o / D), d = (int)(o % D);
    const int e = expert_of_row(off, E, j);
    const float* pr = phi + (int64_t)j * H;
    const float* wd = w_down + (int64_t)e * H * D + d;
    float acc = 0.f;
    for (int h = 0; h < H; ++h) acc = fmaf(pr[h], wd[(int64_t)h * D], acc);
    y[o] = acc;
  }
}

static int f32_grid(int64_t work) {
  return (int)std::max<int64_t>(1, std::min<int64_t>((work + kF32Threads - 1) / kF32Threads,
                                                     (int64_t)num_sms() * 8));
}

lrm_status launch_fwd_f32(const FwdArgs& a, unsigned parts) {
  const lrm_shape* s = a.s;
  const int D = s->D, H = s->H, E = s->E;
  const int64_t N = (int64_t)s->T * s->K;
  if (parts & kPartFc1Fwd)
    f32_f1_kernel<<<f32_grid(N * H), kF32Threads, 0, a.stream>>>(
        a.off, N, E, D, H, (const float*)a.x_disp, (const float*)a.w_gate, (const float*)a.w_up,
        (float*)a.ab, (float*)a.phi);
  if (parts & kPartFc2Fwd)
    f32_f2_kernel<<<f32_grid(N * D), kF32Threads, 0, a.stream>>>(
        a.off, N, E, D, H, (const float*)a.phi, (const float*)a.w_down, (float*)a.y);
  return launch_status();
}

lrm_status launch_bwd_f32(const BwdArgs& a, unsigned parts) {
  const lrm_shape* s = a.s;
  const int D = s->D, H = s->H, E = s->E;
  const int64_t N = (int64_t)s->T * s->K;
  const int sms = num_sms();
  auto grid = [&](int64_t work) {
    return (int)std::max<int64_t>(1, std::min<int64_t>((work + kF32Threads - 1) / kF32Threads,
                                                       (int64_t)sms * 8));
  };
  cudaStream_t cs = a.stream;
  const float* dy = (const float*)a.dy_c;
  if (parts & kPartFc2Dgrad)
    f32_g1_kernel<<<grid(N * H), kF32Threads, 0, cs>>>(a.sel_off, E, D, H, dy,
                                                       (const float*)a.w_down,
                                                       (const float*)a.ab_c, a.sel_pos,
                                                       (float*)a.dab_c);
  if (parts & kPartFc2Wgrad)
    f32_g2_kernel<<<grid((int64_t)E * H * D), kF32Threads, 0, cs>>>(
        a.sel_off, E, D, H, (const float*)a.phi_c, a.sel_pos, dy, a.dw_down);
  if (parts & kPartFc1Wgrad)
    f32_g3_kernel<<<grid((int64_t)E * D * 2 * H), kF32Threads, 0, cs>>>(
        a.sel_off, E, D, H, (const float*)a.x_c, a.tok_c, (const float*)a.dab_c, a.dw_gate,
        a.dw_up);
  if (parts & kPartFc1Dgrad)
    f32_g4_kernel<<<grid(N * D), kF32Threads, 0, cs>>>(a.sel_off, E, D, H,
                                                       (const float*)a.dab_c,
                                                       (const float*)a.w_gate,
                                                       (const float*)a.w_up, a.dx_c);
  return launch_status();
}

}  // namespace lrm
