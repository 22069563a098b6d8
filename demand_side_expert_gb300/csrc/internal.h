// Internal launchers shared between translation units of liblrm.
#pragma once

#include <cuda_runtime.h>

#include "lrm.h"

namespace lrm {

struct BwdArgs {
  const lrm_shape* s;
  const int32_t* sel_off;
  const void *w_gate, *w_up, *w_down;
  const void *dy_c, *x_c, *ab_c, *phi_c;
  void* dab_c;
  float *dx_c, *dw_gate, *dw_up, *dw_down;
  int32_t* err;
  cudaStream_t stream;
  // Gathered operands: when set, ab_c / phi_c hold the uncompacted saved
  // state [N rows, dispatch order] read at row sel_pos[j], and x_c the token
  // rows [T rows] read at row tok_c[j], for compacted row j.
  const int32_t* sel_pos = nullptr;
  const int32_t* tok_c = nullptr;
};

// Sub-steps of the expert backward, in dependency order.
enum : unsigned {
  kPartFc2Dgrad = 1,  // dphi = dy_c W_down^T + SwiGLU gradient -> dab_c
  kPartFc2Wgrad = 2,  // dW_down = phi_c^T dy_c
  kPartFc1Wgrad = 4,  // [dW_gate | dW_up] = x_c^T dab_c
  kPartFc1Dgrad = 8,  // dx_c = dab_c [W_gate | W_up]^T
  kPartAll = 15
};

struct FwdArgs {
  const lrm_shape* s;
  const int32_t* off;  // dispatch group offsets [E+1]
  const void *w_gate, *w_up, *w_down;
  const void* x_disp;
  void *ab, *phi, *y;
  int32_t* err;
  cudaStream_t stream;
};

// Sub-steps of the forward expert pass.
enum : unsigned {
  kPartFc1Fwd = 1,  // [a | b] = x_disp [W_gate | W_up], phi = SiLU(a) * b
  kPartFc2Fwd = 2,  // y = phi W_down
  kPartFwdAll = 3
};

// BF16 path: persistent tcgen05 grouped GEMMs (tensor cores).
lrm_status launch_bwd_tc(const BwdArgs& a, unsigned parts);
// F32 path: the same products on CUDA cores.
lrm_status launch_bwd_f32(const BwdArgs& a, unsigned parts);
// Forward expert products, BF16 (tensor cores) and F32 (CUDA cores).
lrm_status launch_fwd_tc(const FwdArgs& a, unsigned parts);
lrm_status launch_fwd_f32(const FwdArgs& a, unsigned parts);
// Bounded-wait self-test of the grouped GEMM pipeline (see lrm.h).
lrm_status selftest_wait_timeout(void* ws, size_t ws_bytes, cudaStream_t cs);
// Dispatch permutation in one launch of one thread-block cluster, for up to
// dispatch_fused_max_pairs() pairs; no workspace (dispatch.cu).
lrm_status launch_dispatch_fused(const int32_t* topk_idx, int64_t N, int E, int32_t* perm,
                                 int32_t* inv, int32_t* counts, int32_t* off, int32_t* err,
                                 cudaStream_t cs);
int64_t dispatch_fused_max_pairs();
// dx[t] = sum over kept slots of dx_c rows (deterministic, no atomics).
lrm_status launch_dx_gather(const lrm_shape* s, const float* dx_c, const int32_t* inv,
                            const int32_t* row_of_pos, float* dx, int32_t* err,
                            cudaStream_t cs);

}  // namespace lrm
