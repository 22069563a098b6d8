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
};

// BF16 path: four persistent tcgen05 grouped GEMMs (tensor cores).
lrm_status launch_bwd_tc(const BwdArgs& a);
// F32 path: the same four products on CUDA cores.
lrm_status launch_bwd_f32(const BwdArgs& a);
// dx[t] = sum over kept slots of dx_c rows (deterministic, no atomics).
lrm_status launch_dx_gather(const lrm_shape* s, const float* dx_c, const int32_t* inv,
                            const int32_t* row_of_pos, float* dx, int32_t* err,
                            cudaStream_t cs);

}  // namespace lrm
