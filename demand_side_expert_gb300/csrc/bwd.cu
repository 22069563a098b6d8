// lrm_expert_bwd_grouped: argument checks and the launch sequence of the
// expert backward (four grouped products, then the scatter back to tokens).
#include "common.cuh"
#include "internal.h"

using namespace lrm;

extern "C" lrm_status lrm_expert_bwd_grouped(
    const lrm_shape* s, const int32_t* sel_off, const void* w_gate, const void* w_up,
    const void* w_down, const void* dy_c, const void* x_c, const void* ab_c, const void* phi_c,
    const int32_t* inv, const int32_t* row_of_pos, void* dab_c, float* dx_c, float* dw_gate,
    float* dw_up, float* dw_down, float* dx, void* ws, size_t ws_bytes, void* stream) {
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes)) != LRM_OK) return st;
  if (s->K > 32) return LRM_ERR_UNSUPPORTED;
  const void* ptrs[] = {sel_off, w_gate, w_up, w_down, dw_gate, dw_up, dw_down};
  for (const void* p : ptrs)
    if (!p) return LRM_ERR_INVALID_ARG;
  const int64_t N = (int64_t)s->T * s->K;
  if (N > 0) {
    const void* rows[] = {dy_c, x_c, ab_c, phi_c, inv, row_of_pos, dab_c, dx_c, dx};
    for (const void* p : rows)
      if (!p) return LRM_ERR_INVALID_ARG;
  }
  const void* vec[] = {w_gate, w_up, w_down, dy_c, x_c, ab_c, phi_c, dab_c, dx_c,
                       dw_gate, dw_up, dw_down, dx};
  for (const void* p : vec)
    if (p && !aligned16(p)) return LRM_ERR_UNSUPPORTED;
  BwdArgs a{s, sel_off, w_gate, w_up, w_down, dy_c, x_c, ab_c, phi_c, dab_c,
            dx_c, dw_gate, dw_up, dw_down, error_word(ws), (cudaStream_t)stream};
  st = s->dtype == LRM_BF16 ? launch_bwd_tc(a) : launch_bwd_f32(a);
  if (st != LRM_OK) return st;
  return launch_dx_gather(s, dx_c, inv, row_of_pos, dx, error_word(ws), (cudaStream_t)stream);
}
