// Expert-backward entry points: the one-call lrm_expert_bwd_grouped and its
// five sub-steps (the four grouped products of LRMoE Sec. 3.4 and the
// scatter of input gradients back to tokens), with their argument checks.
#include "common.cuh"
#include "internal.h"

using namespace lrm;

namespace {

lrm_status check_common(const lrm_shape* s, const void* ws, size_t ws_bytes,
                        const int32_t* sel_off) {
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes)) != LRM_OK) return st;
  if (!sel_off) return LRM_ERR_INVALID_ARG;
  return LRM_OK;
}

lrm_status run_parts(const BwdArgs& a, unsigned parts) {
  return a.s->dtype == LRM_BF16 ? launch_bwd_tc(a, parts) : launch_bwd_f32(a, parts);
}

}  // namespace

extern "C" lrm_status lrm_expert_fc2_dgrad(const lrm_shape* s, const int32_t* sel_off,
                                           const void* w_down, const void* dy_c,
                                           const void* ab_c, void* dab_c, void* ws,
                                           size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_fc2_dgrad");
  lrm_status st = check_common(s, ws, ws_bytes, sel_off);
  if (st != LRM_OK) return st;
  if ((st = check_ptrs(s, {w_down}, {dy_c, ab_c, dab_c})) != LRM_OK) return st;
  BwdArgs a{s, sel_off, nullptr, nullptr, w_down, dy_c, nullptr, ab_c, nullptr, dab_c,
            nullptr, nullptr, nullptr, nullptr, error_word(ws), (cudaStream_t)stream};
  return run_parts(a, kPartFc2Dgrad);
}

extern "C" lrm_status lrm_expert_fc2_wgrad(const lrm_shape* s, const int32_t* sel_off,
                                           const void* phi_c, const void* dy_c, float* dw_down,
                                           void* ws, size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_fc2_wgrad");
  lrm_status st = check_common(s, ws, ws_bytes, sel_off);
  if (st != LRM_OK) return st;
  if ((st = check_ptrs(s, {dw_down}, {phi_c, dy_c})) != LRM_OK) return st;
  BwdArgs a{s, sel_off, nullptr, nullptr, nullptr, dy_c, nullptr, nullptr, phi_c, nullptr,
            nullptr, nullptr, nullptr, dw_down, error_word(ws), (cudaStream_t)stream};
  return run_parts(a, kPartFc2Wgrad);
}

extern "C" lrm_status lrm_expert_fc1_wgrad(const lrm_shape* s, const int32_t* sel_off,
                                           const void* x_c, const void* dab_c, float* dw_gate,
                                           float* dw_up, void* ws, size_t ws_bytes,
                                           void* stream) {
  LRM_NVTX("lrm_expert_fc1_wgrad");
  lrm_status st = check_common(s, ws, ws_bytes, sel_off);
  if (st != LRM_OK) return st;
  if ((st = check_ptrs(s, {dw_gate, dw_up}, {x_c, dab_c})) != LRM_OK) return st;
  BwdArgs a{s, sel_off, nullptr, nullptr, nullptr, nullptr, x_c, nullptr, nullptr,
            const_cast<void*>(dab_c), nullptr, dw_gate, dw_up, nullptr, error_word(ws),
            (cudaStream_t)stream};
  return run_parts(a, kPartFc1Wgrad);
}

extern "C" lrm_status lrm_expert_fc1_dgrad(const lrm_shape* s, const int32_t* sel_off,
                                           const void* w_gate, const void* w_up,
                                           const void* dab_c, float* dx_c, void* ws,
                                           size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_fc1_dgrad");
  lrm_status st = check_common(s, ws, ws_bytes, sel_off);
  if (st != LRM_OK) return st;
  if ((st = check_ptrs(s, {w_gate, w_up}, {dab_c, dx_c})) != LRM_OK) return st;
  BwdArgs a{s, sel_off, w_gate, w_up, nullptr, nullptr, nullptr, nullptr, nullptr,
            const_cast<void*>(dab_c), dx_c, nullptr, nullptr, nullptr, error_word(ws),
            (cudaStream_t)stream};
  return run_parts(a, kPartFc1Dgrad);
}

extern "C" lrm_status lrm_scatter_dx(const lrm_shape* s, const float* dx_c, const int32_t* inv,
                                     const int32_t* row_of_pos, float* dx, void* ws,
                                     size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_scatter_dx");
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes)) != LRM_OK) return st;
  if (s->K > 32) return LRM_ERR_UNSUPPORTED;
  if ((st = check_ptrs(s, {}, {dx_c, inv, row_of_pos, dx})) != LRM_OK) return st;
  return launch_dx_gather(s, dx_c, inv, row_of_pos, dx, error_word(ws), (cudaStream_t)stream);
}

extern "C" lrm_status lrm_expert_bwd_grouped(
    const lrm_shape* s, const int32_t* sel_off, const void* w_gate, const void* w_up,
    const void* w_down, const void* dy_c, const void* x_c, const void* ab_c, const void* phi_c,
    const int32_t* inv, const int32_t* row_of_pos, void* dab_c, float* dx_c, float* dw_gate,
    float* dw_up, float* dw_down, float* dx, void* ws, size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_bwd_grouped");
  lrm_status st = check_common(s, ws, ws_bytes, sel_off);
  if (st != LRM_OK) return st;
  if (s->K > 32) return LRM_ERR_UNSUPPORTED;
  if ((st = check_ptrs(s, {w_gate, w_up, w_down, dw_gate, dw_up, dw_down},
                       {dy_c, x_c, ab_c, phi_c, inv, row_of_pos, dab_c, dx_c, dx})) != LRM_OK)
    return st;
  BwdArgs a{s, sel_off, w_gate, w_up, w_down, dy_c, x_c, ab_c, phi_c, dab_c,
            dx_c, dw_gate, dw_up, dw_down, error_word(ws), (cudaStream_t)stream};
  if ((st = run_parts(a, kPartAll)) != LRM_OK) return st;
  return launch_dx_gather(s, dx_c, inv, row_of_pos, dx, error_word(ws), (cudaStream_t)stream);
}

extern "C" lrm_status lrm_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_selftest_wait_timeout");
  return selftest_wait_timeout(ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" lrm_status lrm_expert_bwd_gathered(
    const lrm_shape* s, int32_t parts, const int32_t* sel_off, const int32_t* sel_pos,
    const int32_t* tok_c, const void* w_gate, const void* w_up, const void* w_down,
    const void* dy_c, const void* x, const void* ab, const void* phi, const int32_t* inv,
    const int32_t* row_of_pos, void* dab_c, float* dx_c, float* dw_gate, float* dw_up,
    float* dw_down, float* dx, void* ws, size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_expert_bwd_gathered");
  lrm_status st = check_common(s, ws, ws_bytes, sel_off);
  if (st != LRM_OK) return st;
  if (parts < 0 || parts > LRM_BWD_ALL) return LRM_ERR_INVALID_ARG;
  if (s->K > 32) return LRM_ERR_UNSUPPORTED;
  if ((st = check_ptrs(s, {w_gate, w_up, w_down, dw_gate, dw_up, dw_down},
                       {sel_pos, tok_c, dy_c, x, ab, phi, inv, row_of_pos, dab_c, dx_c, dx})) !=
      LRM_OK)
    return st;
  BwdArgs a{s, sel_off, w_gate, w_up, w_down, dy_c, x, ab, phi, dab_c,
            dx_c, dw_gate, dw_up, dw_down, error_word(ws), (cudaStream_t)stream};
  a.sel_pos = sel_pos;
  a.tok_c = tok_c;
  const unsigned gemm_parts = (unsigned)parts & kPartAll;
  if (gemm_parts && (st = run_parts(a, gemm_parts)) != LRM_OK) return st;
  if (parts & LRM_BWD_SCATTER_DX)
    return launch_dx_gather(s, dx_c, inv, row_of_pos, dx, error_word(ws), (cudaStream_t)stream);
  return LRM_OK;
}
