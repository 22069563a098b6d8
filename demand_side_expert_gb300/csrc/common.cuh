// Shared host/device helpers of liblrm (validation, error word, vector I/O).
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>

#include "lrm.h"

namespace lrm {

constexpr size_t kWsHeaderBytes = 256;  // error word, tile-queue counters, reserved
constexpr int kWsHeaderWords = 8;        // words the header clear zeroes

inline int32_t* error_word(void* ws) { return static_cast<int32_t*>(ws); }
// The weight-gradient products' tile queue: next position, CTAs done, tiles
// handed out (words 4..6 of the header, after the error word).
inline int32_t* queue_words(int32_t* err) { return err ? err + 4 : nullptr; }

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int elem_bytes(int32_t dtype) { return dtype == LRM_BF16 ? 2 : 4; }

// Validates the shape fields shared by every call. Returns LRM_OK or a code.
inline lrm_status check_shape(const lrm_shape* s) {
  if (!s) return LRM_ERR_INVALID_ARG;
  if (s->T < 0 || s->D <= 0 || s->H <= 0 || s->E <= 0 || s->K <= 0)
    return LRM_ERR_INVALID_ARG;
  if (s->K > s->E) return LRM_ERR_INVALID_ARG;
  if (s->dtype != LRM_F32 && s->dtype != LRM_BF16) return LRM_ERR_INVALID_ARG;
  if ((int64_t)s->T * s->K >= (int64_t)1 << 31) return LRM_ERR_UNSUPPORTED;
  if (s->D % 8 != 0 || s->H % 8 != 0) return LRM_ERR_UNSUPPORTED;
  if (s->E > 1024) return LRM_ERR_UNSUPPORTED;
  return LRM_OK;
}

size_t workspace_bytes(const lrm_shape* s);

inline lrm_status check_ws(const lrm_shape* s, const void* ws, size_t ws_bytes) {
  if (!ws) return LRM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LRM_ERR_UNSUPPORTED;
  if (ws_bytes < workspace_bytes(s)) return LRM_ERR_WORKSPACE;
  return LRM_OK;
}

// Every listed pointer non-null (row buffers may be null only when there are
// no routed pairs) and 16-byte aligned.
inline lrm_status check_ptrs(const lrm_shape* s, std::initializer_list<const void*> always,
                             std::initializer_list<const void*> rows) {
  for (const void* p : always) {
    if (!p) return LRM_ERR_INVALID_ARG;
    if (!aligned16(p)) return LRM_ERR_UNSUPPORTED;
  }
  const bool has_rows = (int64_t)s->T * s->K > 0;
  for (const void* p : rows) {
    if (!p) {
      if (has_rows) return LRM_ERR_INVALID_ARG;
      continue;
    }
    if (!aligned16(p)) return LRM_ERR_UNSUPPORTED;
  }
  return LRM_OK;
}

// A named NVTX range around one C entry point, so timeline and profiler
// tools (ncu --nvtx, a trace viewer) show which call launched which kernels;
// with no tool attached it costs a check of a function pointer.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define LRM_NVTX(name) ::lrm::NvtxRange lrm_nvtx_range_(name)

inline lrm_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? LRM_OK : LRM_ERR_CUDA;
}

// Programmatic dependent launch. Every kernel of the path is launched with
// the attribute below and starts with pdl_begin(): it waits until the grid
// before it in the stream has completed and its writes are visible, then
// lets the next grid be scheduled. So the next kernel's CTAs can be resident
// (and run setup that touches no global memory) while this one drains, and
// no kernel touches global memory before its predecessor is complete. A
// kernel launched without the attribute, or after a non-kernel operation,
// waits for nothing extra.
#ifndef LRM_PDL
#define LRM_PDL 1
#endif

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = LRM_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

inline int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_begin() {
  pdl_wait();
  pdl_launch_dependents();
}

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 16-byte vector of activations: 8 bf16 or 4 floats, unpacked to floats.
template <typename T>
struct Vec16;

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
  }
};

template <>
struct Vec16<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                      __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

}  // namespace lrm
