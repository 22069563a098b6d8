// lrm_dispatch_permute_noalloc: the dispatch permutation for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: a plugin that is handed
// only its input and output tensors, or a host application whose memory
// manager owns the whole device budget, where a cudaMalloc would bypass its
// accounting and can stall every stream on the device while it runs. This
// variant needs nothing from the caller beyond inputs and outputs: the
// per-chunk count and base tables that lrm_dispatch_permute keeps in the
// caller's workspace live in one file-scope device array of fixed size
// instead, which every GPU that loads the library holds until the process
// exits.
//
// The kernels are the ones lrm_dispatch_permute launches: up to the
// single-launch limit the one-cluster kernel, which needs no scratch at all;
// above it the three launches, whose tables live in the array below.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace lrm {

// kernels of lrm_dispatch_permute (dispatch.cu)
__global__ void dispatch_hist_kernel(const int32_t* idx, int64_t N, int E, int nblk,
                                     int32_t* chunk_hist, int32_t* err);
__global__ void dispatch_scan_kernel(const int32_t* chunk_hist, int E, int nblk,
                                     int32_t* chunk_rel, int32_t* counts);
__global__ void dispatch_scatter_kernel(const int32_t* idx, int64_t N, int E, int nblk,
                                        const int32_t* chunk_rel, const int32_t* counts,
                                        int32_t* off, int32_t* perm, int32_t* inv);

namespace {

constexpr int kChunkPairs = 2048;   // pairs per CTA, as in dispatch.cu
constexpr int kDispThreads = 256;
constexpr int kDispWarps = kDispThreads / 32;

// Count table [E][chunks] followed by the table of each chunk's first position
// inside its expert's segment [E][chunks].
static __device__ __align__(256) int32_t g_dispatch_scratch[2 * LRM_NOALLOC_MAX_CHUNK_ENTRIES];

// Device address of g_dispatch_scratch, resolved once per device.
std::mutex g_mu;
void* g_scratch_addr[256] = {};

lrm_status scratch_for_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return LRM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return LRM_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<int32_t*>(g_scratch_addr[dev]);
  return LRM_OK;
}

}  // namespace
}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_dispatch_permute_noalloc(const lrm_shape* s, const int32_t* topk_idx,
                                                   int32_t* perm, int32_t* inv,
                                                   int32_t* counts, int32_t* off,
                                                   int32_t* dev_err, void* stream) {
  LRM_NVTX("lrm_dispatch_permute_noalloc");
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  const int64_t N = (int64_t)s->T * s->K;
  if ((N > 0 && (!topk_idx || !perm || !inv)) || !counts || !off) return LRM_ERR_INVALID_ARG;
  const int E = s->E;
  const int64_t nblk = N > 0 ? (N + kChunkPairs - 1) / kChunkPairs : 1;
  if ((int64_t)E * nblk > LRM_NOALLOC_MAX_CHUNK_ENTRIES) return LRM_ERR_WORKSPACE;
  if (N <= dispatch_fused_max_pairs())  // one launch, no tables
    return launch_dispatch_fused(topk_idx, N, E, perm, inv, counts, off, dev_err,
                                 (cudaStream_t)stream);
  int32_t* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != LRM_OK) return st;
  // Both tables are written in full before they are read, so the previous
  // call's contents need no clearing.
  int32_t* chunk_hist = scratch;
  int32_t* chunk_rel = scratch + (int64_t)E * nblk;
  cudaStream_t cs = (cudaStream_t)stream;
  const size_t sh1 = (size_t)kDispWarps * E * 4;
  const size_t sh3 = 2 * sh1 + (size_t)E * 4;
  if (sh3 > 48 * 1024) {
    if (cudaFuncSetAttribute(dispatch_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sh1) != cudaSuccess ||
        cudaFuncSetAttribute(dispatch_scatter_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sh3) != cudaSuccess) {
      (void)cudaGetLastError();  // leave no error behind for a later call to report
      return LRM_ERR_CUDA;
    }
  }
  dispatch_hist_kernel<<<(int)nblk, kDispThreads, sh1, cs>>>(topk_idx, N, E, (int)nblk,
                                                             chunk_hist, dev_err);
  dispatch_scan_kernel<<<E, 1024, 0, cs>>>(chunk_hist, E, (int)nblk, chunk_rel, counts);
  dispatch_scatter_kernel<<<(int)nblk, kDispThreads, sh3, cs>>>(topk_idx, N, E, (int)nblk,
                                                                chunk_rel, counts, off, perm,
                                                                inv);
  return launch_status();
}
