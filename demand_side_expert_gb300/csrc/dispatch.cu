// Forward dispatch permutation, row re-index, quota rule, workspace and the
// device error word.
//
// Dispatch is a stable counting sort of the N = T*K pairs by expert id
// ("Least-Loaded Expert Parallelism", Sec. 2.1 re-index and Alg. 4 sort of
// the flattened indices; LRMoE Alg. 1 counts N_e). Up to 2^17 pairs it is one
// launch of one 16-CTA cluster (8 where the GPU cannot schedule 16;
// dispatch_fused_kernel below); beyond that, three launches with no
// inter-CTA waiting:
//   1. per-chunk histogram (each CTA owns kChunk consecutive pairs),
//   2. one CTA per expert scans that expert's chunk counts: the chunk's first
//      position inside the expert's segment, and the expert's count,
//   3. each CTA derives the expert offsets from the counts (a block scan),
//      then replays its chunk warp by warp; inside a warp, lanes that share
//      an expert are ranked with __match_any_sync, so positions follow
//      ascending pair index (stability) without atomics on the output.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace lrm {

constexpr int kDispThreads = 256;  // 8 warps
constexpr int kDispWarps = kDispThreads / 32;
constexpr int kPairsPerWarp = 256;
constexpr int kChunk = kDispWarps * kPairsPerWarp;  // 2048 pairs per CTA

inline int dispatch_chunks(int64_t N) {
  return (int)std::max<int64_t>(1, (N + kChunk - 1) / kChunk);
}

inline size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

size_t workspace_bytes(const lrm_shape* s) {
  const int64_t N = (int64_t)s->T * s->K;
  const size_t chunk_tables = align256((size_t)2 * s->E * dispatch_chunks(N) * 4);
  return kWsHeaderBytes + chunk_tables;
}

__device__ __forceinline__ int clamp_expert(int e, int E, int32_t* err) {
  if (e < 0 || e >= E) {
    flag_error(err, LRM_DEVERR_EXPERT_ID);
    e = e < 0 ? 0 : E - 1;
  }
  return e;
}

// Warp-private histograms of one chunk: hist[w * E + e].
__device__ __forceinline__ void chunk_histogram(const int32_t* __restrict__ idx,
                                                int64_t N, int E, int32_t* hist,
                                                int32_t* err) {
  for (int i = threadIdx.x; i < kDispWarps * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t base = (int64_t)blockIdx.x * kChunk + (int64_t)w * kPairsPerWarp;
  for (int it = 0; it < kPairsPerWarp / 32; ++it) {
    const int64_t p = base + it * 32 + lane;
    const bool valid = p < N;
    int e = valid ? clamp_expert(idx[p], E, err) : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (valid && lane == __ffs(peers) - 1) hist[w * E + e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDispThreads)
dispatch_hist_kernel(const int32_t* __restrict__ idx, int64_t N, int E, int nblk,
                     int32_t* __restrict__ chunk_hist, int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  extern __shared__ int32_t sh[];
  chunk_histogram(idx, N, E, sh, err);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int w = 0; w < kDispWarps; ++w) s += sh[w * E + e];
    chunk_hist[(int64_t)e * nblk + blockIdx.x] = s;
  }
}

// Exclusive scan across the block (blockDim.x a multiple of 32, <= 1024).
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) warp_tot[w] = inc;
  __syncthreads();
  if (w == 0) {
    int x = lane < nw ? warp_tot[lane] : 0;
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += t;
    }
    if (lane < nw) warp_tot[lane] = xi - x;
    if (lane == 31) *total = xi;
  }
  __syncthreads();
  const int r = warp_tot[w] + inc - v;
  __syncthreads();
  return r;
}

// One CTA per expert e: chunk_rel[e][b] = sum of the expert's counts in chunks
// before b (its first position inside the expert's segment); counts[e] = the
// expert's total. Chunks are scanned a block-width at a time with a carry.
__global__ void __launch_bounds__(1024)
dispatch_scan_kernel(const int32_t* __restrict__ chunk_hist, int E, int nblk,
                     int32_t* __restrict__ chunk_rel, int32_t* __restrict__ counts) {
  pdl_begin();  // predecessor complete before any global access
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int e = blockIdx.x;
  if (e >= E) return;
  const int32_t* h = chunk_hist + (int64_t)e * nblk;
  int32_t* rel = chunk_rel + (int64_t)e * nblk;
  int carry = 0;
  for (int b0 = 0; b0 < nblk; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    const int v = b < nblk ? h[b] : 0;
    const int excl = block_exclusive_scan(v, warp_tot, &total);
    if (b < nblk) rel[b] = carry + excl;
    carry += total;  // read before any thread can pass the next scan's first barrier
  }
  if (threadIdx.x == 0) counts[e] = carry;
}

__global__ void __launch_bounds__(kDispThreads)
dispatch_scatter_kernel(const int32_t* __restrict__ idx, int64_t N, int E, int nblk,
                        const int32_t* __restrict__ chunk_rel,
                        const int32_t* __restrict__ counts, int32_t* __restrict__ off,
                        int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  pdl_begin();  // predecessor complete before any global access
  extern __shared__ int32_t sh[];
  int32_t* hist = sh;                       // [8][E]
  int32_t* run = sh + kDispWarps * E;       // [8][E] next position per warp
  int32_t* eoff = run + kDispWarps * E;     // [E] expert offsets
  __shared__ int warp_tot[32];
  __shared__ int total;
  // expert offsets: exclusive scan of the counts, a block-width at a time
  int carry = 0;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    const int v = e < E ? counts[e] : 0;
    const int excl = block_exclusive_scan(v, warp_tot, &total);
    if (e < E) {
      eoff[e] = carry + excl;
      if (blockIdx.x == 0) off[e] = carry + excl;
    }
    carry += total;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) off[E] = carry;
  chunk_histogram(idx, N, E, hist, nullptr);  // starts with a barrier: eoff is visible
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int acc = eoff[e] + chunk_rel[(int64_t)e * nblk + blockIdx.x];
    for (int w = 0; w < kDispWarps; ++w) {
      run[w * E + e] = acc;
      acc += hist[w * E + e];
    }
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t base = (int64_t)blockIdx.x * kChunk + (int64_t)w * kPairsPerWarp;
  for (int it = 0; it < kPairsPerWarp / 32; ++it) {
    const int64_t p = base + it * 32 + lane;
    const bool valid = p < N;
    int e = -1;
    if (valid) {
      e = idx[p];
      e = e < 0 ? 0 : (e >= E ? E - 1 : e);
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const int pos = run[w * E + e] + __popc(peers & lanemask_lt());
      perm[pos] = (int32_t)p;
      inv[p] = pos;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) run[w * E + e] += __popc(peers);
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Single-launch variant for up to kFusedMaxPairs pairs: one cluster of
// 16 CTAs (a non-portable cluster size, used where the GPU can schedule it),
// else 8. Each CTA counts its contiguous share of the pairs per warp
// (warp w of CTA c covers a contiguous sub-range, so warp order = pair order);
// the CTAs read each other's per-expert counts through distributed shared
// memory to get the expert offsets and their own bases, then replay their
// share in order exactly like dispatch_scatter_kernel. No workspace, no
// second launch, and the cluster barriers are hardware barriers (no spin).
// ---------------------------------------------------------------------------
constexpr int kFusedCtas = 8;         // portable cluster size
constexpr int kFusedCtasMax = 16;     // non-portable cluster size, where available
constexpr int kFusedThreads = 1024;
constexpr int kFusedWarps = kFusedThreads / 32;
#ifndef LRM_DISPATCH_FUSED_MAX
#define LRM_DISPATCH_FUSED_MAX (1 << 17)
#endif
constexpr int64_t kFusedMaxPairs = LRM_DISPATCH_FUSED_MAX;

__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ int ld_peer_smem(const int32_t* local, uint32_t rank) {
  uint32_t laddr = static_cast<uint32_t>(__cvta_generic_to_shared(local)), raddr;
  int v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(laddr), "r"(rank));
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(raddr) : "memory");
  return v;
}

// Launched as one cluster spanning the whole grid (gridDim.x CTAs).
__global__ void __launch_bounds__(kFusedThreads)
dispatch_fused_kernel(const int32_t* __restrict__ idx, int64_t N, int E,
                      int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                      int32_t* __restrict__ counts, int32_t* __restrict__ off, int32_t* err) {
  pdl_begin();  // predecessor complete before any global access
  extern __shared__ int32_t sh[];
  int32_t* wh = sh;                        // [32 warps][E]: counts, then exclusive bases
  int32_t* cta_cnt = sh + kFusedWarps * E;  // [E] this CTA's counts (read by peers)
  int32_t* base = cta_cnt + E;             // [E] first position of this CTA's pairs
  __shared__ int warp_tot[32];
  __shared__ int total;
  const uint32_t rank = cluster_ctarank();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nctas = (int)gridDim.x;
  const int64_t per_cta = (N + nctas - 1) / nctas;
  const int64_t per_warp = ((per_cta + kFusedWarps - 1) / kFusedWarps + 31) & ~int64_t(31);
  const int64_t c_lo = (int64_t)rank * per_cta, c_hi = min(N, c_lo + per_cta);
  const int64_t w_lo = min(c_hi, c_lo + w * per_warp), w_hi = min(c_hi, w_lo + per_warp);

  for (int i = threadIdx.x; i < kFusedWarps * E; i += kFusedThreads) wh[i] = 0;
  __syncthreads();
  for (int64_t b = w_lo; b < w_hi; b += 32) {
    const int64_t p = b + lane;
    const bool valid = p < w_hi;
    const int e = valid ? clamp_expert(idx[p], E, err) : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (valid && lane == __ffs(peers) - 1) wh[w * E + e] += __popc(peers);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kFusedThreads) {
    int run = 0;
    for (int v = 0; v < kFusedWarps; ++v) {
      const int c = wh[v * E + e];
      wh[v * E + e] = run;
      run += c;
    }
    cta_cnt[e] = run;
  }
  cluster_barrier();  // every CTA's counts are visible cluster-wide
  for (int e0 = 0; e0 < E; e0 += kFusedThreads) {
    const int e = e0 + threadIdx.x;
    int tot = 0, before = 0;
    if (e < E) {
      for (uint32_t c = 0; c < (uint32_t)nctas; ++c) {
        const int v = ld_peer_smem(&cta_cnt[e], c);
        tot += v;
        if (c < rank) before += v;
      }
    }
    const int excl = block_exclusive_scan(e < E ? tot : 0, warp_tot, &total);
    __shared__ int carry;
    if (threadIdx.x == 0 && e0 == 0) carry = 0;
    __syncthreads();
    if (e < E) {
      base[e] = carry + excl + before;
      if (rank == 0) {
        counts[e] = tot;
        off[e] = carry + excl;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += total;
    __syncthreads();
  }
  if (rank == 0 && threadIdx.x == 0) off[E] = (int32_t)N;
  cluster_barrier();  // no CTA leaves while peers may still read its counts
  for (int64_t b = w_lo; b < w_hi; b += 32) {
    const int64_t p = b + lane;
    const bool valid = p < w_hi;
    int e = -1;
    if (valid) {
      e = idx[p];
      e = e < 0 ? 0 : (e >= E ? E - 1 : e);
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const int pos = base[e] + wh[w * E + e] + __popc(peers & lanemask_lt());
      perm[pos] = (int32_t)p;
      inv[p] = pos;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wh[w * E + e] += __popc(peers);
    __syncwarp();
  }
}

__global__ void permute_rows_kernel(const int32_t* __restrict__ perm, int n_rows,
                                    const uint4* __restrict__ src, uint4* __restrict__ dst,
                                    int64_t vec_per_row) {
  pdl_begin();  // predecessor complete before any global access
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t pos = warp; pos < n_rows; pos += nwarps) {
    const int p = perm[pos];
    if (p < 0 || p >= n_rows) continue;
    const uint4* s = src + (int64_t)p * vec_per_row;
    uint4* d = dst + pos * vec_per_row;
    for (int64_t c = lane; c < vec_per_row; c += 32) d[c] = ld_stream(s + c);
  }
}

__global__ void quota_kernel(const int32_t* __restrict__ counts, int E, int num, int den,
                             int cap, int32_t* __restrict__ quota) {
  pdl_begin();  // predecessor complete before any global access
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int64_t n = counts[e];
  int64_t q = ((int64_t)num * n + den - 1) / den;
  if (cap > 0 && q > cap) q = cap;
  quota[e] = (int32_t)q;
}

__global__ void clear_header_kernel(int32_t* w) {
  if (threadIdx.x < kWsHeaderWords) w[threadIdx.x] = 0;
}

// One launch of the single-cluster dispatch (N <= dispatch_fused_max_pairs()):
// needs no workspace; expert ids outside [0, E) are clamped and flag
// LRM_DEVERR_EXPERT_ID in *err (err may be null).
lrm_status launch_dispatch_fused(const int32_t* topk_idx, int64_t N, int E, int32_t* perm,
                                 int32_t* inv, int32_t* counts, int32_t* off, int32_t* err,
                                 cudaStream_t cs) {
  const size_t shf = ((size_t)kFusedWarps * E + 2 * E) * 4;
  if (shf > 48 * 1024 &&
      cudaFuncSetAttribute(dispatch_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)shf) != cudaSuccess) {
    (void)cudaGetLastError();  // leave no error behind for a later call to report
    return LRM_ERR_CUDA;
  }
  // 16 CTAs (twice the SMs) where a 16-CTA cluster of this kernel fits
  // the GPU, else the portable 8
  int nctas = kFusedCtas;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = shf;
  cfg.stream = cs;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = LRM_PDL ? 2 : 1;
  if (cudaFuncSetAttribute(dispatch_fused_kernel,
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cfg.gridDim = dim3(kFusedCtasMax);
    attr[0].val.clusterDim.x = kFusedCtasMax;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, dispatch_fused_kernel, &cfg) == cudaSuccess &&
        clusters >= 1)
      nctas = kFusedCtasMax;
  }
  (void)cudaGetLastError();  // a refused query leaves the portable size
  cfg.gridDim = dim3(nctas);
  attr[0].val.clusterDim.x = nctas;
  if (cudaLaunchKernelEx(&cfg, dispatch_fused_kernel, topk_idx, N, E, perm, inv, counts, off,
                         err) != cudaSuccess)
    return LRM_ERR_CUDA;
  return launch_status();
}

int64_t dispatch_fused_max_pairs() { return kFusedMaxPairs; }

}  // namespace lrm

using namespace lrm;

extern "C" size_t lrm_workspace_bytes(const lrm_shape* shape) {
  if (check_shape(shape) != LRM_OK) return 0;
  return workspace_bytes(shape);
}

extern "C" const char* lrm_status_string(lrm_status s) {
  switch (s) {
    case LRM_OK: return "LRM_OK";
    case LRM_ERR_INVALID_ARG: return "LRM_ERR_INVALID_ARG";
    case LRM_ERR_UNSUPPORTED: return "LRM_ERR_UNSUPPORTED";
    case LRM_ERR_WORKSPACE: return "LRM_ERR_WORKSPACE";
    case LRM_ERR_CUDA: return "LRM_ERR_CUDA";
  }
  return "LRM_ERR_UNKNOWN";
}

extern "C" lrm_status lrm_clear_device_error(void* ws, size_t ws_bytes, void* stream) {
  LRM_NVTX("lrm_clear_device_error");
  if (!ws || ws_bytes < kWsHeaderBytes) return LRM_ERR_WORKSPACE;
  clear_header_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(error_word(ws));
  return launch_status();
}

extern "C" lrm_status lrm_get_device_error(const void* ws, size_t ws_bytes,
                                           int32_t* code_out, void* stream) {
  LRM_NVTX("lrm_get_device_error");
  if (!ws || ws_bytes < kWsHeaderBytes) return LRM_ERR_WORKSPACE;
  if (!code_out) return LRM_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LRM_ERR_CUDA;
  if (cudaMemcpy(code_out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LRM_ERR_CUDA;
  return LRM_OK;
}

extern "C" lrm_status lrm_dispatch_permute(const lrm_shape* s, const int32_t* topk_idx,
                                           int32_t* perm, int32_t* inv, int32_t* counts,
                                           int32_t* off, void* ws, size_t ws_bytes,
                                           void* stream) {
  LRM_NVTX("lrm_dispatch_permute");
  lrm_status st = check_shape(s);
  if (st != LRM_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes)) != LRM_OK) return st;
  const int64_t N = (int64_t)s->T * s->K;
  if ((N > 0 && (!topk_idx || !perm || !inv)) || !counts || !off)
    return LRM_ERR_INVALID_ARG;
  cudaStream_t cs = (cudaStream_t)stream;
  const int E = s->E;
  if (N <= kFusedMaxPairs)
    return launch_dispatch_fused(topk_idx, N, E, perm, inv, counts, off, error_word(ws), cs);
  const int nblk = dispatch_chunks(N);
  int32_t* chunk_hist = reinterpret_cast<int32_t*>((char*)ws + kWsHeaderBytes);
  int32_t* chunk_rel = chunk_hist + (int64_t)E * nblk;
  const size_t sh1 = (size_t)kDispWarps * E * 4;
  const size_t sh3 = 2 * sh1 + (size_t)E * 4;
  if (sh3 > 48 * 1024) {
    cudaFuncSetAttribute(dispatch_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sh1);
    cudaFuncSetAttribute(dispatch_scatter_kernel,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sh3);
  }
  launch_k(dispatch_hist_kernel, dim3(nblk), dim3(kDispThreads), sh1, cs, topk_idx, N, E, nblk, chunk_hist,
                                                        error_word(ws));
  launch_k(dispatch_scan_kernel, dim3(E), dim3(1024), 0, cs, chunk_hist, E, nblk, chunk_rel,
           counts);
  launch_k(dispatch_scatter_kernel, dim3(nblk), dim3(kDispThreads), sh3, cs, topk_idx, N, E, nblk,
           (const int32_t*)chunk_rel, (const int32_t*)counts, off, perm, inv);
  return launch_status();
}

extern "C" lrm_status lrm_permute_rows(const int32_t* perm, int32_t n_rows, const void* src,
                                       void* dst, int64_t row_bytes, void* stream) {
  LRM_NVTX("lrm_permute_rows");
  if (n_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return LRM_ERR_INVALID_ARG;
  if (n_rows == 0) return LRM_OK;
  if (!perm || !src || !dst) return LRM_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return LRM_ERR_UNSUPPORTED;
  const int64_t vec = row_bytes / 16;
  const int64_t warps = std::min<int64_t>(n_rows, (int64_t)num_sms() * 64);
  const int blocks = (int)((warps + 7) / 8);
  launch_k(permute_rows_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, 
      perm, n_rows, (const uint4*)src, (uint4*)dst, vec);
  return launch_status();
}

extern "C" lrm_status lrm_quota_from_rate(const int32_t* counts, int32_t E, int32_t num,
                                          int32_t den, int32_t cap, int32_t* quota,
                                          void* stream) {
  LRM_NVTX("lrm_quota_from_rate");
  if (E <= 0 || den <= 0 || num < 0 || num > den) return LRM_ERR_INVALID_ARG;
  if (!counts || !quota) return LRM_ERR_INVALID_ARG;
  launch_k(quota_kernel, dim3((E + 255) / 256), dim3(256), 0, (cudaStream_t)stream, counts, E, num, den, cap,
                                                                  quota);
  return launch_status();
}
