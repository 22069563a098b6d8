// Variable-size grouped GEMMs of the SwiGLU expert backward on tcgen05
// tensor cores (BF16 operands, FP32 accumulation in tensor memory).
//
// LRMoE Alg. 1 (PackedExpertBackward) and Sec. 3.4: the four expert-backward
// products run over each expert's retained rows only; the retained count m_e
// is the row dimension of the data-gradient products (G1, G4) and the
// reduction dimension of the weight-gradient products (G2, G3). Group sizes
// are read from device memory (sel_off); nothing is padded:
//   G1  dphi = dy_c W_down[e]^T   [m_e x H], epilogue: SwiGLU gradient
//       -> dab_c = [da | db] (bf16); reads the saved ab_c rows.
//   G2  dW_down[e] = phi_c^T dy_c   [H x D], reduction over m_e.
//   G3  [dW_gate | dW_up][e] = x_c^T dab_c   [D x 2H], reduction over m_e.
//   G4  dx_c = da W_gate[e]^T + db W_up[e]^T   [m_e x D] (fp32).
// The forward expert pass that produces the saved state runs on the same
// kernel over every routed row (groups from the dispatch offsets):
//   F1  [a | b] = x_disp [W_gate[e] | W_up[e]]   [n_e x 2H], epilogue:
//       phi = SiLU(a) * b; writes ab and phi (bf16). A 256-column tile holds
//       128 gate columns and the same 128 up columns, so every thread has the
//       a and b of its outputs.
//   F2  y = phi W_down[e]   [n_e x D] (bf16).
// Both read the weights in their stored layout (MN-major B operands) and
// write an epilogue warp's 32 x 32 output blocks that lie inside the group
// through shared memory with TMA stores (a block crossing the group's end
// takes 16-byte row stores). F1 over
// the compacted retained rows (groups from sel_off, phi not written) is the
// retained-only recompute of [a | b] in the backward.
//
// Kernel shape (one CTA per SM, persistent over a device-computed tile list;
// the data-gradient and forward products run on CTA pairs, 256-row tiles
// with tcgen05.mma.cta_group::2, each CTA reading half of the B tile; the
// weight-gradient products on single CTAs that take their tiles from a queue
// in the workspace header):
//   warp 0    TMA producer: 128x64 A and 256x64 (pair: 128x64) B tiles,
//             128-byte swizzle, a ring of 48 KB (pair: 32 KB) stages, as deep
//             as shared memory allows (at most 6), guarded by mbarriers;
//   warp 1    allocates 512 TMEM columns, one elected lane issues
//             tcgen05.mma (M=128, N=256, K=16) into one of two 256-column
//             accumulators (a wide tile, FC1 dgrad on long K, fills both:
//             256 x 512 per CTA pair, two B boxes per 48 KB stage);
//             tcgen05.commit frees smem stages and hands finished
//             accumulators to the epilogue;
//   warps 2-9 epilogue: tcgen05.ld rows out of TMEM (one row per thread,
//             two warps per 32-lane quarter, each half of the columns);
//             G1 fuses the SwiGLU gradient (saved a, b rows prefetched one
//             32-column chunk ahead); FP32 outputs go through a per-warp
//             32x32 swizzled shared-memory block and a TMA bulk-tensor store,
//             so every 128-byte line is written whole.
//   warps 10-13 (weight-gradient products on single CTAs only): when the A
//             rows are read in place by index (phi rows by dispatch position,
//             x rows by token) instead of from compacted copies, these warps
//             gather them with 16-byte async copies into the swizzled layout.
// Data-gradient tiles are cut at group ends (rows past m_e are computed and
// masked on store). Weight-gradient tiles reduce over [sel_off[e],
// sel_off[e+1]) in 64-row blocks; rows of the last block that belong to the
// next group are zeroed in shared memory before the MMA reads them, and
// 16-row slices past the group end are not issued. Experts with no retained
// rows get zero weight gradients. Every mbarrier wait is bounded: on timeout
// the CTA flags LRM_DEVERR_TIMEOUT, stops issuing, drains its copies and
// MMAs, frees TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace lrm {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64;  // rows per CTA, accumulator columns, K block
constexpr int MAX_STAGES = 6;  // operand ring depth (runtime: as deep as shared memory allows)
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each half the columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kGatherWarps = 4;  // weight-gradient products: A rows gathered by index
// Weight-gradient products on single CTAs take their tiles from a queue in
// the workspace header (1) instead of a fixed deal (0).
#ifndef LRM_TC_WG_QUEUE
#define LRM_TC_WG_QUEUE 1
#endif
// CTAs that take their tiles from the short end of the longest-first list: those
// with blockIdx % 4 below this count (0: every CTA takes from the long end). A
// quarter or half of the CTAs at the short end measured 3-7% slower on the
// weight-gradient products of the large layers: the store-bound short tiles then
// run beside the long ones, whose operand loads slow down under their stores.
#ifndef LRM_TC_WG_TAIL_QUARTERS
#define LRM_TC_WG_TAIL_QUARTERS 0
#endif
// forward products: full 32-row blocks of their bf16 outputs through staged
// TMA stores (1) instead of 16-byte row stores (0)
#ifndef LRM_TC_FWD_STAGED
#define LRM_TC_FWD_STAGED 1
#endif
constexpr int kTQ = 8;  // tile ids in flight between the copy lane and the other roles
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
// B rows a CTA loads: all BN columns alone, half of them in a CTA pair
template <bool PAIR>
struct Cfg {
  static constexpr int kBRows = PAIR ? BN / 2 : BN;
  static constexpr int kTileRows = PAIR ? 2 * BM : BM;  // M of one MMA
};
constexpr uint32_t BOX_BYTES = 64 * 64 * 2;  // one 64x64 MN-major box
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t STAGING_BYTES = 32 * 32 * 4;  // one 32x32 fp32 block, 128B-swizzled
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per pipeline wait
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s per drain wait

enum Mode { kG1 = 0, kG2 = 1, kG3 = 2, kG4 = 3, kF1 = 4, kF2 = 5 };

// Wide tiles (W): a data-gradient product on CTA pairs whose tile is 256 rows
// by 512 columns. One A tile feeds two 256-column accumulators, so a CTA takes
// in 24 KB of operands per 128 x 256 x 64 block of MMA work instead of 32 KB,
// and each ring stage carries eight MMAs; but both accumulators then belong to
// one tile, whose epilogue no longer overlaps the next tile's MMAs. FC1 dgrad
// runs wide when its K extent is long (wide_fc1_dgrad).
template <int MODE, bool PAIR, bool W>
struct Ring {
  static constexpr bool kWide = W && PAIR && (MODE == kG1 || MODE == kG4);
  static constexpr uint32_t kBBytes = Cfg<PAIR>::kBRows * BK * 2;  // one B box of a CTA
  static constexpr uint32_t kStageBytes = A_BYTES + (kWide ? 2 : 1) * kBBytes;  // 32-48 KB
  static constexpr int kTileCols = kWide ? 2 * BN : BN;  // output columns of a tile
};

// Operand maps (A, B, second B for G4 and F1) and output maps (G2: dW_down,
// G3: dW_gate and dW_up, G4: dx_c), passed by value in parameter space.
struct Maps {
  CUtensorMap a, b, b2, o1, o2;
};

struct Params {
  uint64_t wait_ns;  // bound of every pipeline wait
  int selftest;      // 1: the copy warp delivers nothing (bounded-wait self-test)
  int E, D, H;
  int n_rows;      // row capacity of the compacted buffers
  int stage_bufs;  // 32x32 fp32 staging blocks per epilogue warp (0 to 3)
  int stages;      // depth of the operand ring (3 to 6, as shared memory allows)
  const int32_t* sel_off;
  const __nv_bfloat16* ab_c;
  __nv_bfloat16* dab_c;
  float* out0;
  float* out1;
  __nv_bfloat16* ob0;  // F1: ab, F2: y
  __nv_bfloat16* ob1;  // F1: phi
  // gathered operands (null: compacted rows): G1 reads the saved [a | b] row
  // ab_rows[j] of compacted row j; G2 / G3 read their A operand (phi / x)
  // row a_rows[j] of a_src [a_src_rows, a_src_cols] with 16-byte async copies
  const int32_t* ab_rows;
  const int32_t* a_rows;
  const __nv_bfloat16* a_src;
  int a_src_rows, a_src_cols;
  int ab_src_rows;  // rows of the [a | b] source (bound for ab_rows)
  int32_t* err;
  // weight-gradient tile queue: [positions taken from the head | from the tail
  // (one 64-bit word), CTAs done, tiles handed out]
  int32_t* queue;
};

// ----------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity. Returns false when the
// CTA is aborting or after kWaitNs; a timeout raises the abort flag.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity,
                                          volatile int* abort_flag, int32_t* err,
                                          uint64_t limit_ns) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort_flag = 1;
      flag_error(err, LRM_DEVERR_TIMEOUT);
      return false;
    }
  }
}
// Whole-warp bounded wait: every lane polls, lane 0 alone decides to give up,
// so the warp leaves together (tcgen05.ld and .sync.aligned ops that follow
// need a converged warp). A completed phase stays observable until the
// waiting warp itself lets the pipeline advance, so __all_sync terminates.
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity,
                                          volatile int* abort_flag, int32_t* err,
                                          uint64_t limit_ns) {
  const int lane = threadIdx.x & 31;
  uint64_t t0 = 0;
  if (lane == 0) t0 = globaltimer();
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try(b, parity))) return true;
    int give_up = 0;
    if (lane == 0) {
      if (*abort_flag) {
        give_up = 1;
      } else if (globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        flag_error(err, LRM_DEVERR_TIMEOUT);
        give_up = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}
__device__ __forceinline__ void mbar_drain(uint64_t* b, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try(b, parity) && globaltimer() - t0 < kDrainNs) {
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}
// 16-byte asynchronous copy global -> shared (zero-filled when !valid), and
// an arrival on an mbarrier once all of this thread's earlier copies landed
// (counted as one of the barrier's expected arrivals)
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(su32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(su32(bar))
      : "memory");
}
// TMA bulk-tensor stores (shared -> global), completion tracked per bulk group
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x,
                                             int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(su32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x,
                                             int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(su32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until at most `pending` committed bulk groups may still read shared memory
__device__ __forceinline__ void bulk_wait_read(int pending) {
  if (pending >= 2)
    asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory");
  else if (pending == 1)
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
  else
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- CTA pairs (cluster of 2) ----
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t mapa(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(su32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// arrive on a barrier of another CTA of the cluster (release at CTA scope)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// the same without ordering: for arrivals whose data is tracked by tx bytes
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   cluster_addr)
               : "memory");
}
// TMA load whose completion is counted on a barrier of either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t mbar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar_cluster)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t mbar_cluster, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar_cluster)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   su32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the barrier at the same offset in every CTA of `mask` once this
// thread's earlier pair MMAs have completed
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(su32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   su32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}
// 32 TMEM lanes x 32 consecutive 32-bit columns; thread i gets lane (base+i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format:
// start>>4 at [0,14), LBO>>4 at [16,30), SBO>>4 at [32,46), fixed 0b001 at
// [46,49), swizzle mode 2 = 128B at [61,64)).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: FP32 accumulate, BF16 A and B,
// operand majorness (0 = K-major, 1 = MN-major), N>>3 at [17,23), M>>4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) |
         ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int MODE>
struct Geo {
  static constexpr bool kWgrad = (MODE == kG2 || MODE == kG3);
  static constexpr bool kFwd = (MODE == kF1 || MODE == kF2);
  static constexpr bool kAmn = kWgrad;          // A operand MN-major
  static constexpr bool kBmn = kWgrad || kFwd;  // B operand MN-major
};

// Threads of one CTA: copy warp, MMA warp, epilogue warps, and for the
// single-CTA weight-gradient products the warps that gather A rows
template <int MODE, bool PAIR>
struct Threads {
  static constexpr int kGather = (Geo<MODE>::kWgrad && !PAIR) ? kGatherWarps : 0;
  static constexpr int kCount = kThreads + 32 * kGather;
};

// ----------------------------------------------------------------------------
// tile list
// ----------------------------------------------------------------------------
struct Tile {
  int e;       // expert
  int m0;      // dgrad: first compacted row of the unit's tile; wgrad: first output row
  int n0;      // first output column
  int nkb;     // 64-wide K blocks
  int valid;   // dgrad: rows of the unit's tile inside the group; wgrad: rows of the last K block
  int row0;    // wgrad: first compacted row of the group
  int cm0;     // this CTA's first row (m0 + rank * 128)
  int cvalid;  // dgrad: this CTA's rows inside the group (may be <= 0)
};

struct Sched {
  const int* goff;   // [E+1] group offsets (validated copy of sel_off)
  const int* tpre;   // dgrad: [E+1] tile prefix
  const int* order;  // wgrad: experts by retained rows, descending
  int E, ntn, mtiles, kdim_blocks, total, tm;  // tm: rows of a unit's tile (128 or 256)
  int tn;                                      // dgrad: output columns of a tile (256 or 512)
};

template <int MODE>
__device__ __forceinline__ Tile decode(const Sched& s, int tau, int rank) {
  Tile t;
  if constexpr (Geo<MODE>::kWgrad) {
    const int per = s.mtiles * s.ntn;
    const int r = tau / per, loc = tau - r * per;
    t.e = s.order[r];
    t.m0 = (loc / s.ntn) * s.tm;
    t.n0 = (loc % s.ntn) * BN;
    t.row0 = s.goff[t.e];
    const int m = s.goff[t.e + 1] - t.row0;
    t.nkb = (m + BK - 1) / BK;
    t.valid = m - (t.nkb - 1) * BK;
    t.cvalid = 0;
  } else {
    int lo = 0, hi = s.E;  // largest e with tpre[e] <= tau
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s.tpre[mid] <= tau) lo = mid; else hi = mid;
    }
    t.e = lo;
    const int loc = tau - s.tpre[lo];
    const int mt = loc / s.ntn;
    t.m0 = s.goff[lo] + mt * s.tm;
    t.n0 = (loc % s.ntn) * s.tn;
    t.valid = min(s.tm, s.goff[lo + 1] - t.m0);
    t.nkb = s.kdim_blocks;
    t.row0 = 0;
    t.cvalid = t.valid - rank * BM;
  }
  t.cm0 = t.m0 + rank * BM;
  return t;
}

// ----------------------------------------------------------------------------
// epilogues (one thread = one accumulator row, 32 columns per chunk)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void store_f32x32(float* dst, const uint32_t (&r)[32]) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    d[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                       __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
}

// Row `lane` of a 32x32 fp32 block into the 128B-swizzled layout a TMA store
// with a 32 x 32 box expects: 16-byte chunk j of row r sits at chunk j^(r%8).
__device__ __forceinline__ void stage_row(uint8_t* blk, int lane, const uint32_t (&r)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4*>(blk + lane * 128 + ((j ^ (lane & 7)) << 4)) =
        make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
}

// SwiGLU gradient of 32 columns, given the row's a and b values.
__device__ __forceinline__ void swiglu_chunk(const uint32_t (&r)[32], const uint4 (&av)[4],
                                             const uint4 (&bv)[4], uint4 (&dav)[4],
                                             uint4 (&dbv)[4]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float a[8], b[8], da[8], db[8];
    Vec16<__nv_bfloat16>::unpack(av[v], a);
    Vec16<__nv_bfloat16>::unpack(bv[v], b);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float dphi = __uint_as_float(r[8 * v + u]);
      const float s = __fdividef(1.0f, 1.0f + __expf(-a[u]));
      da[u] = dphi * b[u] * s * (1.0f + a[u] * (1.0f - s));
      db[u] = dphi * a[u] * s;
    }
    dav[v] = Vec16<__nv_bfloat16>::pack(da);
    dbv[v] = Vec16<__nv_bfloat16>::pack(db);
  }
}

// ----------------------------------------------------------------------------
// the kernel
// ----------------------------------------------------------------------------
// PAIR = false: one CTA per tile of 128 rows x 256 columns (tcgen05 cta_group::1).
// PAIR = true:  a cluster of two CTAs per tile of 256 x 256; each CTA loads its
//   128 A rows and half of the B rows, the even CTA issues
//   tcgen05.mma.cta_group::2 (M = 256) for both, each CTA's tensor memory holds
//   its 128 accumulator rows. Protocol per ring stage: both CTAs' copies land
//   on the even CTA's full barrier (2 arrivals + bytes); its commits arrive on
//   both CTAs' empty / accumulator-full barriers; both CTAs' epilogue warps
//   arrive on the even CTA's accumulator-empty barrier. A weight-gradient K
//   block whose last 16-row slice crosses the group end is the exception: the
//   odd CTA's copy lands on its own full barrier, its (otherwise idle) MMA warp
//   zeroes the rows past the group end and then arrives on the even CTA's.
template <int MODE, bool PAIR, bool W>
__global__ void __launch_bounds__(Threads<MODE, PAIR>::kCount, 1)
grouped_gemm_kernel(const __grid_constant__ Maps maps, const Params p) {
  constexpr int NT = Threads<MODE, PAIR>::kCount;
  constexpr int NG = Threads<MODE, PAIR>::kGather;
  constexpr bool WG = Geo<MODE>::kWgrad;
  constexpr int BNL = Cfg<PAIR>::kBRows;
  constexpr bool WIDE = Ring<MODE, PAIR, W>::kWide;
  constexpr uint32_t STB = Ring<MODE, PAIR, W>::kStageBytes;
  constexpr uint32_t BBOX = Ring<MODE, PAIR, W>::kBBytes;
  constexpr int TN = Ring<MODE, PAIR, W>::kTileCols;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int STAGES = p.stages;
  uint8_t* stages = smem;
  uint8_t* staging = smem + STAGES * STB;  // kEpiWarps x stage_bufs blocks
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(staging + kEpiWarps * p.stage_bufs * STAGING_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + MAX_STAGES;
  uint64_t* tfull = bars + 2 * MAX_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* tq_full = drain + 1;     // [kTQ] tile id published
  uint64_t* tq_empty = tq_full + kTQ;  // [kTQ] tile id read by every consumer warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tq_empty + kTQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bad_flag = const_cast<int*>(abort_flag) + 1;
  int* goff = bad_flag + 1;          // [E+1]
  int* tab = goff + p.E + 1;         // dgrad: tpre[E+1]; wgrad: order[E]
  int* tq_id = tab + p.E + 1;        // [kTQ]
  const CUtensorMap* mapA = &maps.a;
  const CUtensorMap* mapB = &maps.b;
  const CUtensorMap* mapB2 = &maps.b2;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E;
  const int rank = PAIR ? (int)cluster_rank() : 0;
  const bool leader = rank == 0;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const bool queued = WG && !PAIR && LRM_TC_WG_QUEUE && p.queue != nullptr;
  // wide tiles: output columns of the product; a tile's second accumulator
  // (columns n0 + 256 ...) is skipped, copies and MMAs, when none of its
  // columns exist
  const int dg_cols = MODE == kG1 ? p.H : p.D;
  // warps that read every tile id: MMA, epilogue, and the gather warps at work
  const int gathering = (NG > 0 && p.a_rows && !p.selftest) ? min(NG, STAGES) : 0;

  // --- set-up that reads nothing a kernel writes: barriers, TMEM, maps ----
  if (tid == 0) {
    *abort_flag = 0;
    *bad_flag = 0;
    // full: the copy warp's arrival (two in a pair's even CTA), plus one per
    // lane of the copy warp when it gathers A rows with async copies
    const uint32_t full_count = (PAIR && leader) ? 2u : (NG > 0 && p.a_rows) ? 33u : 1u;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], full_count);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps * (PAIR ? 2 : 1));
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kTQ; ++i) {
      mbar_init(&tq_full[i], 1);
      mbar_init(&tq_empty[i], 1 + kEpiWarps + gathering);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0 && !p.selftest) {
    prefetch_map(mapA);
    prefetch_map(mapB);
    if (MODE == kG4 || MODE == kF1) prefetch_map(mapB2);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  // --- the previous kernel in the stream is complete from here on ----------
  pdl_begin();
  __syncthreads();
  // --- validated group offsets and the tile table --------------------------
  for (int i = tid; i <= E; i += NT) {
    const int v = p.sel_off[i];
    const int prev = i > 0 ? p.sel_off[i - 1] : 0;
    goff[i] = v;
    if (v < prev || (i == 0 && v != 0) || v > p.n_rows) *bad_flag = 1;
  }
  __syncthreads();
  if (*bad_flag) {
    for (int i = tid; i <= E; i += NT) goff[i] = 0;
    if (tid == 0) flag_error(p.err, LRM_DEVERR_INDEX);
  }
  __syncthreads();
  if constexpr (MODE == kG1) {
    // 64 zero rows after the retained ones: the padding the FC1 weight-gradient
    // product reads as B past the last group (see zero_tail)
    if (blockIdx.x == 0 && p.dab_c) {
      const int64_t m = goff[E];
      const int64_t rows = min((int64_t)BK, (int64_t)p.n_rows - m);
      const int64_t n16 = rows * 2 * p.H / 8;  // 16-byte chunks
      uint4* z = reinterpret_cast<uint4*>(p.dab_c + m * 2 * p.H);
      for (int64_t i = tid; i < n16; i += NT) z[i] = make_uint4(0, 0, 0, 0);
    }
  }

  Sched sc;
  sc.goff = goff;
  sc.E = E;
  sc.tm = Cfg<PAIR>::kTileRows;
  sc.tn = TN;
  if constexpr (MODE == kG1) {
    sc.ntn = (p.H + TN - 1) / TN;
    sc.kdim_blocks = p.D / BK;
  } else if constexpr (MODE == kG4) {
    sc.ntn = (p.D + TN - 1) / TN;
    sc.kdim_blocks = 2 * p.H / BK;
  } else if constexpr (MODE == kF1) {
    sc.ntn = (p.H + BN / 2 - 1) / (BN / 2);
    sc.kdim_blocks = p.D / BK;
  } else if constexpr (MODE == kF2) {
    sc.ntn = (p.D + BN - 1) / BN;
    sc.kdim_blocks = p.H / BK;
  } else if constexpr (MODE == kG2) {
    sc.ntn = (p.D + BN - 1) / BN;
    sc.mtiles = (p.H + sc.tm - 1) / sc.tm;
  } else {
    sc.ntn = (2 * p.H + BN - 1) / BN;
    sc.mtiles = (p.D + sc.tm - 1) / sc.tm;
  }
  if constexpr (WG) {
    // experts ordered by retained rows (descending, then by id): longest first
    for (int e = tid; e < E; e += NT) {
      const int m = goff[e + 1] - goff[e];
      int rank_e = 0;
      for (int f = 0; f < E; ++f) {
        const int mf = goff[f + 1] - goff[f];
        rank_e += (mf > m) || (mf == m && f < e);
      }
      tab[rank_e] = e;
    }
    sc.order = tab;
    sc.total = E * sc.mtiles * sc.ntn;
  } else {
    if (warp == 0) {  // tile prefix over experts, 32 at a time
      int carry = 0;
      for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        const int tiles = e < E ? ((goff[e + 1] - goff[e] + sc.tm - 1) / sc.tm) * sc.ntn : 0;
        int inc = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += t;
        }
        if (e < E) tab[e] = carry + inc - tiles;
        carry += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (lane == 0) tab[E] = carry;
    }
    sc.tpre = tab;
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if constexpr (!WG) sc.total = tab[E];
  const uint32_t tmem_base = *tmem_slot;

  // stage s's rows [valid, 16 * ceil(valid / 16)) of every box of this CTA
  // belong to the next group or lie past the retained rows: zero them
  // Rows past the group end in the last K block: a product term vanishes if
  // its A row is zero and its B row finite. B rows there are the next group's
  // (finite), or rows past the retained rows, which the kernels producing
  // the B operands write as zeros for 64 rows (dy_c: the compaction; dab_c:
  // the FC2 dgrad product), or rows past the buffer (zero-filled by TMA). So
  // only the A boxes' rows [valid, 16 * ceil(valid / 16)) are zeroed here
  // (gathered A rows arrive zero-filled and need nothing).
  auto zero_tail = [&](uint8_t* a_s, int valid) {
    const int n = (16 * ((valid + 15) >> 4) - valid) * 8;  // 16-byte chunks per box
#pragma unroll
    for (int bx = 0; bx < BM / 64; ++bx) {
      uint8_t* row0 = a_s + bx * BOX_BYTES + valid * 128;
      for (int idx = lane; idx < n; idx += 32)  // whole 128-byte rows: no swizzle
        *reinterpret_cast<uint4*>(row0 + (idx >> 3) * 128 + (idx & 7) * 16) =
            make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    __syncwarp();
  };

  // The tile sequence every role of this CTA walks, one call per tile r =
  // 0, 1, ...; a value >= sc.total ends it.
  //
  // Fixed deal: tile r of this unit (CTA or CTA pair), serpentine over the
  // units, so that with tiles sorted longest first (weight-gradient products)
  // every unit's total stays close to the mean.
  //
  // Queue (weight-gradient products on single CTAs): the copy lane takes the
  // next position of the longest-first list with an atomic add and publishes
  // the tile id in a ring of kTQ slots that the MMA, epilogue and gather warps
  // read in order. A tile's cost varies with its group (long groups: bound by
  // the tensor pipe; short ones and empty ones: by the fp32 stores) and with
  // the SM, so a fixed deal ends unevenly (CTAs measured up to 20% apart);
  // taking tiles as the CTA frees up ends within about one tile.
  auto tile_of = [&](int r) -> int {
    if (queued) {
      const int slot = r % kTQ;
      if (!warp_wait(&tq_full[slot], (uint32_t)(r / kTQ) & 1u, abort_flag, p.err, p.wait_ns))
        return sc.total;
      const int id = *reinterpret_cast<volatile int*>(&tq_id[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&tq_empty[slot]);
      return id;
    }
    return r * units + ((r & 1) ? units - 1 - unit : unit);
  };

  if (warp == 0) {
    // ===================== TMA producer =====================
    if (lane == 0 && !p.selftest) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      uint32_t tail_parity = 0;  // odd CTA of a pair: its own full barriers flip only on tails
      bool stop = false;
      int handed = 0;        // tiles this CTA took from the queue
      bool drained = false;  // the queue ran out
      // one take: a ticket and a position in one 64-bit atomic (low word: takes
      // from the head, high word: takes from the tail); a take whose two
      // counts already sum to the tile count finds the list exhausted, so the
      // two ends never hand out the same position
      const bool from_tail = (int)(blockIdx.x & 3) < LRM_TC_WG_TAIL_QUARTERS;
      auto take = [&]() -> int {
        const unsigned long long old = atomicAdd(
            reinterpret_cast<unsigned long long*>(p.queue), from_tail ? (1ull << 32) : 1ull);
        const long long h = (long long)(old & 0xffffffffull), tl = (long long)(old >> 32);
        if (h + tl >= (long long)sc.total) return sc.total;
        return from_tail ? (int)(sc.total - 1 - tl) : (int)h;
      };
      // the position of the next tile, taken one tile ahead so that the
      // atomic's round trip overlaps the current tile's copies
      int ahead = queued ? take() : 0;
      auto next = [&](int r) -> int {
        if (!queued) return tile_of(r);
        const int slot = r % kTQ;
        int tau = sc.total;
        if (mbar_wait(&tq_empty[slot], ((uint32_t)(r / kTQ) & 1u) ^ 1u, abort_flag, p.err,
                      p.wait_ns) &&
            !drained) {
          if (ahead >= 0 && ahead < sc.total) {
            tau = ahead;
            ++handed;
            ahead = take();
          } else {
            drained = true;
          }
        }
        tq_id[slot] = tau;  // published by the arrival (release)
        mbar_arrive(&tq_full[slot]);
        return tau;
      };
      for (int ri = 0, tau = next(0); tau < sc.total; tau = stop ? sc.total : next(++ri)) {
        const Tile t = decode<MODE>(sc, tau, rank);
        const bool two = WIDE && t.n0 + BN < dg_cols;
        const uint32_t stb = (WIDE && !two) ? STB - BBOX : STB;  // bytes one CTA copies
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.err, p.wait_ns)) {
            stop = true;
            break;
          }
          uint8_t* a_s = stages + stage * STB;
          uint8_t* b_s = a_s + A_BYTES;
          const bool tailz = WG && kb == t.nkb - 1 && (t.valid & 15);
          // where this CTA's copies complete: its own full barrier, or (pair,
          // odd CTA, ordinary block) the even CTA's
          const bool to_leader = PAIR && !leader && !tailz;
          const uint32_t bar_cl = to_leader ? mapa(&full[stage], 0) : 0u;
          const bool gathered_a = NG > 0 && p.a_rows != nullptr;  // A copied by the gather warps
          // A row tile of a pair whose odd CTA holds no row of the group (a
          // group of at most BM rows): the odd CTA's accumulator rows are
          // never stored, so its A box is not copied (the MMA reads whatever
          // that stage held: it only feeds those discarded rows)
          const bool odd_idle = !WG && PAIR && t.valid <= BM;
          if (!to_leader)
            mbar_expect_tx(&full[stage],
                           gathered_a                       ? STB - A_BYTES
                           : (PAIR && leader && !tailz)     ? 2 * stb - (odd_idle ? A_BYTES : 0)
                                                            : stb);
          auto load2 = [&](uint8_t* dst, const CUtensorMap* m, int x, int y) {
            if (to_leader) tma_load_2d_pair(dst, m, bar_cl, x, y);
            else tma_load_2d(dst, m, &full[stage], x, y);
          };
          auto load3 = [&](uint8_t* dst, const CUtensorMap* m, int x, int y, int z) {
            if (to_leader) tma_load_3d_pair(dst, m, bar_cl, x, y, z);
            else tma_load_3d(dst, m, &full[stage], x, y, z);
          };
          const int nb0 = t.n0 + rank * BNL;  // first B row (N) this CTA loads
          if constexpr (MODE == kG1) {
            if (leader || !odd_idle) load2(a_s, mapA, kb * BK, t.cm0);
            load3(b_s, mapB, kb * BK, nb0, t.e);
            if (WIDE && two) load3(b_s + BBOX, mapB, kb * BK, nb0 + BN, t.e);
          } else if constexpr (MODE == kG4) {
            if (leader || !odd_idle) load2(a_s, mapA, kb * BK, t.cm0);
            const int hb = p.H / BK;
            const CUtensorMap* mb = kb < hb ? mapB : mapB2;
            const int kx = (kb < hb ? kb : kb - hb) * BK;
            load3(b_s, mb, kx, nb0, t.e);
            if (WIDE && two) load3(b_s + BBOX, mb, kx, nb0 + BN, t.e);
          } else if constexpr (MODE == kF1) {
            // tile columns [0, 128): gate h0.., [128, 256): up h0..; 64 x 64 boxes
            if (leader || !odd_idle) load2(a_s, mapA, kb * BK, t.cm0);
            const int h0 = t.n0 / 2;
#pragma unroll
            for (int i = 0; i < BNL / 64; ++i) {
              const int n = rank * BNL + 64 * i;
              load3(b_s + i * BOX_BYTES, n < BN / 2 ? mapB : mapB2, h0 + (n & (BN / 2 - 1)),
                    kb * BK, t.e);
            }
          } else if constexpr (MODE == kF2) {
            if (leader || !odd_idle) load2(a_s, mapA, kb * BK, t.cm0);
#pragma unroll
            for (int i = 0; i < BNL / 64; ++i)
              load3(b_s + i * BOX_BYTES, mapB, nb0 + 64 * i, kb * BK, t.e);
          } else {
            const int y = t.row0 + kb * BK;
            // one copy per operand: the maps view a row as 64-column chunks
            // (x: column in the chunk, y: row, z: chunk), so a box of 64 rows
            // by several chunks lands as consecutive 64 x 64 blocks. (One copy
            // per 64 x 64 box made the even CTA of a pair re-issue each ring
            // slot about 1.6 us late.)
            if (!gathered_a) load3(a_s, mapA, 0, y, t.cm0 / 64);
            load3(b_s, mapB, 0, y, nb0 / 64);
          }
          if (to_leader) {
            mbar_arrive_cluster_relaxed(bar_cl);
          } else {
            uint32_t par = phase;
            if (PAIR && !leader) {
              par = (tail_parity >> stage) & 1u;
              tail_parity ^= 1u << stage;
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (par << stage);
          }
          if (++stage == (uint32_t)STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // copies on this CTA's own barriers must land before the CTA may exit
      // (in a pair the even CTA's barriers also count the odd CTA's bytes)
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s)) mbar_drain(&full[s], (issued_parity >> s) & 1u);
      if (queued) {
        // this CTA takes no more tiles: the last CTA to get here checks that
        // every tile was handed out once and rewinds the queue for the next
        // launch (which reads it only after this grid has completed)
        atomicAdd(p.queue + 3, handed);
        __threadfence();
        const int prev = atomicAdd(p.queue + 2, 1);
        if (prev < 0 || prev >= (int)gridDim.x) flag_error(p.err, LRM_DEVERR_QUEUE);
        if (prev == (int)gridDim.x - 1) {
          __threadfence();
          if (atomicAdd(p.queue + 3, 0) != sc.total) flag_error(p.err, LRM_DEVERR_QUEUE);
          atomicExch(p.queue, 0);
          atomicExch(p.queue + 1, 0);
          atomicExch(p.queue + 2, 0);
          atomicExch(p.queue + 3, 0);
        }
      }
    }
  } else if (warp == 1 && (!PAIR || leader)) {
    // ===================== MMA issuer =====================
    constexpr bool AMN = Geo<MODE>::kAmn, BMN = Geo<MODE>::kBmn;
    constexpr uint32_t idesc = idesc_bf16(Cfg<PAIR>::kTileRows, BN, AMN ? 1 : 0, BMN ? 1 : 0);
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool stop = false, issued_any = false;
    for (int ri = 0, tau = tile_of(0); tau < sc.total && !stop; tau = tile_of(++ri)) {
      const Tile t = decode<MODE>(sc, tau, rank);
      if (t.nkb <= 0) continue;
      if (!warp_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.err, p.wait_ns)) break;
      // a wide tile fills both accumulators (acc is then always 0)
      if (WIDE && !warp_wait(&tempty[1], acc_phase ^ 1, abort_flag, p.err, p.wait_ns)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      const bool two = WIDE && t.n0 + BN < dg_cols;
      for (int kb = 0; kb < t.nkb; ++kb) {
        if (!warp_wait(&full[stage], phase, abort_flag, p.err, p.wait_ns)) {
          stop = true;
          break;
        }
        uint8_t* a_s = stages + stage * STB;
        uint8_t* b_s = a_s + A_BYTES;
        const int valid = (WG && kb == t.nkb - 1) ? t.valid : BK;
        const int nks = (valid + 15) >> 4;
        if constexpr (WG) {
          // rows written by async copies (generic proxy) before the MMA reads them
          if (NG > 0 && p.a_rows) fence_async_smem();
          if ((valid & 15) && !(NG > 0 && p.a_rows)) zero_tail(a_s, valid);
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = su32(a_s), b_addr = su32(b_s);
          // MN-major: 16 K-rows = 2 x 1024 B per step, 64-column boxes
          // BOX_BYTES apart; K-major: 16 elements = 32 B per step
          uint64_t ad[BK / 16], bd[BK / 16];
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            ad[ks] = AMN ? sw128_desc(a_addr + ks * 2048, BOX_BYTES, 1024)
                         : sw128_desc(a_addr + ks * 32, 16, 1024);
            bd[ks] = BMN ? sw128_desc(b_addr + ks * 2048, BOX_BYTES, 1024)
                         : sw128_desc(b_addr + ks * 32, 16, 1024);
          }
          auto issue = [&](int ks) {
            const uint32_t accum = (kb | ks) != 0 ? 1u : 0u;
            if constexpr (PAIR) umma_bf16_pair(d_tmem, ad[ks], bd[ks], idesc, accum);
            else umma_bf16(d_tmem, ad[ks], bd[ks], idesc, accum);
            if constexpr (WIDE) {
              // the second accumulator: same A slice, the second B box (its
              // descriptor differs from the first by the box's offset >> 4)
              if (two)
                umma_bf16_pair(d_tmem + BN, ad[ks], bd[ks] + (BBOX >> 4), idesc, accum);
            }
          };
          if (nks == BK / 16) {  // a whole K block: the four MMAs back to back
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks) issue(ks);
          } else {
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              if (ks < nks) issue(ks);
          }
          if constexpr (PAIR) umma_commit_pair(&empty[stage], 3);
          else umma_commit(&empty[stage]);
        }
        issued_any = true;
        __syncwarp();
        if (++stage == (uint32_t)STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (stop) break;
      if (lane == 0) {
        if constexpr (PAIR) umma_commit_pair(&tfull[acc], 3);
        else umma_commit(&tfull[acc]);
        if constexpr (WIDE) umma_commit_pair(&tfull[1], 3);
      }
      __syncwarp();
      if constexpr (WIDE) {
        acc_phase ^= 1;
      } else {
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
    // all MMAs of this CTA (pair) must finish before TMEM is released
    if (issued_any && lane == 0) {
      if constexpr (PAIR) umma_commit_pair(drain, 1);
      else umma_commit(drain);
      mbar_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===================== odd CTA of a pair: tail forwarder =====================
    if constexpr (PAIR && WG) {
      uint32_t stage = 0, tparity = 0;
      bool stop = false;
      for (int ri = 0, tau = tile_of(0); tau < sc.total && !stop; tau = tile_of(++ri)) {
        const Tile t = decode<MODE>(sc, tau, rank);
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (kb == t.nkb - 1 && (t.valid & 15)) {
            if (!warp_wait(&full[stage], (tparity >> stage) & 1u, abort_flag, p.err, p.wait_ns)) {
              stop = true;
              break;
            }
            tparity ^= 1u << stage;
            zero_tail(stages + stage * STB, t.valid);
            if (lane == 0) mbar_arrive_cluster(mapa(&full[stage], 0));
            __syncwarp();
          }
          if (++stage == (uint32_t)STAGES) stage = 0;
        }
      }
    }
  } else if (warp >= 2 + kEpiWarps) {
    // ===================== A-row gather warps =====================
    // Weight-gradient products whose A rows are read by index: gather warp g
    // fills the A tile of every ng-th K block (g, g + ng, ...), so each warp
    // has ng ring periods to hide the latency of its index loads. ng never
    // exceeds the ring depth: a warp's previous K block is then at most one
    // ring lap behind, so the slot it waits for is at most one phase behind
    // and the parity wait cannot mistake an older phase for the one it needs
    // (with more warps than stages a warp could run two laps ahead). For one K
    // block: lane l fetches the row indices of K-block rows l and l + 32
    // before the ring slot frees; then each instruction copies four whole
    // 128-byte rows of an A box (lane l: row 4i + l/8, 16-byte chunk l%8,
    // placed at its 128-byte swizzle position), and each lane arrives on the
    // stage's full barrier once its copies have landed (32 of its 33
    // arrivals; the copy warp arms it for the B tile). Rows past the group
    // end, and rows or columns outside the source, are zero-filled.
    if constexpr (NG > 0) {
      const int ng = min(NG, STAGES);
      const int g = warp - (2 + kEpiWarps);
      if (p.a_rows && !p.selftest && g < ng) {
        const int chunk = lane & 7;
        const size_t row_bytes = (size_t)p.a_src_cols * 2;
        const char* src_base = reinterpret_cast<const char*>(p.a_src);
        uint32_t it = 0;  // K blocks of this CTA so far
        bool stop = false;
        for (int ri = 0, tau = tile_of(0); tau < sc.total && !stop; tau = tile_of(++ri)) {
          const Tile t = decode<MODE>(sc, tau, rank);
          const int gend = t.row0 + (t.nkb - 1) * BK + t.valid;  // group end
          for (int kb = 0; kb < t.nkb; ++kb, ++it) {
            if ((int)(it % (uint32_t)ng) != g) continue;
            const uint32_t stage = it % (uint32_t)STAGES;
            const uint32_t phase = (it / (uint32_t)STAGES) & 1u;
            const int y = t.row0 + kb * BK;
            const int ia = p.a_rows[min(y + lane, gend - 1)];
            const int ib = p.a_rows[min(y + lane + 32, gend - 1)];
            if (!warp_wait(&empty[stage], phase ^ 1, abort_flag, p.err, p.wait_ns)) {
              stop = true;
              break;
            }
            uint8_t* a_s = stages + stage * STB;
#pragma unroll 4
            for (int i = 0; i < BK / 4; ++i) {
              const int r = 4 * i + (lane >> 3);  // row of the K block
              const int src = __shfl_sync(0xffffffffu, i < BK / 8 ? ia : ib, r & 31);
              const bool row_ok = y + r < gend && src >= 0 && src < p.a_src_rows;
#pragma unroll
              for (int box = 0; box < BM / 64; ++box) {
                const int col = t.cm0 + 64 * box + 8 * chunk;
                const bool ok = row_ok && col < p.a_src_cols;
                const char* gp = ok ? src_base + (size_t)src * row_bytes + (size_t)col * 2
                                    : src_base;
                cp_async16(a_s + box * BOX_BYTES + r * 128 + ((chunk ^ (r & 7)) << 4), gp, ok);
              }
            }
            cp_async_arrive(&full[stage]);
          }
        }
        cp_async_wait_all();
      }
    }
  } else {
    // ===================== epilogue (warps 2..9) =====================
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row_local = q * 32 + lane;
    const int c_lo = ((warp - 2) >> 2) * (BN / 2), c_hi = c_lo + BN / 2;  // its columns
    const int nbuf = p.stage_bufs;
    uint8_t* wst = staging + (warp - 2) * nbuf * STAGING_BYTES;
    int buf = 0;
    const int ncols = MODE == kG3 ? 2 * p.H : p.D;  // output width (G2, G3, G4)
    const int row_lim = MODE == kG2 ? p.H : p.D;    // output rows (G2, G3)
    uint32_t acc = 0, acc_phase = 0;
    // accumulator-empty barrier: the even CTA's, reached remotely from the odd one
    const uint32_t tempty_cl0 = PAIR ? mapa(&tempty[0], 0) : 0u;
    const uint32_t tempty_cl1 = PAIR ? mapa(&tempty[1], 0) : 0u;

    // stage 32 accumulator columns of this warp's 32 rows and store them
    auto staged_store = [&](const uint32_t (&r)[32], const Tile& t, int col) {
      if (lane == 0) bulk_wait_read(nbuf - 1);
      __syncwarp();
      uint8_t* blk = wst + buf * STAGING_BYTES;
      stage_row(blk, lane, r);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        if constexpr (MODE == kG2) {
          tma_store_3d(&maps.o1, blk, col, t.cm0 + q * 32, t.e);
        } else if constexpr (MODE == kG3) {
          if (col < p.H)
            tma_store_3d(&maps.o1, blk, col, t.cm0 + q * 32, t.e);
          else
            tma_store_3d(&maps.o2, blk, col - p.H, t.cm0 + q * 32, t.e);
        } else {
          tma_store_2d(&maps.o1, blk, col, t.cm0 + q * 32);
        }
        bulk_commit();
      }
      if (++buf == nbuf) buf = 0;
    };

    for (int ri = 0, tau = tile_of(0); tau < sc.total; tau = tile_of(++ri)) {
      const Tile t0 = decode<MODE>(sc, tau, rank);
      if (t0.nkb <= 0) {
        // expert without retained rows: its weight gradient is zero
        if constexpr (WG) {
          const Tile& t = t0;
          if (t.cm0 + q * 32 < row_lim) {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
            for (int c = c_lo; c < c_hi; c += 32)
              if (t.n0 + c < ncols) staged_store(z, t, t.n0 + c);
          }
        }
        continue;
      }
      bool quit = false;
      // one accumulator per 256 columns: a wide tile's second one holds
      // columns n0 + 256 ...
      for (int half = 0; half < (WIDE ? 2 : 1); ++half) {
        Tile t = decode<MODE>(sc, tau, rank);  // (decoded again: keeps t0 out of registers)
        t.n0 += half * BN;
        if (!warp_wait(&tfull[acc], acc_phase, abort_flag, p.err, p.wait_ns)) {
          quit = true;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
        if constexpr (MODE == kG1) {
          bool rv = row_local < t.cvalid;
          const int64_t j = (int64_t)t.cm0 + row_local;
          int64_t src = j;  // row of the saved [a | b]
          if (p.ab_rows && rv) {
            src = p.ab_rows[j];
            if (src < 0 || src >= p.ab_src_rows) {
              flag_error(p.err, LRM_DEVERR_INDEX);
              rv = false;
            }
          }
          const __nv_bfloat16* arow = p.ab_c + src * 2 * p.H;
          __nv_bfloat16* drow = p.dab_c + j * 2 * p.H;
          const bool g1_whole = q * 32 + 32 <= t.cvalid;  // warp-uniform
          uint4 a_cur[4], b_cur[4], a_nxt[4], b_nxt[4];
          auto load_ab = [&](int h, uint4 (&av)[4], uint4 (&bv)[4]) {
            if (rv && h < p.H) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                // read-only path: a row's four 16-byte pieces share its L1 lines
                av[v] = __ldg(reinterpret_cast<const uint4*>(arow + h + 8 * v));
                bv[v] = __ldg(reinterpret_cast<const uint4*>(arow + p.H + h + 8 * v));
              }
            }
          };
          load_ab(t.n0 + c_lo, a_cur, b_cur);
#pragma unroll
          for (int c = c_lo; c < c_hi; c += 32) {
            uint32_t r[32];
            tmem_ld32(taddr + c, r);
            if (c + 32 < c_hi) load_ab(t.n0 + c + 32, a_nxt, b_nxt);
            tmem_ld_wait();
            const int h = t.n0 + c;
            if (g1_whole && h < p.H) {
              // the warp's 32 rows lie inside the group: stage the da and db
              // blocks (32 rows x 64 B each, 64-byte swizzle) and write them
              // with two TMA bulk-tensor stores
              uint4 dav[4], dbv[4];
              swiglu_chunk(r, a_cur, b_cur, dav, dbv);
              if (!rv) {
#pragma unroll
                for (int v = 0; v < 4; ++v) dav[v] = dbv[v] = make_uint4(0, 0, 0, 0);
              }
              if (lane == 0) bulk_wait_read(0);
              __syncwarp();
              const int sw = (lane >> 1) & 3;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                *reinterpret_cast<uint4*>(wst + lane * 64 + ((v ^ sw) << 4)) = dav[v];
                *reinterpret_cast<uint4*>(wst + 2048 + lane * 64 + ((v ^ sw) << 4)) = dbv[v];
              }
              fence_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&maps.o1, wst, h, t.cm0 + q * 32);
                tma_store_2d(&maps.o1, wst + 2048, p.H + h, t.cm0 + q * 32);
                bulk_commit();
              }
            } else if (rv && h < p.H) {  // block crossing the group end: row by row
              uint4 dav[4], dbv[4];
              swiglu_chunk(r, a_cur, b_cur, dav, dbv);
              uint4* da_dst = reinterpret_cast<uint4*>(drow + h);
              uint4* db_dst = reinterpret_cast<uint4*>(drow + p.H + h);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                da_dst[v] = dav[v];
                db_dst[v] = dbv[v];
              }
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              a_cur[v] = a_nxt[v];
              b_cur[v] = b_nxt[v];
            }
          }
        } else if constexpr (MODE == kF1) {
          // this warp's 64 gate columns and the matching 64 up columns
          const bool rv = row_local < t.cvalid;
          const int64_t j = (int64_t)t.cm0 + row_local;
          const int hbase = ((warp - 2) >> 2) * (BN / 4);
          // the warp's 32 rows inside the group (warp-uniform): a, b and phi go
          // out as 32 x 32 blocks (64-byte swizzle) through TMA stores
          const bool whole = LRM_TC_FWD_STAGED && q * 32 + 32 <= t.cvalid;
#pragma unroll 1
          for (int cc = 0; cc < BN / 4; cc += 32) {
            const int hl = hbase + cc;
            uint32_t ra[32], rb[32];
            tmem_ld32(taddr + hl, ra);
            tmem_ld32(taddr + BN / 2 + hl, rb);
            tmem_ld_wait();
            const int h = t.n0 / 2 + hl;
            if (whole && h < p.H) {
              uint4 av[4], bv[4], fv[4];
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float a[8], b[8], f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  a[u] = __uint_as_float(ra[8 * v + u]);
                  b[u] = __uint_as_float(rb[8 * v + u]);
                  f[u] = a[u] * __fdividef(1.0f, 1.0f + __expf(-a[u])) * b[u];
                }
                av[v] = Vec16<__nv_bfloat16>::pack(a);
                bv[v] = Vec16<__nv_bfloat16>::pack(b);
                fv[v] = Vec16<__nv_bfloat16>::pack(f);
              }
              // one set of blocks per warp: a second set costs a ring stage
              // and measured slower
              uint8_t* sb = wst;
              if (lane == 0) bulk_wait_read(0);
              __syncwarp();
              const int sw = (lane >> 1) & 3;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                *reinterpret_cast<uint4*>(sb + lane * 64 + ((v ^ sw) << 4)) = av[v];
                *reinterpret_cast<uint4*>(sb + 2048 + lane * 64 + ((v ^ sw) << 4)) = bv[v];
                if (p.ob1)
                  *reinterpret_cast<uint4*>(sb + 4096 + lane * 64 + ((v ^ sw) << 4)) = fv[v];
              }
              fence_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&maps.o1, sb, h, t.cm0 + q * 32);
                tma_store_2d(&maps.o1, sb + 2048, p.H + h, t.cm0 + q * 32);
                if (p.ob1) tma_store_2d(&maps.o2, sb + 4096, h, t.cm0 + q * 32);
                bulk_commit();
              }
            } else if (rv && h < p.H) {
              __nv_bfloat16* arow = p.ob0 + j * 2 * p.H;
              uint4* a_dst = reinterpret_cast<uint4*>(arow + h);
              uint4* b_dst = reinterpret_cast<uint4*>(arow + p.H + h);
              uint4* f_dst = p.ob1 ? reinterpret_cast<uint4*>(p.ob1 + j * p.H + h) : nullptr;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float a[8], b[8], f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  a[u] = __uint_as_float(ra[8 * v + u]);
                  b[u] = __uint_as_float(rb[8 * v + u]);
                  f[u] = a[u] * __fdividef(1.0f, 1.0f + __expf(-a[u])) * b[u];
                }
                a_dst[v] = Vec16<__nv_bfloat16>::pack(a);
                b_dst[v] = Vec16<__nv_bfloat16>::pack(b);
                if (f_dst) f_dst[v] = Vec16<__nv_bfloat16>::pack(f);
              }
            }
          }
        } else if constexpr (MODE == kF2) {
          const bool rv = row_local < t.cvalid;
          const int64_t j = (int64_t)t.cm0 + row_local;
          const bool whole = LRM_TC_FWD_STAGED && q * 32 + 32 <= t.cvalid;  // as in F1
#pragma unroll 1
          for (int c = c_lo; c < c_hi; c += 32) {
            uint32_t r[32];
            tmem_ld32(taddr + c, r);
            tmem_ld_wait();
            const int col = t.n0 + c;
            if (whole && col < p.D) {
              uint4 yv[4];
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] = __uint_as_float(r[8 * v + u]);
                yv[v] = Vec16<__nv_bfloat16>::pack(f);
              }
              // one y block per warp: a second one in turn measured slower
              uint8_t* yb = wst;
              if (lane == 0) bulk_wait_read(0);
              __syncwarp();
              const int sw = (lane >> 1) & 3;
#pragma unroll
              for (int v = 0; v < 4; ++v)
                *reinterpret_cast<uint4*>(yb + lane * 64 + ((v ^ sw) << 4)) = yv[v];
              fence_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&maps.o1, yb, col, t.cm0 + q * 32);
                bulk_commit();
              }
            } else if (rv && col < p.D) {
              uint4* dst = reinterpret_cast<uint4*>(p.ob0 + j * p.D + col);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] = __uint_as_float(r[8 * v + u]);
                dst[v] = Vec16<__nv_bfloat16>::pack(f);
              }
            }
          }
        } else {
          const bool rows_in = WG ? (t.cm0 + q * 32 < row_lim) : (q * 32 < t.cvalid);
          const bool whole = WG || (q * 32 + 32 <= t.cvalid);  // G4: block inside the group
#pragma unroll 1
          for (int c = c_lo; c < c_hi; c += 32) {
            uint32_t r[32];
            tmem_ld32(taddr + c, r);
            tmem_ld_wait();
            const int col = t.n0 + c;
            if (!rows_in || col >= ncols) continue;
            if (whole) {
              staged_store(r, t, col);
            } else if (row_local < t.cvalid) {  // G4 block crossing the group end
              store_f32x32(p.out0 + (int64_t)(t.cm0 + row_local) * p.D + col, r);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && !leader) mbar_arrive_cluster(acc ? tempty_cl1 : tempty_cl0);
          else mbar_arrive(&tempty[acc]);
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (quit) break;
    }
    if (lane == 0) bulk_wait_all();  // staged stores done before smem goes away
    __syncwarp();
  }

  if (PAIR && *abort_flag) {
    // an aborted pair may leave copies of the odd CTA in flight that only the
    // even CTA's barriers count: give them time to land before smem is freed
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 100000ull) {
    }
  }
  __syncwarp();
  tc_fence_before();
  if constexpr (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// Row-major [rows, cols] (rank 2) or [E, rows, cols] (rank 3) map with a
// 128-byte swizzle; bf16 operands or fp32 outputs.
static bool make_map(CUtensorMap* m, const void* base, bool fp32, int rank, uint64_t E,
                     uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
                     int swizzle_bytes = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[3] = {cols, rows, E};
  cuuint64_t strides[2] = {cols * es, rows * cols * es};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows, cols] bf16 matrix (cols a multiple of 64) seen as 3-D
// {64 columns, rows, cols / 64 chunks}: a box of 64 rows by `chunks` chunks
// lands in shared memory as `chunks` consecutive 64 x 64 blocks (128-byte
// swizzle), the layout of that many separate 64 x 64 boxes.
static bool make_chunked_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                             uint32_t chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || cols % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, 64, chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kSmemLimit = 232448;  // 227 KB per block

static size_t smem_bytes(int E, int stages, uint32_t stage_bytes, int stage_bufs) {
  return 1024 + (size_t)stages * stage_bytes + (size_t)kEpiWarps * stage_bufs * STAGING_BYTES +
         8 * (2 * MAX_STAGES + 5 + 2 * kTQ) + 16 + (size_t)(2 * (E + 1) + 2 + kTQ) * 4;
}

// Staging blocks per epilogue warp for fp32 outputs (two keep twice the store
// bytes in flight at the cost of ring depth).
#ifndef LRM_TC_STAGE_BUFS
#define LRM_TC_STAGE_BUFS 1
#endif
// the same for the weight-gradient products, whose epilogue stores bound them
#ifndef LRM_TC_WG_STAGE_BUFS
#define LRM_TC_WG_STAGE_BUFS 1
#endif

template <int MODE, bool PAIR, bool W = false>
static lrm_status launch_mode(const Maps& maps, Params p, int64_t tiles, cudaStream_t cs) {
  constexpr uint32_t STB = Ring<MODE, PAIR, W>::kStageBytes;
  // forward: a, b and phi blocks (F1) or y blocks (F2) for the staged stores
  p.stage_bufs = Geo<MODE>::kFwd ? (LRM_TC_FWD_STAGED ? (MODE == kF1 ? 2 : 1) : 0)
                 : Geo<MODE>::kWgrad                ? LRM_TC_WG_STAGE_BUFS
                                                    : LRM_TC_STAGE_BUFS;
  p.stages = MAX_STAGES;
  while (p.stages > 2 && smem_bytes(p.E, p.stages, STB, p.stage_bufs) > kSmemLimit) --p.stages;
  const size_t smem = smem_bytes(p.E, p.stages, STB, p.stage_bufs);
  if (smem > kSmemLimit) return LRM_ERR_UNSUPPORTED;
  auto kern = grouped_gemm_kernel<MODE, PAIR, W>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return LRM_ERR_CUDA;
  const int sms = num_sms();
  const int per_unit = PAIR ? 2 : 1;
  const int64_t units = std::max<int64_t>(1, std::min<int64_t>(tiles, sms / per_unit));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * per_unit), 1, 1);
  cfg.blockDim = dim3(Threads<MODE, PAIR>::kCount, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = cs;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (LRM_PDL) {  // see launch_k: the kernel starts with pdl_begin()
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, maps, p) != cudaSuccess) return LRM_ERR_CUDA;
  return launch_status();
}

// Which products run on CTA pairs (bit per mode, G1 = 1 ... G4 = 8, F1 = 16,
// F2 = 32). Pairs pay off where the weights are the B operand (G1, G4: +1-4%
// on the large layers; F1, F2 likewise read each weight tile once per 256
// rows); the weight-gradient products measured as fast or faster on single
// CTAs.
#ifndef LRM_TC_PAIR_MODES
#define LRM_TC_PAIR_MODES 57
#endif

template <int MODE>
static lrm_status launch_any(const Maps& single, const Maps& pair, const Params& p,
                             int64_t tiles_single, int64_t tiles_pair, cudaStream_t cs) {
  if constexpr (((LRM_TC_PAIR_MODES >> MODE) & 1) != 0)
    return launch_mode<MODE, true>(pair, p, tiles_pair, cs);
  else
    return launch_mode<MODE, false>(single, p, tiles_single, cs);
}

// FC1 dgrad runs on wide tiles when its K extent (2H) spans at least this many
// 64-deep blocks: measured 2-4% faster at 2H = 2,816 (44 blocks), 2-3% slower
// at 2H = 1,536 (24 blocks), where the exposed epilogue weighs more. (FC2
// dgrad, whose epilogue also reads the saved [a | b] rows, measured 10-40%
// slower on wide tiles.)
constexpr int kWideMinKBlocks = 32;
static bool wide_fc1_dgrad(int H) {
  return ((LRM_TC_PAIR_MODES >> kG4) & 1) != 0 && 2 * H / BK >= kWideMinKBlocks;
}

// Weight-gradient products with gathered A rows run on single CTAs (the
// gather producer is written for one CTA per tile).
template <int MODE>
static lrm_status launch_gather_or_any(const Maps& m, const Maps& mp, const Params& p,
                                       int64_t tiles_single, int64_t tiles_pair,
                                       cudaStream_t cs) {
  if (p.a_rows) return launch_mode<MODE, false>(m, p, tiles_single, cs);
  return launch_any<MODE>(m, mp, p, tiles_single, tiles_pair, cs);
}

}  // namespace tc

lrm_status launch_bwd_tc(const BwdArgs& a, unsigned parts) {
  using namespace tc;
  const lrm_shape* s = a.s;
  const int D = s->D, H = s->H, E = s->E;
  if (D % 64 != 0 || H % 64 != 0) return LRM_ERR_UNSUPPORTED;
  const uint64_t N = (uint64_t)s->T * s->K;
  const uint64_t rows = std::max<uint64_t>(N, 1);

  Params p;
  p.wait_ns = kWaitNs;
  p.selftest = 0;
  p.E = E;
  p.D = D;
  p.H = H;
  p.n_rows = (int)N;
  p.stage_bufs = 0;
  p.stages = 4;
  p.sel_off = a.sel_off;
  p.ab_c = reinterpret_cast<const __nv_bfloat16*>(a.ab_c);
  p.dab_c = reinterpret_cast<__nv_bfloat16*>(a.dab_c);
  p.out0 = nullptr;
  p.out1 = nullptr;
  p.ob0 = nullptr;
  p.ob1 = nullptr;
  p.ab_rows = nullptr;
  p.a_rows = nullptr;
  p.a_src = nullptr;
  p.a_src_rows = p.a_src_cols = 0;
  p.ab_src_rows = (int)N;
  p.err = a.err;
  p.queue = queue_words(a.err);
  lrm_status st = LRM_OK;
  const bool gathered = a.sel_pos != nullptr;
  if (gathered && !a.tok_c) return LRM_ERR_INVALID_ARG;
  const uint64_t tok_rows = std::max<uint64_t>(s->T, 1);
  // upper bounds of the tile counts (the exact ones depend on device-side sizes)
  auto dg_tiles = [&](int tm, int ncols) {
    return ((int64_t)N / tm + E) * ((ncols + BN - 1) / BN);
  };
  auto wg_tiles = [&](int tm, int mrows, int ncols) {
    return (int64_t)E * ((mrows + tm - 1) / tm) * ((ncols + BN - 1) / BN);
  };
  // K-major operands (data-gradient products): 64 x 128 A boxes and 64 x 256
  // (single CTA) or 64 x 128 (pair) weight boxes, one expert per 3-D slice;
  // MN-major operands (weight-gradient products): 64 rows by 2 or 4 chunks of
  // 64 columns per copy; fp32 outputs: 32 x 32 boxes.
  if (parts & kPartFc2Dgrad) {
    Maps m1, m2;
    if (!make_map(&m1.a, a.dy_c, false, 2, 1, rows, D, 64, BM) ||
        !make_map(&m1.b, a.w_down, false, 3, E, H, D, 64, BN) ||
        !make_map(&m2.b, a.w_down, false, 3, E, H, D, 64, BN / 2))
      return LRM_ERR_CUDA;
    // dab_c as 32 x 32 bf16 blocks (64-byte rows, 64-byte swizzle) for the
    // epilogue's staged stores
    if (!make_map(&m1.o1, a.dab_c, false, 2, 1, rows, 2 * H, 32, 32, 64)) return LRM_ERR_CUDA;
    m2.a = m1.a;
    m1.b2 = m1.o2 = m1.b;
    m2.b2 = m2.o2 = m2.b;
    m2.o1 = m1.o1;
    p.ab_rows = gathered ? a.sel_pos : nullptr;
    if ((st = launch_any<kG1>(m1, m2, p, dg_tiles(BM, H), dg_tiles(2 * BM, H), a.stream)) !=
        LRM_OK)
      return st;
    p.ab_rows = nullptr;
  }
  if (parts & kPartFc2Wgrad) {
    Maps m, mp;  // single CTAs (B: 256 columns) and CTA pairs (B: 128 per CTA)
    if (!make_map(&m.o1, a.dw_down, true, 3, E, H, D, 32, 32) ||
        !make_chunked_map(&m.a, a.phi_c, rows, H, BM / 64) ||
        !make_chunked_map(&m.b, a.dy_c, rows, D, BN / 64) ||
        !make_chunked_map(&mp.b, a.dy_c, rows, D, BN / 128))
      return LRM_ERR_CUDA;
    m.b2 = m.b;
    m.o2 = m.o1;
    mp.a = m.a;
    mp.b2 = mp.b;
    mp.o1 = mp.o2 = m.o1;
    p.out0 = a.dw_down;
    p.a_rows = gathered ? a.sel_pos : nullptr;
    p.a_src = reinterpret_cast<const __nv_bfloat16*>(a.phi_c);
    p.a_src_rows = (int)N;
    p.a_src_cols = H;
    if ((st = launch_gather_or_any<kG2>(m, mp, p, wg_tiles(BM, H, D), wg_tiles(2 * BM, H, D),
                                        a.stream)) != LRM_OK)
      return st;
    p.a_rows = nullptr;
  }
  if (parts & kPartFc1Wgrad) {
    Maps m, mp;  // single CTAs (B: 256 columns) and CTA pairs (B: 128 per CTA)
    if (!make_map(&m.o1, a.dw_gate, true, 3, E, D, H, 32, 32) ||
        !make_map(&m.o2, a.dw_up, true, 3, E, D, H, 32, 32) ||
        !make_chunked_map(&m.a, a.x_c, gathered ? tok_rows : rows, D, BM / 64) ||
        !make_chunked_map(&m.b, a.dab_c, rows, 2 * H, BN / 64) ||
        !make_chunked_map(&mp.b, a.dab_c, rows, 2 * H, BN / 128))
      return LRM_ERR_CUDA;
    m.b2 = m.b;
    mp.a = m.a;
    mp.b2 = mp.b;
    mp.o1 = m.o1;
    mp.o2 = m.o2;
    p.out0 = a.dw_gate;
    p.out1 = a.dw_up;
    p.a_rows = gathered ? a.tok_c : nullptr;
    p.a_src = reinterpret_cast<const __nv_bfloat16*>(a.x_c);
    p.a_src_rows = s->T;
    p.a_src_cols = D;
    if ((st = launch_gather_or_any<kG3>(m, mp, p, wg_tiles(BM, D, 2 * H),
                                        wg_tiles(2 * BM, D, 2 * H), a.stream)) != LRM_OK)
      return st;
    p.a_rows = nullptr;
  }
  if (parts & kPartFc1Dgrad) {
    Maps m1, m2;
    if (!make_map(&m1.a, a.dab_c, false, 2, 1, rows, 2 * H, 64, BM) ||
        !make_map(&m1.b, a.w_gate, false, 3, E, D, H, 64, BN) ||
        !make_map(&m1.b2, a.w_up, false, 3, E, D, H, 64, BN) ||
        !make_map(&m2.b, a.w_gate, false, 3, E, D, H, 64, BN / 2) ||
        !make_map(&m2.b2, a.w_up, false, 3, E, D, H, 64, BN / 2) ||
        !make_map(&m1.o1, a.dx_c, true, 2, 1, rows, D, 32, 32))
      return LRM_ERR_CUDA;
    m2.a = m1.a;
    m1.o2 = m1.o1;
    m2.o1 = m2.o2 = m1.o1;
    p.out0 = a.dx_c;
    p.out1 = nullptr;
    st = wide_fc1_dgrad(H)
             ? launch_mode<kG4, true, true>(m2, p, dg_tiles(2 * BM, D), a.stream)
             : launch_any<kG4>(m1, m2, p, dg_tiles(BM, D), dg_tiles(2 * BM, D), a.stream);
    if (st != LRM_OK) return st;
  }
  return st;
}

lrm_status launch_fwd_tc(const FwdArgs& a, unsigned parts) {
  using namespace tc;
  const lrm_shape* s = a.s;
  const int D = s->D, H = s->H, E = s->E;
  if (D % 64 != 0 || H % 64 != 0) return LRM_ERR_UNSUPPORTED;
  const uint64_t N = (uint64_t)s->T * s->K;
  const uint64_t rows = std::max<uint64_t>(N, 1);
  Params p = {};
  p.wait_ns = kWaitNs;
  p.E = E;
  p.D = D;
  p.H = H;
  p.n_rows = (int)N;
  p.sel_off = a.off;
  p.err = a.err;
  p.queue = queue_words(a.err);
  lrm_status st = LRM_OK;
  // upper bound of the tile count: every group may end in a partial tile
  auto tiles = [&](int tm, int ntn) { return ((int64_t)N / tm + E) * ntn; };
  // K-major activations (64 x 128 boxes) against the weights in their stored
  // layout, read as MN-major 64 x 64 boxes, one expert per 3-D slice
  if (parts & kPartFc1Fwd) {
    Maps m;
    if (!make_map(&m.a, a.x_disp, false, 2, 1, rows, D, 64, BM) ||
        !make_map(&m.b, a.w_gate, false, 3, E, D, H, 64, 64) ||
        !make_map(&m.b2, a.w_up, false, 3, E, D, H, 64, 64))
      return LRM_ERR_CUDA;
    // ab and phi as 32 x 32 bf16 blocks (64-byte rows, 64-byte swizzle)
    if (!make_map(&m.o1, a.ab, false, 2, 1, rows, 2 * H, 32, 32, 64)) return LRM_ERR_CUDA;
    m.o2 = m.o1;
    if (a.phi && !make_map(&m.o2, a.phi, false, 2, 1, rows, H, 32, 32, 64)) return LRM_ERR_CUDA;
    p.ob0 = reinterpret_cast<__nv_bfloat16*>(a.ab);
    p.ob1 = reinterpret_cast<__nv_bfloat16*>(a.phi);
    const int ntn = (H + BN / 2 - 1) / (BN / 2);
    if ((st = launch_any<kF1>(m, m, p, tiles(BM, ntn), tiles(2 * BM, ntn), a.stream)) != LRM_OK)
      return st;
  }
  if (parts & kPartFc2Fwd) {
    Maps m;
    if (!make_map(&m.a, a.phi, false, 2, 1, rows, H, 64, BM) ||
        !make_map(&m.b, a.w_down, false, 3, E, H, D, 64, 64))
      return LRM_ERR_CUDA;
    m.b2 = m.b;
    if (!make_map(&m.o1, a.y, false, 2, 1, rows, D, 32, 32, 64)) return LRM_ERR_CUDA;
    m.o2 = m.o1;
    p.ob0 = reinterpret_cast<__nv_bfloat16*>(a.y);
    p.ob1 = nullptr;
    const int ntn = (D + BN - 1) / BN;
    if ((st = launch_any<kF2>(m, m, p, tiles(BM, ntn), tiles(2 * BM, ntn), a.stream)) != LRM_OK)
      return st;
  }
  return st;
}

__global__ void selftest_init_kernel(int32_t* err, int32_t* sel_off) {
  *err = 0;
  sel_off[0] = 0;
  sel_off[1] = 64;
}

// One grouped-GEMM CTA (FC1 dgrad, 1 expert, D = H = 64, 64 rows) whose copy
// warp delivers nothing: the MMA warp's wait for its first operand stage must
// give up after 20 ms, flag LRM_DEVERR_TIMEOUT, and the CTA must release its
// tensor memory and return. Only the workspace header is touched.
lrm_status selftest_wait_timeout(void* ws, size_t ws_bytes, cudaStream_t cs) {
  using namespace tc;
  if (!ws || ws_bytes < kWsHeaderBytes) return LRM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LRM_ERR_UNSUPPORTED;
  int32_t* err = error_word(ws);
  int32_t* sel_off = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + 64);
  selftest_init_kernel<<<1, 1, 0, cs>>>(err, sel_off);
  Params p = {};
  p.wait_ns = 20000000ull;
  p.selftest = 1;
  p.E = 1;
  p.D = 64;
  p.H = 64;
  p.n_rows = 64;
  p.sel_off = sel_off;
  p.err = err;
  Maps m;
  memset(&m, 0, sizeof(m));
  return launch_mode<kG4, false>(m, p, 1, cs);
}

}  // namespace lrm
