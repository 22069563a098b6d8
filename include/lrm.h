/*
 * lrm.h -- C ABI of the recalibrated MoE expert backward on one GB300 GPU.
 *
 * The path follows "LRMoE: Demand-Side Load Re-Calibration for Efficient MoE
 * Training on Memory-Constrained Nodes" (arXiv 2610.37720) on a single GPU:
 *   forward dispatch permutation -> LRM score of every routed pair ->
 *   per-expert top-q selection -> physical compaction -> SwiGLU expert
 *   backward as variable-size grouped GEMMs over the retained rows only.
 * Multi-GPU routing, replicas, all-to-all and the CPU offload queue of the
 * paper are not part of this library.
 *
 * Notation: T tokens, D model dim, H expert FFN dim, E experts, K routed
 * experts per token, N = T*K routed pairs; pair index p = t*K + k.
 * "Dispatch order" lists the pairs grouped by expert (expert-major), inside a
 * group by ascending p.
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated; the
 *    library never allocates or frees memory and keeps no global state
 *    (calls on different streams are independent).
 *  - All calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = legacy default stream) and never synchronise the host, except
 *    lrm_get_device_error.
 *  - Row-major contiguous layouts. Floating-point activations and weights
 *    (x, g, ab, phi, W_*, dy_c, x_c, ab_c, phi_c, dab_c) have the element type
 *    of lrm_shape.dtype (LRM_BF16: bfloat16, LRM_F32: float); routing weights,
 *    scores and all gradients in float32; indices int32.
 *  - Every pointer must be 16-byte aligned and D, H multiples of 8, else
 *    LRM_ERR_UNSUPPORTED. The BF16 grouped backward also needs D and H to be
 *    multiples of 64.
 *  - Argument errors are returned before anything is launched. A failed
 *    launch returns LRM_ERR_CUDA. Bad DATA found on the device (an expert id
 *    outside [0, E), a quota outside [0, n_e], an index out of range, a
 *    pipeline wait that timed out) never traps: the kernel clamps or skips,
 *    ORs an LRM_DEVERR_* bit into the device error word kept in the first 4
 *    bytes of the caller's workspace, and the call returns LRM_OK; read the
 *    word with lrm_get_device_error.
 *  - ws / ws_bytes: caller-owned device workspace of at least
 *    lrm_workspace_bytes(shape) bytes, 256-byte aligned. Its first 256 bytes
 *    are a header: the device error word and the tile-queue counters of the
 *    weight-gradient products, which every such launch leaves at zero for
 *    the next one. Zero the header once with lrm_clear_device_error before
 *    first use, and let one workspace serve one stream at a time (two
 *    weight-gradient launches in flight together would share the queue).
 */
#ifndef LRM_H_
#define LRM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lrm_status {
  LRM_OK = 0,
  LRM_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size */
  LRM_ERR_UNSUPPORTED = 2, /* alignment / dimension not supported */
  LRM_ERR_WORKSPACE = 3,   /* workspace missing or too small */
  LRM_ERR_CUDA = 4         /* a CUDA launch or runtime call failed */
} lrm_status;

typedef enum lrm_dtype { LRM_F32 = 0, LRM_BF16 = 1 } lrm_dtype;

/* Layer shape. dtype is an lrm_dtype. N = T*K must be < 2^31. */
typedef struct lrm_shape {
  int32_t T, D, H, E, K;
  int32_t dtype;
} lrm_shape;

/* Bits of the device error word. */
#define LRM_DEVERR_EXPERT_ID 1 /* topk_idx outside [0,E): clamped          */
#define LRM_DEVERR_QUOTA 2     /* quota outside [0,n_e]: clamped           */
#define LRM_DEVERR_INDEX 4     /* inv / perm / sel_pos out of range: row skipped */
#define LRM_DEVERR_TIMEOUT 8   /* a GEMM pipeline wait gave up: outputs invalid */
#define LRM_DEVERR_QUEUE 16    /* a weight-gradient tile queue did not hand out
                                  every tile once (header not zeroed before first
                                  use, or shared by concurrent launches): outputs
                                  invalid; the queue is rewound for the next call */

/* Bytes of workspace every call of this shape needs (host only, pure). */
size_t lrm_workspace_bytes(const lrm_shape* shape);

/* Zero the workspace header (the device error word in its first 4 bytes and
 * the tile-queue counters). Async on stream. */
lrm_status lrm_clear_device_error(void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream`, then copy the device error word into *code_out. */
lrm_status lrm_get_device_error(const void* ws, size_t ws_bytes,
                                int32_t* code_out, void* stream);

/* Human-readable name of a status code (static string). */
const char* lrm_status_string(lrm_status status);

/*
 * Forward dispatch permutation: a stable counting sort of the pairs by
 * expert id. "Least-Loaded Expert Parallelism" (LLEP) Sec. 2.1 re-index
 * (tokens [a,b,c,d] routed to experts [2,6,2,1] become [d,a,c,b]) and LLEP
 * Alg. 4 sort of the flattened indices; LRMoE Alg. 1 forward admission
 * counts N_e = |P_e|.
 *   topk_idx [T,K] int32 : expert of pair p = t*K+k (read).
 *   perm     [N]   int32 : perm[pos] = p, dispatch position -> pair (written).
 *   inv      [N]   int32 : inv[p] = pos (written).
 *   counts   [E]   int32 : n_e (written).
 *   off      [E+1] int32 : exclusive prefix of counts, off[E] = N (written).
 * Ids outside [0,E) are clamped into range and flag LRM_DEVERR_EXPERT_ID.
 */
lrm_status lrm_dispatch_permute(const lrm_shape* shape, const int32_t* topk_idx,
                                int32_t* perm, int32_t* inv, int32_t* counts,
                                int32_t* off, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * Row re-index into dispatch order, dst[pos] = src[perm[pos]] for
 * pos < n_rows (LLEP Sec. 2.1: B' is B with its rows taken in dispatch
 * order). row_bytes must be a positive multiple of 16; src and dst must not
 * overlap. Rows whose perm entry is outside [0, n_rows) are left untouched.
 */
lrm_status lrm_permute_rows(const int32_t* perm, int32_t n_rows, const void* src,
                            void* dst, int64_t row_bytes, void* stream);

/*
 * Per-expert retention quota q_e = min(ceil(num/den * n_e), cap), computed
 * in exact integer arithmetic; cap <= 0 means no cap. LRMoE Sec. 3.1: quotas
 * satisfy 0 <= K_e <= N_e with retention rate rho = sum_e K_e / N, fixed for
 * the invocation. Needs 0 <= num <= den, den > 0.
 *   counts [E] int32 (read), quota [E] int32 (written).
 */
lrm_status lrm_quota_from_rate(const int32_t* counts, int32_t E, int32_t num,
                               int32_t den, int32_t cap, int32_t* quota,
                               void* stream);

/*
 * Load Recalibration Metric of every routed pair, LRMoE Sec. 3.2 Prop. 3.1
 * Eq. 3 and Sec. 7.1 Eq. 12: R_u = alpha_u^2 * ||g_t||^2 * ||phi_u||^2, the
 * squared Frobenius norm of the pair's rank-one FC2 weight-gradient
 * contribution (alpha_u g_t) phi_u^T; g_t is the cotangent at the MoE output
 * before the routing weight (Sec. 7.1 Eq. 5). FP32 accumulation.
 *   g     [T,D] dtype          : output cotangent (read).
 *   phi   [N,H] dtype          : saved FC2 input, dispatch order (read).
 *   alpha [T,K] float          : routing weights (read).
 *   inv   [N]   int32          : from lrm_dispatch_permute (read).
 *   score [N]   float          : R in dispatch order (written).
 */
lrm_status lrm_score(const lrm_shape* shape, const void* g, const void* phi,
                     const float* alpha, const int32_t* inv, float* score,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * The selection criteria LRMoE Sec. 4.7 (Table 2) compares LRM against,
 * computed like lrm_score and written to score [N] in dispatch order:
 *   LRM_METRIC_LRM       alpha_u^2 ||g_t||^2 ||phi_u||^2   (= lrm_score)
 *   LRM_METRIC_GRAD_SQ   ||g_t||_2^2       squared gradient norm
 *   LRM_METRIC_GRAD_ABS  sum_d |g_t,d|     absolute gradient magnitude
 *   LRM_METRIC_RANDOM    output p+1 of SplitMix64 seeded with `seed`, top 24
 *                        bits as a float in [0,1): random selection
 * The gradient-only criteria read g only (alpha and phi may be NULL); the
 * random one reads neither (g may be NULL too). All are non-negative, so
 * lrm_select_quota applies to them unchanged.
 */
typedef enum lrm_metric {
  LRM_METRIC_LRM = 0,
  LRM_METRIC_GRAD_SQ = 1,
  LRM_METRIC_GRAD_ABS = 2,
  LRM_METRIC_RANDOM = 3
} lrm_metric;
lrm_status lrm_score_variant(const lrm_shape* shape, int32_t metric, uint64_t seed,
                             const void* g, const void* phi, const float* alpha,
                             const int32_t* inv, float* score, void* ws,
                             size_t ws_bytes, void* stream);

/*
 * Per-expert top-q selection, LRMoE Alg. 1 (TopK per expert) and Sec. 7.2
 * Prop. 7.1 (keeping the largest scores inside each expert is optimal for
 * fixed per-expert quotas). Inside each segment [off[e], off[e+1]) the q_e
 * largest scores are kept; equal scores are broken by the lower pair index,
 * which inside a segment is the lower dispatch position. Scores must be
 * non-negative and not NaN (they are sums of squares).
 *   score   [N]   float (read), off [E+1] int32 (read), quota [E] int32 (read).
 *   keep    [N]   uint8 : 1 if retained, dispatch order (written).
 *   sel_off [E+1] int32 : exclusive prefix of the quotas (written).
 *   sel_pos [N]   int32 : capacity N; the first M = sel_off[E] entries are
 *                         the retained dispatch positions, ascending inside
 *                         each expert (written).
 * Quotas outside [0, n_e] are clamped and flag LRM_DEVERR_QUOTA.
 */
lrm_status lrm_select_quota(const lrm_shape* shape, const float* score,
                            const int32_t* off, const int32_t* quota,
                            uint8_t* keep, int32_t* sel_off, int32_t* sel_pos,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * Physical compaction, LRMoE Sec. 3.1 (compact runtime) and Sec. 3.4 Fig. 4:
 * retained gradient rows and their saved state are gathered into contiguous
 * expert-major segments, with no zero-masked rows. For retained row
 * j < M = sel_off[E]: i = sel_pos[j], p = perm[i], t = p / K:
 *   dy_c[j]  = alpha[p] * g[t]   (product in float32, rounded once to dtype)
 *   x_c[j]   = x[t],  ab_c[j] = ab[i],  phi_c[j] = phi[i],  tok_c[j] = t
 *   row_of_pos[i] = j, and -1 at every position with keep[i] == 0.
 * Inputs: perm [N], keep [N], sel_off [E+1], sel_pos [N], alpha [T,K],
 *   x [T,D], g [T,D], ab [N,2H] (gate|up pre-activations, dispatch order),
 *   phi [N,H] (dispatch order).
 * Outputs (capacity N rows each, first M written): dy_c [N,D], x_c [N,D],
 *   ab_c [N,2H], phi_c [N,H], tok_c [N] int32; row_of_pos [N] int32.
 * Rows [M, min(M + 64, N)) of dy_c are written as zeros: the weight-gradient
 * products read them as padding past the last group.
 * x_c, ab_c and phi_c may each be NULL: that copy is skipped and its source
 * may be NULL too (see lrm_expert_fc1_recompute, which rebuilds [a | b], and
 * lrm_expert_bwd_gathered, which reads x, ab and phi rows in place). A
 * non-NULL destination with a NULL source is an error.
 * M is read from sel_off[E] on the device: a value outside [0, N] (sel_off
 * not produced by a selection call) is clamped into that range and flags
 * LRM_DEVERR_INDEX in the workspace error word; out-of-range sel_pos or perm
 * entries are skipped and flag the same bit.
 */
lrm_status lrm_compact(const lrm_shape* shape, const int32_t* perm,
                       const uint8_t* keep, const int32_t* sel_off,
                       const int32_t* sel_pos, const float* alpha, const void* x,
                       const void* g, const void* ab, const void* phi, void* dy_c,
                       void* x_c, void* ab_c, void* phi_c, int32_t* tok_c,
                       int32_t* row_of_pos, void* ws, size_t ws_bytes,
                       void* stream);

/*
 * SwiGLU expert backward over the retained rows, LRMoE Alg. 1
 * (PackedExpertBackward) and Sec. 3.4: four variable-size grouped products
 * per expert e over its m_e = sel_off[e+1] - sel_off[e] compacted rows J
 * (m_e is the row dimension of the data-gradient products and the reduction
 * dimension of the weight-gradient products; no padding):
 *   dphi       = dy_c[J] W_down[e]^T,  then the SwiGLU gradient
 *                da = dphi*b*s*(1 + a*(1-s)), db = dphi*a*s, s = sigmoid(a),
 *                (a, b) = ab_c[J] halves  -> dab_c[J] = [da | db]   (dtype)
 *   dW_down[e] = phi_c[J]^T dy_c[J]                               (H x D)
 *   dW_gate[e] = x_c[J]^T da,  dW_up[e] = x_c[J]^T db             (D x H)
 *   dx_c[J]    = da W_gate[e]^T + db W_up[e]^T                    (float32)
 * then the scatter back to tokens (Sec. 3.1: zero-initialised dense buffer):
 *   dx[t] = sum over kept slots k, ascending, of dx_c[row_of_pos[inv[t*K+k]]]
 * (deterministic, no atomics). BF16 runs on tcgen05 tensor cores with FP32
 * accumulation in tensor memory; F32 runs on CUDA cores.
 *   w_gate, w_up [E,D,H] dtype; w_down [E,H,D] dtype (read).
 *   dy_c, x_c [N,D]; ab_c [N,2H]; phi_c [N,H]  (read, first M rows used).
 *   inv [N], row_of_pos [N] int32 (read).
 *   dab_c [N,2H] dtype, dx_c [N,D] float : intermediates (first M rows written).
 *   dw_gate, dw_up [E,D,H] float; dw_down [E,H,D] float : OVERWRITTEN
 *     (zero for experts with no retained rows).
 *   dx [T,D] float : overwritten.
 * Pipeline waits are bounded; a timeout flags LRM_DEVERR_TIMEOUT.
 */
lrm_status lrm_expert_bwd_grouped(const lrm_shape* shape, const int32_t* sel_off,
                                  const void* w_gate, const void* w_up,
                                  const void* w_down, const void* dy_c,
                                  const void* x_c, const void* ab_c,
                                  const void* phi_c, const int32_t* inv,
                                  const int32_t* row_of_pos, void* dab_c,
                                  float* dx_c, float* dw_gate, float* dw_up,
                                  float* dw_down, float* dx, void* ws,
                                  size_t ws_bytes, void* stream);

/*
 * Self-test of the failure detection in the grouped GEMMs (no counterpart on
 * the pages). Every pipeline wait in those kernels is bounded; this launches
 * one grouped-GEMM CTA whose copy warp is told to deliver nothing, so the MMA
 * warp's wait for its first operand stage runs out after 20 ms. The CTA then
 * ORs LRM_DEVERR_TIMEOUT into the error word, frees its tensor memory and
 * returns; the CUDA context stays usable. It clears the error word first and
 * writes only the first 256 bytes of ws. Read the result with
 * lrm_get_device_error (expect LRM_DEVERR_TIMEOUT).
 */
lrm_status lrm_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/*
 * lrm_dispatch_permute for callers that cannot allocate device memory (the
 * paper has no counterpart; this is a deployment variant). Some callers are
 * handed only their input and output tensors, e.g. a plugin inside a host
 * whose memory manager owns the whole device budget; a cudaMalloc there
 * would bypass that accounting and can stall the whole device. This entry
 * point allocates nothing. Up to 2^17 routed pairs it runs the one-cluster
 * dispatch, which needs no scratch; above that, the per-chunk tables of the
 * three-launch dispatch live in one file-scope device array of
 * 2 * LRM_NOALLOC_MAX_CHUNK_ENTRIES int32 (512 KiB), which every GPU that
 * loads the library holds until the process exits.
 *  - Same outputs as lrm_dispatch_permute (bit for bit). dev_err may be
 *    NULL; otherwise LRM_DEVERR_EXPERT_ID is ORed into *dev_err (a 4-byte
 *    device word the caller clears).
 *  - Limit: E * ceil(T*K / 2048) <= LRM_NOALLOC_MAX_CHUNK_ENTRIES, else
 *    LRM_ERR_WORKSPACE is returned before anything is launched (the built-in
 *    scratch is too small; use lrm_dispatch_permute with a workspace).
 *  - The first call on each device that needs the array (more than 2^17
 *    pairs) looks up its device address with cudaGetSymbolAddress (once,
 *    with that device current); make that first call before any stream
 *    capture.
 *  - All calls share the one array: calls whose kernels overlap on the GPU
 *    (different streams, or several host threads) race and corrupt each
 *    other's results; serialise them. Every table entry a call reads is
 *    written earlier in the same call, so stale contents are harmless.
 */
#define LRM_NOALLOC_MAX_CHUNK_ENTRIES 65536
lrm_status lrm_dispatch_permute_noalloc(const lrm_shape* shape,
                                        const int32_t* topk_idx, int32_t* perm,
                                        int32_t* inv, int32_t* counts,
                                        int32_t* off, int32_t* dev_err,
                                        void* stream);

/*
 * The five sub-steps of lrm_expert_bwd_grouped as separate calls, same
 * arithmetic, arguments and layouts as documented there (LRMoE Sec. 3.4:
 * both layers' data- and weight-gradient products run over the retained
 * rows). Issue them in this order on one stream; each reads only
 * what the earlier ones wrote.
 *   lrm_expert_fc2_dgrad : dab_c = SwiGLU-grad(dy_c W_down[e]^T, ab_c); also
 *                          zeroes rows [M, min(M + 64, N)) of dab_c (padding
 *                          read by lrm_expert_fc1_wgrad past the last group)
 *   lrm_expert_fc2_wgrad : dW_down[e] = phi_c^T dy_c        (overwritten)
 *   lrm_expert_fc1_wgrad : dW_gate[e], dW_up[e] = x_c^T dab_c (overwritten)
 *   lrm_expert_fc1_dgrad : dx_c = dab_c [W_gate | W_up][e]^T
 *   lrm_scatter_dx       : dx[t] = sum of the token's kept dx_c rows
 */
lrm_status lrm_expert_fc2_dgrad(const lrm_shape* shape, const int32_t* sel_off,
                                const void* w_down, const void* dy_c,
                                const void* ab_c, void* dab_c, void* ws,
                                size_t ws_bytes, void* stream);
lrm_status lrm_expert_fc2_wgrad(const lrm_shape* shape, const int32_t* sel_off,
                                const void* phi_c, const void* dy_c,
                                float* dw_down, void* ws, size_t ws_bytes,
                                void* stream);
lrm_status lrm_expert_fc1_wgrad(const lrm_shape* shape, const int32_t* sel_off,
                                const void* x_c, const void* dab_c,
                                float* dw_gate, float* dw_up, void* ws,
                                size_t ws_bytes, void* stream);
lrm_status lrm_expert_fc1_dgrad(const lrm_shape* shape, const int32_t* sel_off,
                                const void* w_gate, const void* w_up,
                                const void* dab_c, float* dx_c, void* ws,
                                size_t ws_bytes, void* stream);
lrm_status lrm_scatter_dx(const lrm_shape* shape, const float* dx_c,
                          const int32_t* inv, const int32_t* row_of_pos,
                          float* dx, void* ws, size_t ws_bytes, void* stream);

/*
 * Forward expert pass: the pass that produces the saved state the backward
 * reads. LRMoE Sec. 3.1 (design overview) and Alg. 1
 * (FullForwardAndSaveContext): every routed pair runs through its expert,
 * the outputs are combined, and [a | b] and phi are kept per pair. LLEP
 * Sec. 2.1: token rows are re-indexed into per-expert groups (the
 * lrm_dispatch_permute order), one product per expert and group, and the
 * MoE output is the routing-weighted sum h_t = sum_k alpha_tk y_(t,k).
 * SwiGLU experts: a = x W_gate[e], b = x W_up[e], phi = SiLU(a) * b,
 * y = phi W_down[e]. FP32 accumulation; [a | b], phi and y are rounded once
 * to the layer dtype (phi from the unrounded a and b).
 * Groups come from `off` (lrm_dispatch_permute), read on the device; every
 * routed row is processed. BF16 layers need D and H multiples of 64.
 *
 * lrm_gather_tokens: x_disp[pos] = x[perm[pos] / K].
 *   perm [N] int32 (read); x [T,D] dtype (read); x_disp [N,D] dtype (written).
 *   perm entries outside [0,N) skip the row and flag LRM_DEVERR_INDEX.
 * lrm_expert_fc1_fwd: ab [N,2H] = [a | b] and phi [N,H] (dtype, written)
 *   from x_disp [N,D] and W_gate, W_up [E,D,H] (dtype, read).
 * lrm_expert_fc2_fwd: y [N,D] dtype (written) from phi [N,H] and
 *   W_down [E,H,D] (dtype, read).
 * lrm_combine: out [T,D] float (written) = sum over slots k ascending of
 *   alpha[t,k] * y[inv[t*K+k]]; alpha [T,K] float, inv [N] int32 (read).
 *   Needs K <= 32.
 * lrm_expert_fwd_grouped: the four in order, on one stream.
 * Buffers are caller-owned device memory, 16-byte aligned, not overlapping.
 * Sizes whose off[E] exceeds N, or non-monotone off, process no rows and
 * flag LRM_DEVERR_INDEX. Host argument errors return before any launch.
 */
lrm_status lrm_gather_tokens(const lrm_shape* shape, const int32_t* perm, const void* x,
                             void* x_disp, void* ws, size_t ws_bytes, void* stream);
lrm_status lrm_expert_fc1_fwd(const lrm_shape* shape, const int32_t* off,
                              const void* x_disp, const void* w_gate, const void* w_up,
                              void* ab, void* phi, void* ws, size_t ws_bytes,
                              void* stream);
lrm_status lrm_expert_fc2_fwd(const lrm_shape* shape, const int32_t* off, const void* phi,
                              const void* w_down, void* y, void* ws, size_t ws_bytes,
                              void* stream);
lrm_status lrm_combine(const lrm_shape* shape, const void* y, const float* alpha,
                       const int32_t* inv, float* out, void* ws, size_t ws_bytes,
                       void* stream);
lrm_status lrm_expert_fwd_grouped(const lrm_shape* shape, const int32_t* perm,
                                  const int32_t* inv, const int32_t* off, const float* alpha,
                                  const void* x, const void* w_gate, const void* w_up,
                                  const void* w_down, void* x_disp, void* ab, void* phi,
                                  void* y, float* out, void* ws, size_t ws_bytes,
                                  void* stream);

/*
 * Retained-only recompute of [a | b] in the backward (RelayMoE Sec. 3.3,
 * memory-efficient MoE recomputation: the backward rebuilds the expert
 * intermediates it consumes; LRMoE Sec. 3.1: FC1 and the activation use the
 * retained identities). ab_c [M,2H] dtype (written, rows of sel_off's
 * segments) = [x_c W_gate[e] | x_c W_up[e]] from x_c [N,D] (compacted rows,
 * read) with the layer's FP32 accumulation and one rounding, the same as
 * lrm_expert_fc1_fwd over the routed rows. With it the saved state needs no
 * [a | b]: lrm_compact then takes ab = ab_c = NULL and copies none.
 */
lrm_status lrm_expert_fc1_recompute(const lrm_shape* shape, const int32_t* sel_off,
                                    const void* x_c, const void* w_gate, const void* w_up,
                                    void* ab_c, void* ws, size_t ws_bytes, void* stream);

/*
 * The expert backward with its row operands read in place instead of from
 * compacted copies. LRMoE Sec. 3.1 (compact runtime) asks that the products
 * run over the retained rows only, in a consistent pair order, with no
 * zero-masked rows; here the compaction writes only the gradient rows
 * dy_c = alpha * g (lrm_compact with x_c = ab_c = phi_c = NULL) and the
 * products gather the rest by index:
 *   FC2 dgrad + SwiGLU grad  reads [a | b] row sel_pos[j] of ab  [N,2H];
 *   FC2 wgrad                reads phi row sel_pos[j] of phi     [N,H];
 *   FC1 wgrad                reads x row tok_c[j] of x           [T,D];
 * (j = compacted row; ab and phi in dispatch order as lrm_score reads them).
 * The FC1 dgrad product and the dx scatter are those of
 * lrm_expert_bwd_grouped. The results equal the compacted form's bit for
 * bit: the same tiles and reduction order, only the operand source differs.
 * parts: an OR of LRM_BWD_* selecting the sub-steps to run, in this order.
 * Other arguments as lrm_expert_bwd_grouped. Row indices outside their
 * source are read as zero rows (FC2 / FC1 wgrad) or skipped and flagged
 * LRM_DEVERR_INDEX (FC2 dgrad).
 */
enum {
  LRM_BWD_FC2_DGRAD = 1,
  LRM_BWD_FC2_WGRAD = 2,
  LRM_BWD_FC1_WGRAD = 4,
  LRM_BWD_FC1_DGRAD = 8,
  LRM_BWD_SCATTER_DX = 16,
  LRM_BWD_ALL = 31
};
lrm_status lrm_expert_bwd_gathered(const lrm_shape* shape, int32_t parts,
                                   const int32_t* sel_off, const int32_t* sel_pos,
                                   const int32_t* tok_c, const void* w_gate,
                                   const void* w_up, const void* w_down, const void* dy_c,
                                   const void* x, const void* ab, const void* phi,
                                   const int32_t* inv, const int32_t* row_of_pos,
                                   void* dab_c, float* dx_c, float* dw_gate, float* dw_up,
                                   float* dw_down, float* dx, void* ws, size_t ws_bytes,
                                   void* stream);

/*
 * lrm_quota_from_rate and lrm_select_quota in one launch: the quotas
 * q_e = min(ceil(num/den * n_e), cap) (cap <= 0: none; exact integers, as
 * lrm_quota_from_rate) are computed from off inside the selection and also
 * written to quota [E] int32. Needs 0 <= num <= den, den > 0. Other
 * arguments, outputs and error behaviour as lrm_select_quota.
 */
lrm_status lrm_select_rate(const lrm_shape* shape, const float* score, const int32_t* off,
                           int32_t num, int32_t den, int32_t cap, int32_t* quota,
                           uint8_t* keep, int32_t* sel_off, int32_t* sel_pos, void* ws,
                           size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LRM_H_ */
