"""Float64 NumPy oracle of the LRMoE recalibrated expert backward on one GPU.

TEST INFRASTRUCTURE ONLY (see the package docstring): plain, slow and
written to be checked against the pages by eye. No blocking, fusion or
reordering beyond what each cited passage states. Library primitives used as
single steps: ``np.bincount``, ``np.cumsum``, ``@`` (matrix product),
``sorted``.

Sources, cited by page title and section / equation / figure:
  [LRMoE]  "LRMoE: Demand-Side Load Re-Calibration for Efficient MoE Training
           on Memory-Constrained Nodes" (arXiv 2610.37720).
  [LLEP]   "Least-Loaded Expert Parallelism: Load Balancing an Imbalanced
           Mixture-of-Experts" (papercache digest).

Notation (row-vector convention, one MoE layer):
  T tokens, D model dim, H expert FFN dim, E experts, K routed experts per
  token, N = T*K routed pairs. Pair index p = t*K + k (token-major, slot k).
  topk_idx[t, k] is the expert of pair p; alpha[t, k] its routing weight.
  Saved forward state per pair, in dispatch (expert-major) order:
    ab[pos]  = [a | b] with a = x_t W_gate[e], b = x_t W_up[e]   (2H)
    phi[pos] = SiLU(a) * b                                        (H)
  Expert e maps phi -> phi W_down[e] (W_gate, W_up: D x H; W_down: H x D).
  g[t] is the cotangent arriving at the MoE output for token t, BEFORE the
  routing weight is applied ([LRMoE] Sec. 7.1, Eq. 5).

Readings taken where the pages leave a step open are marked READING.
"""

from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    """Exact upcast (BF16 and FP32 values are representable in FP64)."""
    if hasattr(a, "detach"):  # a torch tensor handed over by a test
        a = a.detach().cpu()
        if str(a.dtype) == "torch.bfloat16":
            a = a.float()
        a = a.numpy()
    return np.asarray(a, dtype=F64)


def _i64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.asarray(a, dtype=np.int64)


# ---------------------------------------------------------------------------
# Step 1: forward dispatch permutation
# ---------------------------------------------------------------------------
def dispatch_permute(topk_idx, E: int):
    """Stable re-index of the routed pairs by expert id (counting sort).

    [LLEP] Sec. 2.1 ("Implementation"): the batch is re-indexed into
    per-expert groups B' = [B_0, B_1, ...]; its example routes tokens
    [a, b, c, d] to experts [2, 6, 2, 1] and forms [d, a, c, b], i.e. groups
    in expert order and, inside a group, the original order (a before c).
    [LLEP] Alg. 4 sorts the flattened (token, slot) indices the same way.
    [LRMoE] Alg. 1 (forward admission) counts N_e = |P_e| per expert.

    Returns (perm, inv, counts, off), all int64:
      perm[pos] = p   pair index stored at dispatch position pos
      inv[p]    = pos inverse of perm
      counts[e] = n_e number of pairs routed to expert e
      off[e]    = sum_{e' < e} n_e' (length E + 1; off[E] = N)
    """
    idx = _i64(topk_idx)
    if idx.ndim != 2:
        raise ValueError("topk_idx must be [T, K]")
    flat = idx.reshape(-1)
    N = flat.shape[0]
    if N and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    off = np.zeros(E + 1, dtype=np.int64)
    off[1:] = np.cumsum(counts)
    cursor = off[:E].copy()
    perm = np.empty(N, dtype=np.int64)
    inv = np.empty(N, dtype=np.int64)
    for p in range(N):  # ascending pair index => stable inside each group
        e = flat[p]
        pos = cursor[e]
        perm[pos] = p
        inv[p] = pos
        cursor[e] += 1
    return perm, inv, counts, off


def permute_rows(src, perm) -> np.ndarray:
    """Row re-index into dispatch order: dst[pos] = src[perm[pos]].

    [LLEP] Sec. 2.1: B' is B with its rows taken in dispatch order. Used to
    lay out the saved forward state the way the expert GEMMs produced it.
    """
    return np.asarray(src)[_i64(perm)]


# ---------------------------------------------------------------------------
# Quota rule
# ---------------------------------------------------------------------------
def quota_from_rate(counts, num: int, den: int, cap: int | None = None):
    """Per-expert retention quota q_e = min(ceil(rho * n_e), cap), rho = num/den.

    [LRMoE] Sec. 3.1: quotas 0 <= K_e <= N_e, retention rate
    rho = sum_e K_e / N; they are fixed before backward. The closed form
    ceil(rho * n_e) (optionally capped) is the workload's quota rule.
    READING: the ceiling is taken in exact integer arithmetic,
    (num * n_e + den - 1) // den, because a floating-point ceil of
    rho * n_e rounds the wrong way for some n_e.
    """
    if den <= 0 or num < 0 or num > den:
        raise ValueError("rate must satisfy 0 <= num <= den, den > 0")
    q = []
    for n in (int(c) for c in np.asarray(counts).reshape(-1)):
        v = (num * n + den - 1) // den
        if cap is not None and cap > 0:
            v = min(v, int(cap))
        q.append(v)
    return np.asarray(q, dtype=np.int64)


# ---------------------------------------------------------------------------
# Step 2: Load Recalibration Metric
# ---------------------------------------------------------------------------
def score(g, phi, alpha, perm, K: int) -> np.ndarray:
    """LRM score of every routed pair, in dispatch order.

    [LRMoE] Sec. 3.2, Prop. 3.1, Eq. 1-3 and Sec. 7.1, Eq. 11-12:
        R_u = || (alpha_u g_t) phi_u^T ||_F^2
            = alpha_u^2 * ||g_t||_2^2 * ||phi_u||_2^2,
    u = (t, e) with g_t taken before the routing weight and phi_u the saved
    input of the protected projection (FC2 of the SwiGLU expert).
    [LRMoE] Alg. 1 (backward calibration) computes it for every routed pair.

    g: [T, D]; phi: [N, H] in dispatch order; alpha: [T, K];
    perm: dispatch permutation. Returns R: float64 [N], R[pos] for the pair
    stored at dispatch position pos.
    """
    g64, phi64, a64 = _f64(g), _f64(phi), _f64(alpha)
    perm = _i64(perm)
    g_sq = np.sum(g64 * g64, axis=1)          # ||g_t||^2, one per token
    phi_sq = np.sum(phi64 * phi64, axis=1)    # ||phi_u||^2, one per pair
    t_of_pos = perm // K
    alpha_of_pos = a64.reshape(-1)[perm]
    return alpha_of_pos * alpha_of_pos * g_sq[t_of_pos] * phi_sq


# ---------------------------------------------------------------------------
# Step 2 variants: the ablation's alternative selection criteria
# ---------------------------------------------------------------------------
METRIC_LRM, METRIC_GRAD_SQ, METRIC_GRAD_ABS, METRIC_RANDOM = 0, 1, 2, 3
_GAMMA = 0x9E3779B97F4A7C15
_MASK64 = (1 << 64) - 1


def splitmix64(state: int) -> int:
    """One output of SplitMix64 for the state AFTER its increment.

    Published generator (Steele, Lea and Flood, "Fast splittable pseudorandom
    number generators", OOPSLA 2014; Vigna's splitmix64.c): the state
    advances by 0x9E3779B97F4A7C15 and is mixed by two xor-shift-multiply
    rounds and a final xor-shift.
    """
    z = state & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def random_score(seed: int, p: int) -> float:
    """Random criterion: output p+1 of SplitMix64 seeded with `seed`, top 24
    bits scaled into [0, 1) (exact in float32)."""
    z = splitmix64((seed + (p + 1) * _GAMMA) & _MASK64)
    return float(z >> 40) * 2.0 ** -24


def score_variant(metric: int, g, phi, alpha, perm, K: int, seed: int = 0) -> np.ndarray:
    """Per-pair selection score under the criteria compared in [LRMoE] Sec. 4.7
    (Table 2), in dispatch order.

      METRIC_LRM       alpha_u^2 ||g_t||^2 ||phi_u||^2 (``score``)
      METRIC_GRAD_SQ   ||g_t||_2^2                 READING of the squared-gradient-norm row
      METRIC_GRAD_ABS  ||g_t||_1 = sum_d |g_t,d|   READING of the absolute-gradient row
      METRIC_RANDOM    random_score(seed, p)       READING of the random-selection row
    The gradient-only criteria use the cotangent g_t alone, so all K pairs of
    a token score the same; Sec. 4.7 contrasts exactly that with LRM, which
    also weighs the pair's activation phi_u.
    """
    perm = _i64(perm)
    if metric == METRIC_LRM:
        return score(g, phi, alpha, perm, K)
    t_of_pos = perm // K
    if metric == METRIC_GRAD_SQ:
        g64 = _f64(g)
        return np.sum(g64 * g64, axis=1)[t_of_pos]
    if metric == METRIC_GRAD_ABS:
        return np.sum(np.abs(_f64(g)), axis=1)[t_of_pos]
    if metric == METRIC_RANDOM:
        return np.array([random_score(seed, int(p)) for p in perm], dtype=F64)
    raise ValueError("unknown metric")


# ---------------------------------------------------------------------------
# Step 3: per-expert top-q selection
# ---------------------------------------------------------------------------
def select_quota(R, off, quota, perm):
    """Keep, inside each expert segment, the q_e highest-scoring pairs.

    [LRMoE] Alg. 1 (backward calibration): S*_e = TopK(P_e, {v_p}, K_e) for
    each expert e. Sec. 7.2, Prop. 7.1 / Eq. 13-17: with fixed per-expert
    drop counts, keeping the largest scores inside every partition is
    optimal; solutions differ only among tied boundary scores.
    READING: ties are broken by the lower pair index p = t*K + k.
    READING: retained rows are listed in ascending dispatch position
    ([LRMoE] Sec. 3.1, compact runtime: retained pairs keep one consistent order).

    Returns (keep uint8 [N] in dispatch order, sel_off int64 [E+1] =
    exclusive scan of the quotas, sel_pos int64 [M] retained dispatch
    positions, ascending inside each segment).
    """
    R = np.asarray(R, dtype=F64)
    off = _i64(off)
    quota = _i64(quota)
    perm = _i64(perm)
    E = quota.shape[0]
    N = R.shape[0]
    keep = np.zeros(N, dtype=np.uint8)
    sel_off = np.zeros(E + 1, dtype=np.int64)
    chosen = []
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        q = int(quota[e])
        if q < 0 or q > hi - lo:
            raise ValueError(f"quota of expert {e} outside [0, n_e]")
        ranked = sorted(range(lo, hi), key=lambda pos: (-R[pos], perm[pos]))
        kept = sorted(ranked[:q])
        for pos in kept:
            keep[pos] = 1
        chosen.extend(kept)
        sel_off[e + 1] = sel_off[e] + q
    return keep, sel_off, np.asarray(chosen, dtype=np.int64)


# ---------------------------------------------------------------------------
# Step 4: physical compaction
# ---------------------------------------------------------------------------
def compact(perm, sel_off, sel_pos, alpha, x, g, ab, phi, K: int):
    """Gather retained rows into contiguous expert-major segments.

    [LRMoE] Sec. 3.1 ("compact runtime") and Sec. 3.4 / Fig. 4: retained
    gradient rows and their matching saved activations are packed in a
    consistent pair order; counts and offsets define variable-size grouped
    GEMMs; no zero-masked full-size tensors. [LRMoE] Sec. 7.1, Eq. 5: the
    gradient row handed to the expert is delta_u = alpha_u * g_t.

    For retained row j: i = sel_pos[j], p = perm[i], t = p // K:
      dy_c[j] = alpha[p] * g[t]  (float64 here)
      x_c[j]  = x[t];  ab_c[j] = ab[i];  phi_c[j] = phi[i];  tok_c[j] = t
      row_of_pos[i] = j, and -1 for every dropped dispatch position.
    """
    perm, sel_pos = _i64(perm), _i64(sel_pos)
    M = int(_i64(sel_off)[-1])
    assert sel_pos.shape[0] == M
    a64 = _f64(alpha).reshape(-1)
    p = perm[sel_pos]
    t = p // K
    out = {
        "dy_c": a64[p][:, None] * _f64(g)[t],
        "x_c": _f64(x)[t],
        "ab_c": _f64(ab)[sel_pos],
        "phi_c": _f64(phi)[sel_pos],
        "tok_c": t,
    }
    row_of_pos = np.full(perm.shape[0], -1, dtype=np.int64)
    row_of_pos[sel_pos] = np.arange(M, dtype=np.int64)
    out["row_of_pos"] = row_of_pos
    return out


# ---------------------------------------------------------------------------
# Step 5: SwiGLU expert backward over the retained rows
# ---------------------------------------------------------------------------
def swiglu_grad(dphi, a, b):
    """Gradient of phi = SiLU(a) * b, SiLU(z) = z * sigmoid(z).

    The activation step between FC2 and FC1 ([LRMoE] Sec. 3.1, "FC2, the
    activation function, FC1"); the experts are SwiGLU feed-forward blocks
    (LLEP Sec. 4 setup; RelayMoE Sec. 4.2 Table 3).
    READING: SiLU on the gate half a, linear up half b.
      d phi / d a = b * sigmoid(a) * (1 + a * (1 - sigmoid(a)))
      d phi / d b = SiLU(a)
    """
    dphi, a, b = _f64(dphi), _f64(a), _f64(b)
    s = 1.0 / (1.0 + np.exp(-a))
    da = dphi * b * s * (1.0 + a * (1.0 - s))
    db = dphi * a * s
    return da, db


def expert_bwd(sel_off, w_gate, w_up, w_down, dy_c, x_c, ab_c, phi_c,
               experts=None):
    """Per-expert SwiGLU backward over the compacted retained rows.

    [LRMoE] Alg. 1 (PackedExpertBackward) and Sec. 3.4: four variable-size
    products per expert (FC2 dgrad and wgrad, FC1 dgrad and wgrad) over the
    m_e retained rows only; m_e is the row dimension of the data-gradient
    products and the reduction dimension of the weight-gradient products.
    [LRMoE] Sec. 7.1, Eq. 8-9: the FC2 weight gradient is the sum over pairs
    of delta_u phi_u^T (stored here transposed, H x D, row convention).

    Per expert e with rows J_e = [sel_off[e], sel_off[e+1]):
      dW_down[e] = phi_c[J]^T dy_c[J]                      (H x D)
      dphi       = dy_c[J] W_down[e]^T                     (m x H)
      da, db     = swiglu_grad(dphi, a, b)
      dW_gate[e] = x_c[J]^T da ;  dW_up[e] = x_c[J]^T db   (D x H)
      dx_c[J]    = da W_gate[e]^T + db W_up[e]^T           (m x D)
    Experts with no retained rows get zero weight gradients.
    ``experts`` restricts the work to a subset (others stay zero).
    """
    sel_off = _i64(sel_off)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    dy, xc, abc, phic = _f64(dy_c), _f64(x_c), _f64(ab_c), _f64(phi_c)
    E, D, H = wg.shape
    M = int(sel_off[-1])
    dW_gate = np.zeros((E, D, H), dtype=F64)
    dW_up = np.zeros((E, D, H), dtype=F64)
    dW_down = np.zeros((E, H, D), dtype=F64)
    dab_c = np.zeros((M, 2 * H), dtype=F64)
    dx_c = np.zeros((M, D), dtype=F64)
    for e in (range(E) if experts is None else experts):
        lo, hi = int(sel_off[e]), int(sel_off[e + 1])
        if hi == lo:
            continue
        d_y = dy[lo:hi]
        dW_down[e] = phic[lo:hi].T @ d_y
        dphi = d_y @ wd[e].T
        da, db = swiglu_grad(dphi, abc[lo:hi, :H], abc[lo:hi, H:])
        dW_gate[e] = xc[lo:hi].T @ da
        dW_up[e] = xc[lo:hi].T @ db
        dx_c[lo:hi] = da @ wg[e].T + db @ wu[e].T
        dab_c[lo:hi, :H] = da
        dab_c[lo:hi, H:] = db
    return {"dw_gate": dW_gate, "dw_up": dW_up, "dw_down": dW_down,
            "dab_c": dab_c, "dx_c": dx_c}


def expert_bwd_rows(rows, sel_off, w_gate, w_up, w_down, dy_rows, ab_rows):
    """Data-gradient rows only (dab_c[j], dx_c[j]) for a list of compacted rows.

    Same arithmetic as ``expert_bwd`` restricted to the rows asked for:
    ``rows`` are compacted row indices j (each row's expert is the segment of
    sel_off that holds it) and dy_rows[n], ab_rows[n] hold dy_c[rows[n]],
    ab_c[rows[n]]. Used to check sampled rows of full-size runs one by one.
    """
    sel_off = _i64(sel_off)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    H = wg.shape[2]
    rows = _i64(rows)
    dy, abr = _f64(dy_rows), _f64(ab_rows)
    dab = np.zeros((rows.shape[0], 2 * H), dtype=F64)
    dxc = np.zeros((rows.shape[0], wg.shape[1]), dtype=F64)
    for n, j in enumerate(rows):
        e = int(np.searchsorted(sel_off, j, side="right") - 1)
        dphi = dy[n] @ wd[e].T
        da, db = swiglu_grad(dphi, abr[n, :H], abr[n, H:])
        dab[n, :H], dab[n, H:] = da, db
        dxc[n] = da @ wg[e].T + db @ wu[e].T
    return dab, dxc


def dx_gather(dx_c, inv, row_of_pos, T: int, K: int) -> np.ndarray:
    """Scatter the retained input-gradient rows back to their tokens.

    [LRMoE] Sec. 3.1 and Sec. 3.4: returned input-gradient contributions are
    added at their original token / routing-slot positions in a
    zero-initialised dense buffer; dropped pairs contribute nothing.
    READING: the dense target is the per-token sum dx[t] = sum over kept
    slots k (ascending) of dx_c[row_of_pos[inv[t*K + k]]].
    """
    dxc = _f64(dx_c)
    inv, rop = _i64(inv), _i64(row_of_pos)
    D = dxc.shape[1] if dxc.ndim == 2 else 0
    dx = np.zeros((T, D), dtype=F64)
    for t in range(T):
        for k in range(K):
            j = rop[inv[t * K + k]]
            if j >= 0:
                dx[t] += dxc[j]
    return dx


def expert_bwd_masked_dense(keep, off, perm, alpha, x, g, ab, phi,
                            w_gate, w_up, w_down, K: int):
    """Zero-masked full-size variant of the same backward.

    [LRMoE] Sec. 3.4: masking dropped rows in full-size tensors yields the
    same gradients as the packed computation "apart from ordinary
    floating-point differences" (but not its savings). Every routed pair
    takes part; dropped rows carry a zero gradient row. Returns
    (dW_gate, dW_up, dW_down, dx) in float64.
    """
    keep = np.asarray(keep).astype(F64)
    off, perm = _i64(off), _i64(perm)
    a64 = _f64(alpha).reshape(-1)
    xx, gg, abd, phid = _f64(x), _f64(g), _f64(ab), _f64(phi)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    E, D, H = wg.shape
    T = xx.shape[0]
    t_of_pos = perm // K
    dY = (a64[perm] * keep)[:, None] * gg[t_of_pos]   # masked rows are zero
    dW_gate = np.zeros((E, D, H))
    dW_up = np.zeros((E, D, H))
    dW_down = np.zeros((E, H, D))
    dx = np.zeros((T, D))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        dW_down[e] = phid[lo:hi].T @ dY[lo:hi]
        dphi = dY[lo:hi] @ wd[e].T
        da, db = swiglu_grad(dphi, abd[lo:hi, :H], abd[lo:hi, H:])
        xs = xx[t_of_pos[lo:hi]]
        dW_gate[e] = xs.T @ da
        dW_up[e] = xs.T @ db
        dxe = da @ wg[e].T + db @ wu[e].T
        for r, pos in enumerate(range(lo, hi)):
            dx[t_of_pos[pos]] += dxe[r]
    return dW_gate, dW_up, dW_down, dx


# ---------------------------------------------------------------------------
# Forward expert pass (produces the saved state the backward consumes)
# ---------------------------------------------------------------------------
def gather_tokens(x, perm, K: int) -> np.ndarray:
    """x_disp[pos] = x[t] with t = perm[pos] // K: the token rows in dispatch
    order, one per routed pair ([LLEP] Sec. 2.1: B' = [B_0, B_1, ...], each
    B_i holding the tokens routed to expert i)."""
    xd = _f64(x)
    return xd[_i64(perm) // K]


def expert_fwd(off, w_gate, w_up, w_down, x_disp):
    """Per-expert SwiGLU feed-forward over the dispatch-ordered rows.

    [LLEP] Sec. 2.1 ("Implementation"): one product B_i W_i per activated
    expert over its group of rows. [LRMoE] Sec. 3.1 (design overview) and
    Alg. 1 (FullForwardAndSaveContext): the full forward runs every routed
    pair through its expert and keeps the intermediates the backward needs.
    READING (as in ``swiglu_grad``): a = x W_gate[e], b = x W_up[e],
    phi = SiLU(a) * b, y = phi W_down[e]; the saved state is [a | b] and phi.
    Returns (ab [N,2H], phi [N,H], y [N,D]) in dispatch order.
    """
    off = _i64(off)
    Wg, Wu, Wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    xd = _f64(x_disp)
    E, D, H = Wg.shape
    N = xd.shape[0]
    ab = np.zeros((N, 2 * H), dtype=F64)
    phi = np.zeros((N, H), dtype=F64)
    y = np.zeros((N, D), dtype=F64)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        a = xd[lo:hi] @ Wg[e]
        b = xd[lo:hi] @ Wu[e]
        ph = a / (1.0 + np.exp(-a)) * b
        ab[lo:hi, :H] = a
        ab[lo:hi, H:] = b
        phi[lo:hi] = ph
        y[lo:hi] = ph @ Wd[e]
    return ab, phi, y


def combine(y, alpha, inv, K: int) -> np.ndarray:
    """MoE output h_t = sum_k alpha[t, k] * y[inv[t*K + k]].

    [LLEP] Sec. 2.1, MoE output formula: the gated sum of the selected
    experts' outputs (g_i = s_i for the top-K experts, no renormalisation);
    [LRMoE] Sec. 3.1: the forward combines the expert outputs into the dense
    representation handed to the next layer. Slots summed in ascending k.
    """
    yd, al, inv = _f64(y), _f64(alpha), _i64(inv)
    T = al.shape[0]
    out = np.zeros((T, yd.shape[1]), dtype=F64)
    for t in range(T):
        for k in range(K):
            out[t] += al[t, k] * yd[inv[t * K + k]]
    return out


def moe_forward(topk_idx, alpha, x, w_gate, w_up, w_down, E: int):
    """Dispatch, gather, per-expert forward and combine, end to end."""
    idx = _i64(topk_idx)
    T, K = idx.shape
    perm, inv, counts, off = dispatch_permute(idx, E)
    x_disp = gather_tokens(x, perm, K)
    ab, phi, y = expert_fwd(off, w_gate, w_up, w_down, x_disp)
    out = combine(y, alpha, inv, K)
    return {"perm": perm, "inv": inv, "counts": counts, "off": off, "x_disp": x_disp,
            "ab": ab, "phi": phi, "y": y, "out": out}


# ---------------------------------------------------------------------------
# Retained-only recompute of the FC1 outputs
# ---------------------------------------------------------------------------
def recompute_ab(sel_off, w_gate, w_up, x_c):
    """[a | b] of the retained rows rebuilt from their token rows during the
    backward instead of read from saved state.

    RelayMoE Sec. 3.3 (memory-efficient MoE recomputation, Fig. 8): the
    backward reconstructs the expert intermediates it needs, consumes them
    and releases them. [LRMoE] Sec. 3.1: FC2, the activation and FC1 use the
    same retained identities, so only retained rows are rebuilt.
    a = x_c W_gate[e], b = x_c W_up[e] per expert segment of the compacted rows.
    """
    sel_off = _i64(sel_off)
    Wg, Wu = _f64(w_gate), _f64(w_up)
    xc = _f64(x_c)
    E, D, H = Wg.shape
    ab = np.zeros((xc.shape[0], 2 * H), dtype=F64)
    for e in range(E):
        lo, hi = int(sel_off[e]), int(sel_off[e + 1])
        if hi > lo:
            ab[lo:hi, :H] = xc[lo:hi] @ Wg[e]
            ab[lo:hi, H:] = xc[lo:hi] @ Wu[e]
    return ab


# ---------------------------------------------------------------------------
# The whole path
# ---------------------------------------------------------------------------
def recalibrated_backward(topk_idx, alpha, x, g, ab_pair, phi_pair,
                          w_gate, w_up, w_down, E: int,
                          num: int | None = None, den: int | None = None,
                          cap: int | None = None, quota=None, recompute: bool = False):
    """Dispatch, score, select, compact and expert backward, end to end.

    [LRMoE] Alg. 1: forward counts N_e (admission), backward computes v_p,
    TopK per expert, compacts and runs the packed expert backward, then
    scatters input gradients with zeros. Single GPU: no routing across
    instances, no all-to-all, no CPU offload queue.

    ab_pair / phi_pair hold the saved state per pair index p (token-major);
    it is laid out in dispatch order here, as the forward expert products
    produced it ([LLEP] Sec. 2.1 re-index). Either a rate (num/den, cap) or
    an explicit per-expert ``quota`` is given. With ``recompute`` the
    retained rows' [a | b] come from ``recompute_ab`` instead of ab_pair
    (which may then be None).
    """
    idx = _i64(topk_idx)
    T, K = idx.shape
    perm, inv, counts, off = dispatch_permute(idx, E)
    phi = permute_rows(_f64(phi_pair), perm)
    H = phi.shape[1]
    ab = (np.zeros((perm.shape[0], 2 * H)) if recompute
          else permute_rows(_f64(ab_pair), perm))
    if quota is None:
        quota = quota_from_rate(counts, num, den, cap)
    R = score(g, phi, alpha, perm, K)
    keep, sel_off, sel_pos = select_quota(R, off, quota, perm)
    c = compact(perm, sel_off, sel_pos, alpha, x, g, ab, phi, K)
    if recompute:
        c["ab_c"] = recompute_ab(sel_off, w_gate, w_up, c["x_c"])
    b = expert_bwd(sel_off, w_gate, w_up, w_down,
                   c["dy_c"], c["x_c"], c["ab_c"], c["phi_c"])
    dx = dx_gather(b["dx_c"], inv, c["row_of_pos"], T, K)
    out = {"perm": perm, "inv": inv, "counts": counts, "off": off,
           "quota": _i64(quota), "score": R, "keep": keep,
           "sel_off": sel_off, "sel_pos": sel_pos, "dx": dx,
           "ab": ab, "phi": phi}
    out.update(c)
    out.update(b)
    return out
