"""Helpers of the GPU parity tests: run the CUDA path and the oracle on the
same seeded inputs and compare them under the parity rules.

Parity rules:
  dispatch permutation, selection and compaction indices: bit-exact;
  selection bit-exact against the oracle's selector run on the GPU's own
  FP32 scores, and in set agreement with the oracle's FP64 scores outside a
  1e-5 relative band around each expert's q_e-th score;
  scores within 1e-5 relative;
  BF16 gradients within 2e-2 relative Frobenius error of the FP64 oracle
  (FP32 layers: 1e-5).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

SCORE_RTOL = 1e-5
BAND = 1e-5
GRAD_TOL = {"bf16": 2e-2, "f32": 1e-5}


def to_np(t) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy()


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def run_gpu(pipe, inp: dict, rate=(1, 1), cap=0, quota=None, metric=0, seed=0, gathered=False):
    """Dispatch, lay out the saved state, run the whole path. Returns (ab, phi)."""
    pipe.dispatch(inp["topk_idx"])
    ab = pipe.to_dispatch_order(inp["ab_pair"])
    phi = pipe.to_dispatch_order(inp["phi_pair"])
    pipe.step(inp["topk_idx"], inp["alpha"], inp["x"], inp["g"], ab, phi, inp["w_gate"],
              inp["w_up"], inp["w_down"], rate=rate, cap=cap, quota=quota, metric=metric,
              seed=seed, gathered=gathered)
    torch.cuda.synchronize()
    return ab, phi


def check_dispatch(pipe, topk_idx_np, E):
    perm, inv, counts, off = oracle.dispatch_permute(topk_idx_np, E)
    N = perm.shape[0]
    assert np.array_equal(to_np(pipe.perm)[:N], perm)
    assert np.array_equal(to_np(pipe.inv)[:N], inv)
    assert np.array_equal(to_np(pipe.counts), counts)
    assert np.array_equal(to_np(pipe.off), off)
    return perm, inv, counts, off


def check_scores(gpu_score, ref_score):
    gpu = np.asarray(gpu_score, dtype=np.float64)
    ref = np.asarray(ref_score, dtype=np.float64)
    err = np.abs(gpu - ref)
    bad = err > SCORE_RTOL * np.abs(ref) + 1e-30
    assert not bad.any(), (
        f"{int(bad.sum())} scores off by > {SCORE_RTOL} rel; worst "
        f"{float((err / np.maximum(np.abs(ref), 1e-30)).max()):.3e}")


def check_selection(pipe, perm, off, quota):
    """Bit-exact against the oracle selector run on the GPU's FP32 scores."""
    N = perm.shape[0]
    gscore = to_np(pipe.score)[:N].astype(np.float64)
    keep, sel_off, sel_pos = oracle.select_quota(gscore, off, quota, perm)
    assert np.array_equal(to_np(pipe.keep)[:N], keep)
    assert np.array_equal(to_np(pipe.sel_off), sel_off)
    M = int(sel_off[-1])
    assert np.array_equal(to_np(pipe.sel_pos)[:M], sel_pos)
    return keep, sel_off, sel_pos


def check_set_agreement(keep_gpu, ref_score, off, quota):
    """Same keep decision as the FP64 oracle outside the band around tau_e."""
    R = np.asarray(ref_score, dtype=np.float64)
    for e in range(quota.shape[0]):
        lo, hi, q = int(off[e]), int(off[e + 1]), int(quota[e])
        if q == 0 or q == hi - lo:
            continue
        seg = R[lo:hi]
        tau = np.sort(seg)[::-1][q - 1]
        clear = np.abs(seg - tau) > BAND * tau
        want = seg > tau
        assert np.array_equal(keep_gpu[lo:hi][clear].astype(bool), want[clear]), f"expert {e}"


def check_compaction(pipe, inp_np, perm, sel_off, sel_pos, ab_np, phi_np, K, dtype,
                     copies=True):
    """Compacted rows and maps; `copies=False` when only the gradient rows
    were written (the products read x, ab and phi in place)."""
    M = int(sel_off[-1])
    c = oracle.compact(perm, sel_off, sel_pos, inp_np["alpha"], inp_np["x"], inp_np["g"],
                       ab_np, phi_np, K)
    assert np.array_equal(to_np(pipe.tok_c)[:M], c["tok_c"])
    N = perm.shape[0]
    assert np.array_equal(to_np(pipe.row_of_pos)[:N], c["row_of_pos"])
    for name in ("x_c", "ab_c", "phi_c") if copies else ():  # pure copies: bitwise
        assert np.array_equal(to_np(getattr(pipe, name))[:M], c[name]), name
    dy = to_np(pipe.dy_c)[:M].astype(np.float64)
    # one rounding of alpha*g to the layer dtype
    ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -23
    assert np.all(np.abs(dy - c["dy_c"]) <= ulp * np.abs(c["dy_c"]) + 1e-30)
    return c


def check_backward(pipe, inp_np, c, sel_off, inv, T, K, dtype):
    """Gradients vs the FP64 oracle run on the same selection."""
    b = oracle.expert_bwd(sel_off, inp_np["w_gate"], inp_np["w_up"], inp_np["w_down"],
                          c["dy_c"], c["x_c"], c["ab_c"], c["phi_c"])
    dx = oracle.dx_gather(b["dx_c"], inv, c["row_of_pos"], T, K)
    tol = GRAD_TOL[dtype]
    M = int(sel_off[-1])
    errs = {
        "dw_gate": rel_fro(to_np(pipe.dw_gate), b["dw_gate"]),
        "dw_up": rel_fro(to_np(pipe.dw_up), b["dw_up"]),
        "dw_down": rel_fro(to_np(pipe.dw_down), b["dw_down"]),
        "dab_c": rel_fro(to_np(pipe.dab_c)[:M], b["dab_c"]),
        "dx_c": rel_fro(to_np(pipe.dx_c)[:M], b["dx_c"]),
        "dx": rel_fro(to_np(pipe.dx)[:T], dx),
    }
    for k, v in errs.items():
        assert v <= tol, f"{k}: rel. Frobenius error {v:.3e} > {tol}"
    return errs


def numpy_inputs(inp: dict) -> dict:
    return {k: (to_np(v) if torch.is_tensor(v) else v) for k, v in inp.items()}
