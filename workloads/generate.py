"""Seeded generation of one MoE layer's backward inputs.

Recipe (all draws from one ``torch.Generator`` seeded with ``seed``, in this
order, in float32, then rounded to nearest even into the layer dtype):
  x      ~ N(0, 1)                      [T, D]   token activations (router input)
  W_r    ~ N(0, 1/D)                    [D, E]   router weight
  W_gate, W_up ~ N(0, 1/D)              [E, D, H]
  W_down ~ N(0, 1/D)                    [E, H, D]
  z      ~ N(0, 1)  [T, D];  s_t = exp(0.5 * N(0, 1))  (lognormal(0, 0.5))
  g      = z * s_t                      [T, D]   cotangent at the MoE output
Router (LLEP Sec. 2.1 MoE formula): logits = x W_r + b, b_e = -zipf*ln(e+1),
softmax over all E in float64, the K largest kept WITHOUT renormalisation
(ties to the lower expert id); alpha stored as float32.
Saved forward state per pair p = t*K + k (token-major): a = x_t W_gate[e],
b = x_t W_up[e] (float32 products of the stored values), phi = SiLU(a) * b,
each rounded to the layer dtype. The stress workload replaces the Zipf
biases: 16 dead experts (bias -1e4), 4 hot experts whose shared bias is
bisected until they hold 70% of the mean softmax mass (each then holds
>= 99% of the tokens), and two experts whose bias admits exactly one token
each.
"""

from __future__ import annotations

import math

import torch

from .configs import LayerConfig

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _topk_stable(logits: torch.Tensor, K: int) -> torch.Tensor:
    # descending by value, ties to the lower expert id (stable sort)
    order = torch.sort(-logits, dim=1, stable=True).indices
    return order[:, :K]


def _stress_bias(raw: torch.Tensor, E: int, K: int) -> torch.Tensor:
    """Router biases of the stress workload, built on float64 raw logits."""
    dev = raw.device
    bias = torch.zeros(E, dtype=torch.float64, device=dev)
    hot = torch.arange(0, 4, device=dev)
    dead = torch.arange(E - 16, E, device=dev)
    single = [E - 18, E - 17]
    bias[dead] = -1e4
    bias[single] = -1e4

    def hot_mass(bh: float) -> float:
        b = bias.clone()
        b[hot] = bh
        p = torch.softmax(raw + b, dim=1)
        return float(p[:, hot].sum(1).mean())

    lo, hi = 0.0, 30.0
    for _ in range(80):
        mid = 0.5 * (lo + hi)
        if hot_mass(mid) < 0.70:
            lo = mid
        else:
            hi = mid
    bias[hot] = 0.5 * (lo + hi)

    # each single-row expert enters the top-K of exactly one token
    for s in single:
        logits = raw + bias
        kth = torch.topk(logits, K, dim=1).values[:, K - 1]
        thr = torch.sort(kth - raw[:, s]).values
        bias[s] = 0.5 * (thr[0] + thr[1])
    return bias


@torch.no_grad()
def generate(cfg: LayerConfig, device="cpu", seed: int | None = None) -> dict:
    """Draw one layer's inputs on ``device``. Returns a dict of tensors."""
    seed = cfg.seed if seed is None else seed
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    T, D, H, E, K = cfg.T, cfg.D, cfg.H, cfg.E, cfg.K
    dt = _DTYPES[cfg.dtype]
    f32 = torch.float32

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=f32)

    x32 = randn(T, D)
    w_r = randn(D, E) / math.sqrt(D)
    w_gate = (randn(E, D, H) / math.sqrt(D)).to(dt)
    w_up = (randn(E, D, H) / math.sqrt(D)).to(dt)
    w_down = (randn(E, H, D) / math.sqrt(D)).to(dt)
    z = randn(T, D)
    s = torch.exp(0.5 * randn(T))
    g = (z * s[:, None]).to(dt)
    del z

    raw = x32.double() @ w_r.double()
    if cfg.stress:
        bias = _stress_bias(raw, E, K)
    else:
        e = torch.arange(E, dtype=torch.float64, device=dev)
        bias = -cfg.zipf * torch.log(e + 1.0)
    logits = raw + bias
    probs = torch.softmax(logits, dim=1)
    topk_idx = _topk_stable(logits, K)
    alpha = probs.gather(1, topk_idx).to(f32)
    probs_hot_mass = probs[:, :4].sum(1).mean() if cfg.stress else 0.0
    topk_idx = topk_idx.to(torch.int32).contiguous()
    x = x32.to(dt)
    del x32, raw, logits, probs

    # saved forward state, one row per pair p = t*K + k
    N = T * K
    ab_pair = torch.empty(N, 2 * H, dtype=dt, device=dev)
    phi_pair = torch.empty(N, H, dtype=dt, device=dev)
    flat = topk_idx.reshape(-1).long()
    xf = x.to(f32)
    for ex in range(E):
        pairs = torch.nonzero(flat == ex).reshape(-1)
        if pairs.numel() == 0:
            continue
        xs = xf[pairs // K]
        a = xs @ w_gate[ex].to(f32)
        b = xs @ w_up[ex].to(f32)
        phi = torch.nn.functional.silu(a) * b
        ab_pair[pairs, :H] = a.to(dt)
        ab_pair[pairs, H:] = b.to(dt)
        phi_pair[pairs] = phi.to(dt)

    out = {
        "cfg": cfg,
        "topk_idx": topk_idx,
        "alpha": alpha.contiguous(),
        "x": x.contiguous(),
        "g": g.contiguous(),
        "w_gate": w_gate.contiguous(),
        "w_up": w_up.contiguous(),
        "w_down": w_down.contiguous(),
        "ab_pair": ab_pair,
        "phi_pair": phi_pair,
    }
    if cfg.stress:
        counts = torch.bincount(flat, minlength=E)
        assert int((counts == 0).sum()) >= 16, "stress: fewer than 16 empty experts"
        assert int((counts == 1).sum()) >= 1, "stress: no single-row expert"
        assert int(counts.max()) >= (99 * T) // 100, "stress: no near-full expert"
        mass = float(probs_hot_mass)
        assert abs(mass - 0.70) <= 0.01, f"stress: hot mass {mass:.4f}"
    return out
