"""Host-side checks of the seeded workload generator (no GPU)."""

import torch

from workloads import generate, get_config


def test_tiny_is_deterministic_and_shaped():
    cfg = get_config("tiny")
    a = generate(cfg)
    b = generate(cfg)
    for k in ("topk_idx", "alpha", "x", "g", "w_down", "ab_pair", "phi_pair"):
        assert torch.equal(a[k], b[k])
    assert a["topk_idx"].shape == (64, 2) and a["alpha"].dtype == torch.float32
    assert a["ab_pair"].shape == (128, 32) and a["phi_pair"].shape == (128, 16)
    # distinct experts per token, alpha not renormalised (top-K of a softmax)
    idx = a["topk_idx"]
    assert all(len(set(r.tolist())) == 2 for r in idx)
    assert float(a["alpha"].sum(1).max()) < 1.0


def test_stress_construction_small_width():
    cfg = get_config("stress-e256", D=64, H=64)
    out = generate(cfg)  # asserts dead / single-row / full-T groups and 70% mass
    counts = torch.bincount(out["topk_idx"].reshape(-1).long(), minlength=cfg.E)
    assert int(counts.max()) >= 0.99 * cfg.T
    assert int((counts == 0).sum()) >= 16 and int((counts == 1).sum()) >= 1
    assert cfg.cap == 1280


def test_strong_skew_small_width():
    cfg = get_config("qwen3-30b-a3b-t32k", D=64, H=32)
    out = generate(cfg)
    counts = torch.bincount(out["topk_idx"].reshape(-1).long(), minlength=cfg.E)
    assert float(counts.max()) > 10 * float(counts.float().mean())
