"""MoE layer shapes of the synthetic workloads.

Shapes follow the LRMoE paper's evaluation setup (Sec. 4.1: 128 experts,
top-8, hidden 2048, expert FFN 768, 4 x 8192 tokens per GPU, Qwen3-30B-A3B
and GLM4.5-106B-A12B) and the LLEP digest's imbalance simulation (Sec. 4
setup: 30-95% of tokens concentrated on a few experts).
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int            # tokens
    D: int            # model (hidden) dim
    H: int            # expert FFN dim
    E: int            # experts
    K: int            # routed experts per token
    dtype: str        # "f32" or "bf16": element type of activations/weights
    zipf: float       # router bias b_e = -zipf * ln(e + 1)
    rates: tuple      # retention rates rho as exact fractions (num, den)
    cap: int = 0      # per-expert quota cap (0: none)
    stress: bool = False  # dead / hot / single-row expert construction
    seed: int = 0

    @property
    def N(self) -> int:
        return self.T * self.K


def _stress_cap(T: int, K: int, E: int) -> int:
    # capacity C = ceil(1.25 * T * K / E), exact: ceil(5 T K / (4 E))
    return (5 * T * K + 4 * E - 1) // (4 * E)


CONFIGS = {
    # tiny layer in fp32 throughout; the oracle finishes in well under 1 s
    "tiny": LayerConfig("tiny", T=64, D=32, H=16, E=8, K=2, dtype="f32",
                        zipf=1.0, rates=((1, 2),)),
    # one Qwen3-30B-A3B-shaped MoE layer, 4096 tokens
    "qwen3-30b-a3b-t4k": LayerConfig(
        "qwen3-30b-a3b-t4k", T=4096, D=2048, H=768, E=128, K=8,
        dtype="bf16", zipf=1.2, rates=((3, 5),)),
    # the same layer at the full micro-batch (4 x 8192 tokens), strong skew
    "qwen3-30b-a3b-t32k": LayerConfig(
        "qwen3-30b-a3b-t32k", T=32768, D=2048, H=768, E=128, K=8,
        dtype="bf16", zipf=1.5, rates=((1, 2),)),
    # one GLM4.5-106B-A12B-shaped MoE layer, retention sweep
    "glm45-106b-a12b-t16k": LayerConfig(
        "glm45-106b-a12b-t16k", T=16384, D=4096, H=1408, E=128, K=8,
        dtype="bf16", zipf=1.2, rates=((1, 4), (1, 2), (3, 4), (1, 1))),
    # stress: 256 experts, 70% of the routing mass on 4 experts, >= 16 dead
    # experts, single-row experts, quota capped at C = ceil(1.25 T K / E)
    "stress-e256": LayerConfig(
        "stress-e256", T=32768, D=2048, H=512, E=256, K=8, dtype="bf16",
        zipf=0.0, rates=((1, 2),), cap=_stress_cap(32768, 8, 256),
        stress=True),
}


def with_tokens(cfg: LayerConfig, T: int) -> LayerConfig:
    """The same layer recipe with T tokens (the stress cap follows T)."""
    fields = dict(cfg.__dict__)
    fields["T"] = T
    if cfg.stress:
        fields["cap"] = _stress_cap(T, cfg.K, cfg.E)
    return LayerConfig(**fields)


def get_config(name: str, **overrides) -> LayerConfig:
    """Look up a workload by name; keyword overrides give scaled variants."""
    base = CONFIGS[name]
    if not overrides:
        return base
    fields = dict(base.__dict__)
    fields.update(overrides)
    if "cap" not in overrides and base.stress:
        fields["cap"] = _stress_cap(fields["T"], fields["K"], fields["E"])
    return LayerConfig(**fields)
