"""Plain CPU oracle for the recalibrated MoE expert backward.

TEST INFRASTRUCTURE ONLY. This package is the slow, obviously correct
statement of what the GPU path computes, written in float64 NumPy from the
LRMoE paper ("LRMoE: Demand-Side Load Re-Calibration for Efficient MoE
Training on Memory-Constrained Nodes") and the LLEP digest ("Least-Loaded
Expert Parallelism"). Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (``demand_side_expert_gb300``) never imports it, and it
never imports the product path: the two share no code.

Every function is pinned by a ``-m "not gpu"`` test against something other
than itself (worked examples printed on the pages, closed forms, brute force,
finite differences); see ``tests/test_oracle_pins.py``.
"""

from .lrm_oracle import (  # noqa: F401
    dispatch_permute,
    quota_from_rate,
    score,
    score_variant,
    splitmix64,
    random_score,
    METRIC_LRM,
    METRIC_GRAD_SQ,
    METRIC_GRAD_ABS,
    METRIC_RANDOM,
    select_quota,
    compact,
    expert_bwd,
    expert_bwd_masked_dense,
    expert_bwd_rows,
    dx_gather,
    swiglu_grad,
    recalibrated_backward,
    gather_tokens,
    expert_fwd,
    combine,
    moe_forward,
    recompute_ab,
)
