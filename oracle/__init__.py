"""Oracle for the routed-expert MoE layer iteration -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 CPU restatement of what one refinement iteration of an
Epoch MoE layer computes. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import it; the product
library never does, and the two share no code (the seeded input generators
live in the separate ``synth`` package).
"""
from .epoch_moe import (  # noqa: F401
    IterResult,
    LayerOracle,
    AtlasResult,
    PlanResult,
    atlas_support,
    softmax_rows,
    Router,
    chosen_groups,
    group_scores,
    route_position,
    sigmoid,
    classify_positions,
    coverage_threshold,
    dense_moe,
    dense_probabilities,
    selection_weights,
    gate_logits,
    hit_counts,
    near_tie,
    plan_support,
    rank_eligible,
    renorm_softmax,
    silu,
    swiglu_expert,
    topk_select,
)
