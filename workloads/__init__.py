"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark."""
from .synth import (  # noqa: F401
    Workload, chain_tree, complete_binary_tree, draft_tokens, make_qkv, make_workload,
    ml_expansion_tree, node_depths, normal, planted_logits, random_parent_tree,
    uniform_parent_tree,
)
