"""CPU oracle for tree-masked speculative verification.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package smoke check and
by the benchmark's CPU-baseline leg, never by the product path.  See
oracle/tree_verify.py (verification), oracle/tree_expand.py (the draft side:
tree expansion and re-rooting) and oracle/tree_sample.py (sampling
verification) for what each function follows.
"""
from .tree_verify import (  # noqa: F401
    accepted_tokens, ancestor_bitmask, ancestor_mask, ancestors_inclusive, check_tree,
    default_scale, greedy_walk, kv_compact, kv_head_of, reroot, strict_descendants,
    target_argmax, tree_accept, tree_attention,
)
from .tree_expand import (  # noqa: F401
    candidate_scores, draft_reroot, log_softmax, ml_expand,
)
from .lm_head import lm_head_argmax, lm_head_logits  # noqa: F401
from .tree_sample import (  # noqa: F401
    draw_by_inversion, node_uniform, philox4x64_10, sample_tokens, target_probs,
    tree_accept_sampled,
)
