"""The oracle's pins must catch plausible mistakes.  Each test plants one
mistake in the oracle (on the CPU, through monkeypatching the oracle module)
and checks that at least one pin from tests/test_oracle_*.py then fails."""
import numpy as np
import pytest

import oracle.tree_verify as tv
from tests import test_oracle_accept as acc
from tests import test_oracle_attention as att
from tests import test_oracle_compact as cmp


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, ValueError, IndexError, KeyError):
        return True
    return False


def _attention_pins(golden_dir):
    return [
        lambda: att.check_worked_examples(golden_dir),
        lambda: att.check_chain_is_causal(0, 37, 9),
        lambda: att.check_single_node_is_decode(0, 100),
        lambda: att.check_node_is_attention_over_own_path(0),
    ]


def _some_fail(pins):
    return any(_fails(p) for p in pins)


def test_pins_pass_unmutated(golden_dir):
    assert not _some_fail(_attention_pins(golden_dir))


def test_exclusive_self_is_caught(monkeypatch, golden_dir):
    orig = tv.ancestors_inclusive
    monkeypatch.setattr(tv, "ancestors_inclusive", lambda parent, i: orig(parent, i)[1:])
    assert _some_fail(_attention_pins(golden_dir))


def test_wrong_gqa_map_is_caught(monkeypatch, golden_dir):
    monkeypatch.setattr(tv, "kv_head_of", lambda h, hq, hkv: h % hkv)
    assert _some_fail(_attention_pins(golden_dir))


def test_wrong_scale_is_caught(monkeypatch, golden_dir):
    monkeypatch.setattr(tv, "default_scale", lambda d: 1.0 / d)
    assert _some_fail(_attention_pins(golden_dir))


def test_parent_only_mask_is_caught(monkeypatch, golden_dir):
    # a node that sees itself and its parent but not the rest of its path
    def two_levels(parent, i):
        return [i] + ([int(parent[i])] if parent[i] >= 0 else [])
    monkeypatch.setattr(tv, "ancestors_inclusive", two_levels)
    assert _some_fail(_attention_pins(golden_dir))


def test_transposed_qk_is_caught(monkeypatch, golden_dir):
    real = tv.tree_attention

    def mutant(q, k, v, P, parent, scale=None):
        q = np.asarray(q, dtype=np.float64)
        # heads and nodes swapped when the shapes allow it
        if q.shape[0] == q.shape[1]:
            q = q.transpose(1, 0, 2).copy()
        return real(q, k, v, P, parent, scale)
    monkeypatch.setattr(att.oracle, "tree_attention", mutant)
    pins = _attention_pins(golden_dir) + [lambda: att.check_chain_is_causal(1, 5, 4, hq=4, hkv=2)]
    assert _some_fail(pins)


def _accept_pins(golden_dir):
    return [
        lambda: acc.check_accept_worked_examples(golden_dir),
        lambda: acc.check_bruteforce_small_trees(max_n=5, trials=2),
    ]


def test_highest_index_tie_is_caught(monkeypatch, golden_dir):
    def walk(am, token, parent):
        path = [0]
        while True:
            u = path[-1]
            m = [c for c in range(len(parent)) if parent[c] == u and token[c] == am[u]]
            if not m:
                return path
            path.append(max(m))
    monkeypatch.setattr(tv, "greedy_walk", walk)
    assert _some_fail(_accept_pins(golden_dir))


def test_wrong_bonus_token_is_caught(monkeypatch, golden_dir):
    monkeypatch.setattr(tv, "accepted_tokens",
                        lambda path, am, token: [int(token[a]) for a in path[1:]] + [int(am[path[0]])])
    assert _some_fail(_accept_pins(golden_dir))


def test_new_parent_off_by_one_is_caught(monkeypatch, golden_dir):
    real = tv.reroot

    def mutant(parent, path, P):
        new_pos, new_parent, r = real(parent, path, P)
        new_parent = np.where(new_parent >= 0, new_parent + 1, new_parent)
        return new_pos, new_parent, r
    monkeypatch.setattr(tv, "reroot", mutant)
    assert _fails(acc.check_accept_worked_examples, golden_dir)


def test_inclusive_survivors_is_caught(monkeypatch, golden_dir):
    real = tv.strict_descendants
    monkeypatch.setattr(tv, "strict_descendants", lambda parent, u: [u] + real(parent, u))
    assert _fails(acc.check_accept_worked_examples, golden_dir)


def test_compaction_from_wrong_row_is_caught(monkeypatch):
    def mutant(cache, P, new_pos):
        old = np.asarray(cache)
        new = old.copy()
        for i, pos in enumerate(new_pos):
            if pos >= 0:
                new[..., pos, :] = old[..., P + i - 1 if i else P, :]
        return new
    monkeypatch.setattr(cmp.oracle, "kv_compact", mutant)
    assert _fails(cmp.test_compaction_is_a_permutation_copy, 1) or \
        _fails(cmp.test_reroot_preserves_survivor_attention)


def test_last_occurrence_argmax_is_caught(monkeypatch):
    def mutant(logits):
        x = np.asarray(logits)
        return (x.shape[1] - 1 - np.argmax(x[:, ::-1], axis=1)).astype(np.int32)
    monkeypatch.setattr(acc.oracle, "target_argmax", mutant)
    assert _fails(acc.test_argmax_ties_and_nan_follow_first_occurrence)


# ------------------------------------------------------------ draft side

import oracle.tree_expand as te  # noqa: E402
from tests import test_oracle_expand as exp  # noqa: E402


def _expand_pins():
    return [
        exp.check_worked_expansion,
        lambda: exp.check_brute_force_by_probability(0),
        lambda: exp.check_brute_force_by_probability(1),
        lambda: exp.check_single_root_is_argmax(0),
        exp.check_ties_go_to_lower_position_then_token,
    ]


def _reroot_pins():
    return [lambda: exp.check_worked_reroot(c) for c in "ABC"]


def test_draft_pins_pass_unmutated():
    assert not _some_fail(_expand_pins())
    assert not _some_fail(_reroot_pins())


def test_expansion_without_path_score_is_caught(monkeypatch):
    monkeypatch.setattr(te, "candidate_scores",
                        lambda logits, frontier, cum: te.log_softmax(logits))
    assert _some_fail(_expand_pins())


def test_expansion_on_probabilities_is_caught(monkeypatch):
    def prob_scores(logits, frontier, cum):
        base = np.array([float(cum[int(u)]) for u in frontier])
        return base[:, None] + np.exp(te.log_softmax(logits))
    monkeypatch.setattr(te, "candidate_scores", prob_scores)
    assert _some_fail(_expand_pins())


def test_reversed_tie_rule_is_caught(monkeypatch):
    def ml_expand_high_token_first(logits, frontier, cum, w):
        scores = te.candidate_scores(logits, frontier, cum)
        nf, vocab = scores.shape
        flat = scores.ravel()
        order = np.lexsort((-np.arange(flat.size), -flat))[:w]
        f, v = np.divmod(order, vocab)
        parent = np.array([int(frontier[int(i)]) for i in f], dtype=np.int32)
        return parent, v.astype(np.int32), flat[order]
    monkeypatch.setattr(te, "ml_expand", ml_expand_high_token_first)
    monkeypatch.setattr(exp.oracle, "ml_expand", ml_expand_high_token_first)
    assert _some_fail(_expand_pins())


def test_target_side_survivors_on_the_draft_side_are_caught(monkeypatch):
    # the subtree under a_m itself (the target side's rule), bonus ignored
    def strict_desc_rule(parent, token, cum, path, bonus, prefix_len):
        n = len(parent)
        path = [int(a) for a in path]
        surv = [i for i in range(n) if i != path[-1]
                and path[-1] in te.ancestors_inclusive(parent, i)]
        new_pos = np.full(n, -1, dtype=np.int32)
        for idx, node in enumerate(path + surv):
            new_pos[node] = prefix_len + idx
        rank = {node: k for k, node in enumerate(surv)}
        new_parent = np.full(n, -1, dtype=np.int32)
        new_token = np.full(n, -1, dtype=np.int32)
        new_cum = np.zeros(n)
        for k, node in enumerate(surv):
            new_parent[k] = rank.get(int(parent[node]), -1)
            new_token[k] = int(token[node])
            new_cum[k] = float(cum[node]) - float(cum[path[-1]])
        return {"new_pos": new_pos, "new_parent": new_parent, "new_token": new_token,
                "new_cum": new_cum, "n_survivors": len(surv), "new_root": path[-1]}
    monkeypatch.setattr(exp.oracle, "draft_reroot", strict_desc_rule)
    assert _some_fail(_reroot_pins())


def test_unrebased_path_scores_are_caught(monkeypatch):
    orig = te.draft_reroot

    def no_rebase(parent, token, cum, path, bonus, prefix_len):
        res = orig(parent, token, cum, path, bonus, prefix_len)
        r = res["n_survivors"]
        if r:
            b = res["new_root"]
            res["new_cum"][:r] += float(cum[b])
        return res
    monkeypatch.setattr(exp.oracle, "draft_reroot", no_rebase)
    assert _some_fail(_reroot_pins())


# ------------------------------------------------------------ sampling

import oracle.tree_sample as ts  # noqa: E402
from tests import test_oracle_sample as smp  # noqa: E402


def _sample_pins():
    return [lambda: smp.check_drawn_distribution(0.5), lambda: smp.check_drawn_distribution(2.0),
            smp.test_inversion_edges, lambda: smp.test_philox_matches_numpy((1, 2))]


def test_sampling_pins_pass_unmutated():
    assert not _some_fail(_sample_pins())


def test_temperature_multiplied_is_caught(monkeypatch):
    orig = ts.target_probs
    monkeypatch.setattr(ts, "target_probs", lambda logits, T: orig(logits, 1.0 / T))
    assert _some_fail(_sample_pins())


def test_inversion_at_or_above_is_caught(monkeypatch):
    def left(probs_row, u):
        c = np.cumsum(np.asarray(probs_row, dtype=np.float64))
        return int(min(np.searchsorted(c, u, side="left"), len(c) - 1))
    monkeypatch.setattr(ts, "draw_by_inversion", left)
    monkeypatch.setattr(smp.oracle, "draw_by_inversion", left)
    assert _some_fail(_sample_pins())


def test_philox_without_key_schedule_is_caught(monkeypatch):
    monkeypatch.setattr(ts, "_W0", 0)
    assert _some_fail(_sample_pins())


# ------------------------------------------------------------ LM head

def _lm_head_pins():
    from tests import test_oracle_lm_head as lm
    return [lambda: lm.check_matches_torch(0), lm.check_hand_built_winner_and_tie]


def test_lm_head_pins_pass_unmutated():
    assert not _some_fail(_lm_head_pins())


def test_lm_head_highest_id_tie_is_caught(monkeypatch):
    import oracle

    def last_max(hidden, weight, nodes=None):
        z = oracle.lm_head_logits(hidden, weight)
        return (z.shape[1] - 1 - np.argmax(z[:, ::-1], axis=1)).astype(np.int32)
    monkeypatch.setattr(oracle, "lm_head_argmax", last_max)
    assert _some_fail(_lm_head_pins())


def test_lm_head_dropped_last_feature_is_caught(monkeypatch):
    import oracle
    real = oracle.lm_head_logits
    monkeypatch.setattr(oracle, "lm_head_logits",
                        lambda h, w: real(np.asarray(h)[:, :-1], np.asarray(w)[:, :-1]))
    assert _some_fail(_lm_head_pins())


def test_lm_head_argmin_is_caught(monkeypatch):
    import oracle
    monkeypatch.setattr(oracle, "lm_head_argmax",
                        lambda h, w, nodes=None: np.argmin(oracle.lm_head_logits(h, w), axis=1))
    assert _some_fail(_lm_head_pins())


# ------------------------------------------------------------ losslessness

def _lossless_fails():
    from tests import test_oracle_lossless as ll
    try:
        for plant in (0.7, 1.0):
            ll.test_speculative_equals_autoregressive(1, 12, plant)
    except AssertionError:
        return True
    return False


def test_lossless_pin_passes_unmutated():
    assert not _lossless_fails()


def test_lossless_catches_parent_only_mask(monkeypatch):
    def two_levels(parent, i):
        return [i] + ([parent[i]] if parent[i] >= 0 else [])
    monkeypatch.setattr(tv, "ancestors_inclusive", two_levels)
    assert _lossless_fails()


def test_lossless_catches_compaction_from_the_wrong_row(monkeypatch):
    real = tv.kv_compact

    def shifted(cache, prefix_len, new_pos):
        return real(cache, prefix_len + 1, new_pos)
    monkeypatch.setattr(tv, "kv_compact", shifted)
    import oracle
    monkeypatch.setattr(oracle, "kv_compact", shifted)
    assert _lossless_fails()


def test_lossless_catches_a_wrong_bonus_token(monkeypatch):
    real = tv.accepted_tokens
    monkeypatch.setattr(tv, "accepted_tokens",
                        lambda path, am, token: real(path, am, token)[:-1] + [int(token[path[-1]])])
    assert _lossless_fails()
