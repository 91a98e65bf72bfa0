"""The routing comparison used by the GPU parity tests, checked on CPU with
hand-made oracle scores (no GPU): exact where the oracle's ranking has a
clear gap, any order inside a run of near-equal scores, and near-tie tokens
accepted only with valid choices (k distinct ids, only from groups that may
be kept, carrying the weights the oracle's rule gives that selection)."""
import numpy as np
import pytest

import moe_inputs as mi
import oracle as orc
from gpu_util import check_routing, routing_alternatives

SHAPE = mi.TINY_F32.with_(n_experts=6, top_k=3)


def _ref(score, ids):
    """Oracle-shaped routing of one softmax token whose probabilities are
    `score` (logits log(score), so softmax(logits) = score / sum(score))."""
    score = np.asarray(score, np.float64)
    z = np.log(score)
    return {"ids": np.array([ids]), "score": np.array([score / score.sum()]),
            "weights": np.array([orc.selection_weights(z, ids, SHAPE)]),
            "group_score": np.zeros((1, 1)), "logits": np.array([z]), "bias": None}


def test_clear_gaps_need_exact_order():
    score = [0.40, 0.25, 0.15, 0.10, 0.06, 0.04]
    ref = _ref(score, [0, 1, 2])
    w = ref["weights"]
    assert check_routing(np.array([[0, 1, 2]]), w, ref, SHAPE) == (0, {})
    with pytest.raises(AssertionError):
        check_routing(np.array([[1, 0, 2]]), w[:, [1, 0, 2]], ref, SHAPE)
    with pytest.raises(AssertionError):
        check_routing(np.array([[0, 1, 3]]), w, ref, SHAPE)


def test_tie_run_accepts_any_order_inside_it():
    # slots 1 and 2 nearly tie; the gap after slot 2 is large
    score = [0.40, 0.20, 0.20 - 1e-8, 0.10, 0.06, 0.04 + 1e-8]
    ref = _ref(score, [0, 1, 2])
    w = ref["weights"]
    assert check_routing(np.array([[0, 2, 1]]), w[:, [0, 2, 1]], ref, SHAPE) == (0, {})
    with pytest.raises(AssertionError):
        check_routing(np.array([[2, 0, 1]]), w[:, [2, 0, 1]], ref, SHAPE)


def test_near_tie_at_the_cut_accepts_only_valid_choices():
    # the 3rd and 4th scores tie: either may be selected, not the 5th
    score = [0.40, 0.25, 0.12, 0.12 - 1e-7, 0.07, 0.04]
    ref = _ref(score, [0, 1, 2])
    z = ref["logits"][0]
    w_alt = orc.selection_weights(z, [0, 1, 3], SHAPE)[None, :]
    near, alts = check_routing(np.array([[0, 1, 3]]), w_alt, ref, SHAPE)
    assert near == 1 and alts == {0: [0, 1, 3]}
    with pytest.raises(AssertionError):
        check_routing(np.array([[0, 1, 4]]), w_alt, ref, SHAPE)


def test_near_tie_rejects_a_duplicated_id():
    score = [0.40, 0.25, 0.12, 0.12 - 1e-7, 0.07, 0.04]
    ref = _ref(score, [0, 1, 2])
    w = ref["weights"]
    with pytest.raises(AssertionError, match="duplicate"):
        check_routing(np.array([[0, 2, 2]]), w, ref, SHAPE)


def test_near_tie_rejects_dropping_a_clear_winner():
    # both tied ids chosen but the clear first choice left out
    score = [0.40, 0.25, 0.12, 0.12 - 1e-7, 0.07, 0.04]
    ref = _ref(score, [0, 1, 2])
    z = ref["logits"][0]
    w = orc.selection_weights(z, [1, 2, 3], SHAPE)[None, :]
    with pytest.raises(AssertionError):
        check_routing(np.array([[1, 2, 3]]), w, ref, SHAPE)


def test_near_tie_alternative_needs_its_own_weights():
    # the alternative set is valid, but its weights are the oracle's set's
    score = [0.40, 0.25, 0.12, 0.12 - 1e-4 / 2, 0.07, 0.04]
    ref = _ref(score, [0, 1, 2])
    z = ref["logits"][0]
    own = orc.selection_weights(z, [0, 1, 3], SHAPE)[None, :]
    assert check_routing(np.array([[0, 1, 3]]), own, ref, SHAPE)[0] == 1
    # 0.12 vs 0.12 - 5e-5 changes the renormalised weights by ~2e-5 > 1e-5
    with pytest.raises(AssertionError):
        check_routing(np.array([[0, 1, 3]]), ref["weights"], ref, SHAPE)


GROUPS = mi.TINY_F32.with_(router="sigmoid_group", n_experts=8, top_k=2, n_group=4,
                           topk_group=2, routed_scaling=2.5)


def _group_ref(z, bias):
    z = np.asarray(z, np.float64)
    b = np.asarray(bias, np.float64)
    return orc.route_tokens(z[None, :], GROUPS, b)


def test_group_near_tie_rejects_an_id_of_a_clearly_dropped_group():
    # groups of two experts; selection scores s + b. Group 3 loses the group
    # stage by far; inside the kept groups the 2nd and 3rd experts tie.
    s = np.array([0.9, 0.1, 0.7, 0.1, 0.7 - 1e-6, 0.1, 0.2, 0.15])
    bias = np.zeros(8)
    z = np.log(s / (1 - s))
    ref = _group_ref(z, bias)
    assert ref["ids"][0].tolist() == [0, 2]
    valid = routing_alternatives(ref, GROUPS, 0)
    assert frozenset([0, 4]) in valid and frozenset([0, 6]) not in valid
    w_ok = orc.selection_weights(z, [0, 4], GROUPS)[None, :]
    near, alts = check_routing(np.array([[0, 4]]), w_ok, ref, GROUPS)
    assert near == 1 and alts == {0: [0, 4]}
    w_bad = orc.selection_weights(z, [0, 6], GROUPS)[None, :]
    with pytest.raises(AssertionError):
        check_routing(np.array([[0, 6]]), w_bad, ref, GROUPS)


def test_group_stage_near_tie_allows_either_group():
    # groups 1 and 2 tie at the group stage (group score = sum of both
    # members); either may be kept, and its best expert is then selected
    s = np.array([0.9, 0.1, 0.5, 0.3, 0.3, 0.5 - 1e-6, 0.05, 0.05])
    bias = np.zeros(8)
    z = np.log(s / (1 - s))
    ref = _group_ref(z, bias)
    valid = routing_alternatives(ref, GROUPS, 0)
    assert frozenset([0, 2]) in valid and frozenset([0, 5]) in valid
    w = orc.selection_weights(z, [0, 5], GROUPS)[None, :]
    assert check_routing(np.array([[0, 5]]), w, ref, GROUPS)[0] == 1
