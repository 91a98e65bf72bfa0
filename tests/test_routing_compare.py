"""The routing comparison used by the GPU parity tests, checked on CPU with
hand-made oracle scores (no GPU): exact where the oracle's ranking has a
clear gap, any order inside a run of near-equal scores, and near-tie tokens
accepted only with valid choices."""
import numpy as np
import pytest

import moe_inputs as mi
from gpu_util import check_routing

SHAPE = mi.TINY_F32.with_(n_experts=6, top_k=3)


def _ref(score, ids):
    w = np.asarray(score)[ids] / np.sum(np.asarray(score)[ids])
    return {"ids": np.array([ids]), "weights": np.array([w]), "score": np.array([score]),
            "group_score": np.zeros((1, 1))}


def test_clear_gaps_need_exact_order():
    score = [0.40, 0.25, 0.15, 0.10, 0.06, 0.04]
    ref = _ref(score, [0, 1, 2])
    w = ref["weights"]
    assert check_routing(np.array([[0, 1, 2]]), w, ref, SHAPE) == 0
    with pytest.raises(AssertionError):
        check_routing(np.array([[1, 0, 2]]), w[:, [1, 0, 2]], ref, SHAPE)
    with pytest.raises(AssertionError):
        check_routing(np.array([[0, 1, 3]]), w, ref, SHAPE)


def test_tie_run_accepts_any_order_inside_it():
    # slots 1 and 2 nearly tie; the gap after slot 2 is large
    score = [0.40, 0.20, 0.20 - 1e-8, 0.10, 0.06, 0.04 + 1e-8]
    ref = _ref(score, [0, 1, 2])
    w = ref["weights"]
    assert check_routing(np.array([[0, 2, 1]]), w[:, [0, 2, 1]], ref, SHAPE) == 0
    with pytest.raises(AssertionError):
        check_routing(np.array([[2, 0, 1]]), w[:, [2, 0, 1]], ref, SHAPE)


def test_near_tie_at_the_cut_accepts_only_valid_choices():
    # the 3rd and 4th scores tie: either may be selected, not the 5th
    score = [0.40, 0.25, 0.12, 0.12 - 1e-7, 0.07, 0.04]
    ref = _ref(score, [0, 1, 2])
    w = ref["weights"]
    assert check_routing(np.array([[0, 1, 3]]), w, ref, SHAPE) == 1
    with pytest.raises(AssertionError):
        check_routing(np.array([[0, 1, 4]]), w, ref, SHAPE)
