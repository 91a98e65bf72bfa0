"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something the pages or the mathematics fix:
worked examples built by hand (tests/golden), closed forms, identities the
pages state, brute-force enumeration on tiny inputs, and special cases that
reduce to library routines (numpy sorts, scipy's logistic, torch fp64 linear
algebra). A mistake such as a dropped term, a flipped sign, a wrong index or a
transposed operand in the oracle fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import moe_inputs as mi
import oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# storage encodings
# ----------------------------------------------------------------------------
def test_bf16_decode_exact_values():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x4049, 0x3800], np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0, 3.140625, 2.0 ** -15]
    assert orc.bf16_bits_to_f64(bits).tolist() == want


def test_generator_bf16_rounding_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7
    vals = np.array([one + ulp / 2, one + 1.5 * ulp, one + 0.49 * ulp, -one - 0.51 * ulp],
                    np.float32)
    got = mi.f32_to_bf16_bits(vals)
    assert got.tolist() == [0x3F80, 0x3F82, 0x3F80, 0xBF81]


def test_q4_dequant_golden_example():
    g = _gold("q4_affine_g64_example.json")
    q = np.array(g["packed"], np.uint8)[None, :]
    sc = np.array(g["scale_bits"], np.uint16)[None, :]
    mn = np.array(g["min_bits"], np.uint16)[None, :]
    w = orc.dequant_q4_affine_g64(q, sc, mn)
    assert w.shape == (1, 128)
    assert w[0].tolist() == g["expected"]


def test_q4_generator_roundtrip_within_half_step():
    rng = np.random.default_rng(5)
    w = rng.standard_normal((3, 256)).astype(np.float32) * 0.02
    q, s, m = mi.quantize_q4_affine_g64(w)
    deq = orc.dequant_q4_affine_g64(q, s, m)
    step = np.repeat(orc.bf16_bits_to_f64(s), 64, axis=1)
    # bf16 rounding of min/scale adds at most a few ulps on top of half a step
    assert np.all(np.abs(deq - w) <= 0.5 * step + 2e-4)


# ----------------------------------------------------------------------------
# elementwise closed forms
# ----------------------------------------------------------------------------
def test_sigmoid_and_silu_closed_forms():
    v = np.linspace(-9, 9, 37)
    assert orc.sigmoid(0.0) == 0.5
    np.testing.assert_allclose(orc.sigmoid(v), scipy.special.expit(v), rtol=1e-15, atol=0)
    np.testing.assert_allclose(orc.sigmoid(-v), 1 - orc.sigmoid(v), atol=1e-15)
    assert orc.silu(0.0) == 0.0
    # silu(x) - silu(-x) = x (sigma(x) + sigma(-x) = 1)
    np.testing.assert_allclose(orc.silu(v) - orc.silu(-v), v, atol=1e-14)
    np.testing.assert_allclose(orc.silu(v), v * scipy.special.expit(v), rtol=1e-15)


def test_softmax_closed_form_and_shift():
    z = np.log(np.array([1.0, 2.0, 3.0]))
    np.testing.assert_allclose(orc.softmax(z), [1 / 6, 2 / 6, 3 / 6], rtol=1e-15)
    np.testing.assert_allclose(orc.softmax(z + 100.0), [1 / 6, 2 / 6, 3 / 6], rtol=1e-14)
    np.testing.assert_allclose(orc.softmax(z), scipy.special.softmax(z), rtol=1e-15)


# ----------------------------------------------------------------------------
# top-k
# ----------------------------------------------------------------------------
def _brute_topk(scores, k):
    """All k-subsets; the best has the largest sum, then the smallest sorted
    index tuple (lowest index wins ties). Returned in descending score order,
    equal scores lower index first."""
    best = None
    for sub in itertools.combinations(range(len(scores)), k):
        key = (-sum(scores[i] for i in sub), sub)
        if best is None or key < best:
            best = key
    return sorted(best[1], key=lambda i: (-scores[i], i))


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    E, k = 10, 4
    s = rng.standard_normal(E)
    if seed % 2:  # plant exact ties, including at the k-th boundary
        s[[1, 3, 7]] = s[5]
    assert orc.topk_desc(s, k).tolist() == _brute_topk(list(s), k)


def test_topk_lowest_index_wins_ties():
    s = np.array([3.0, 1.0, 3.0, 3.0])
    assert orc.topk_desc(s, 2).tolist() == [0, 2]
    assert orc.topk_desc(np.zeros(5), 3).tolist() == [0, 1, 2]


# ----------------------------------------------------------------------------
# softmax top-k routing ("Routing math")
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("E,k", [(16, 4), (256, 8), (8, 2), (5, 5)])
def test_softmax_renorm_equals_softmax_over_selected_logits(E, k):
    rng = np.random.default_rng(E * 31 + k)
    for _ in range(20):
        z = rng.normal(0, 1.5, E)
        ids, alpha, p = orc.softmax_topk_route(z, k)
        # identity stated on the page: the global denominator cancels
        direct = np.exp(z[ids]) / np.sum(np.exp(z[ids]))
        np.testing.assert_allclose(alpha, direct, rtol=1e-13, atol=1e-16)
        assert abs(alpha.sum() - 1.0) < 1e-14
        # ranking on p equals ranking on z (softmax is monotone)
        assert set(ids.tolist()) == set(np.argsort(-z, kind="stable")[:k].tolist())
        # the clamp cannot bind: selected mass >= k/E >= 2^-14
        assert p[ids].sum() >= k / E - 1e-15


def test_renorm_clamp_binds_on_tiny_mass():
    p = np.array([2.0 ** -20, 2.0 ** -19])
    a = orc.renormalise_clamped(p, 2.0 ** -14)
    assert a.tolist() == [2.0 ** -6, 2.0 ** -5]
    b = orc.renormalise_clamped(np.array([0.25, 0.5]), 2.0 ** -14)
    np.testing.assert_allclose(b, [1 / 3, 2 / 3], rtol=1e-15)


def test_softmax_route_ids_descending_order():
    z = np.array([0.1, 2.0, -1.0, 1.5, 0.7])
    ids, alpha, _ = orc.softmax_topk_route(z, 3)
    assert ids.tolist() == [1, 3, 4]
    assert np.all(np.diff(alpha) < 0)


# ----------------------------------------------------------------------------
# sigmoid group top-k ("Sigmoid group top-k")
# ----------------------------------------------------------------------------
def _brute_group_route(z, bias, n_group, topk_group, k, rs):
    E = len(z)
    gs = E // n_group
    s = scipy.special.expit(z)
    sel = s + bias
    # group score: the largest sum over any two members
    gscore = []
    for g in range(n_group):
        mem = sel[g * gs:(g + 1) * gs]
        gscore.append(max(mem[i] + mem[j] for i, j in itertools.combinations(range(gs), 2)))
    kept = _brute_topk(gscore, topk_group)
    cand = [e for g in sorted(kept) for e in range(g * gs, (g + 1) * gs)]
    best = None
    for sub in itertools.combinations(cand, k):
        key = (-sum(sel[i] for i in sub), tuple(sorted(sub)))
        if best is None or key < best:
            best = key
    ids = sorted(best[1], key=lambda i: (-sel[i], i))
    w = s[ids] / s[ids].sum() * rs
    return ids, w, sorted(kept)


@pytest.mark.parametrize("seed", range(8))
def test_sigmoid_group_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    E, n_group, topk_group, k, rs = 16, 4, 2, 4, 2.5
    z = rng.normal(0, 1.0, E)
    bias = rng.uniform(-0.3, 0.3, E)
    ids, w, sel, gsc, kept = orc.sigmoid_group_topk_route(z, bias, n_group, topk_group, k, rs)
    bids, bw, bkept = _brute_group_route(z, bias, n_group, topk_group, k, rs)
    assert ids.tolist() == bids
    assert sorted(kept.tolist()) == bkept
    np.testing.assert_allclose(w, bw, rtol=1e-14)
    assert abs(w.sum() - rs) < 1e-13


def test_sigmoid_group_reduces_to_plain_topk():
    rng = np.random.default_rng(7)
    E, k = 32, 6
    z = rng.normal(0, 1, E)
    bias = rng.uniform(-0.1, 0.1, E)
    # every group kept: plain top-k of the selection score
    ids, w, sel, _, _ = orc.sigmoid_group_topk_route(z, bias, 4, 4, k, 1.0)
    s = scipy.special.expit(z)
    assert ids.tolist() == np.argsort(-(s + bias), kind="stable")[:k].tolist()
    # one group and no bias: textbook top-k of sigmoid(z), i.e. of z
    ids1, w1, _, _, _ = orc.sigmoid_group_topk_route(z, None, 1, 1, k, 1.0)
    assert ids1.tolist() == np.argsort(-z, kind="stable")[:k].tolist()
    np.testing.assert_allclose(w1, s[ids1] / s[ids1].sum(), rtol=1e-15)


def test_bias_selects_but_does_not_weight():
    rng = np.random.default_rng(11)
    E, k = 16, 4
    z = rng.normal(0, 1, E)
    bias = np.zeros(E)
    ids0, w0, *_ = orc.sigmoid_group_topk_route(z, bias, 4, 2, k, 2.5)
    # a small bias change that leaves the selection unchanged leaves weights unchanged
    bias2 = bias.copy()
    bias2[ids0] += 1e-3
    ids2, w2, *_ = orc.sigmoid_group_topk_route(z, bias2, 4, 2, k, 2.5)
    assert set(ids2.tolist()) == set(ids0.tolist())
    d0 = dict(zip(ids0.tolist(), w0.tolist()))
    for i, w in zip(ids2.tolist(), w2.tolist()):
        assert abs(d0[i] - w) < 1e-15
    # a large bias forces an expert in; its weight uses the raw sigmoid score
    loser = int(np.argmin(z))
    bias3 = np.zeros(E)
    bias3[loser] = 10.0
    ids3, w3, *_ = orc.sigmoid_group_topk_route(z, bias3, 4, 2, k, 2.5)
    assert ids3[0] == loser
    s = scipy.special.expit(z)
    np.testing.assert_allclose(w3[0], s[loser] / s[ids3].sum() * 2.5, rtol=1e-14)


def test_only_kept_groups_contribute():
    rng = np.random.default_rng(12)
    E, n_group, topk_group, k = 128, 8, 4, 8
    for _ in range(50):
        z = rng.normal(0, 1, E)
        bias = rng.uniform(-0.1, 0.1, E)
        ids, w, sel, gsc, kept = orc.sigmoid_group_topk_route(z, bias, n_group, topk_group, k, 2.5)
        groups = set((ids // (E // n_group)).tolist())
        assert groups <= set(kept.tolist())
        assert len(kept) == topk_group
        # kept groups outrank every dropped group
        dropped = [g for g in range(n_group) if g not in kept]
        assert min(gsc[kept]) >= max(gsc[dropped])


# ----------------------------------------------------------------------------
# experts and the layer
# ----------------------------------------------------------------------------
def _tiny_shape(E=1, k=1, d=16, I=8, Is=8):
    return mi.MoEShape("t", 99, d_model=d, n_experts=E, top_k=k, d_ff=I, d_ff_shared=Is,
                       act_dtype="f32", expert_dtype="f32")


def _tiny_layer(shape, T, seed=0):
    rng = np.random.default_rng(seed)
    d, E, I, Is = shape.d_model, shape.n_experts, shape.d_ff, shape.d_ff_shared
    f = lambda *s: (rng.standard_normal(s) * 0.3).astype(np.float32)
    L = {"x": f(T, d), "r_attn": f(T, d), "W_router": f(E, d),
         "W_gate": f(E, I, d), "W_up": f(E, I, d), "W_down": f(E, d, I)}
    if Is:
        L.update({"w_shared": f(d), "Ws_gate": f(Is, d), "Ws_up": f(Is, d), "Ws_down": f(d, Is)})
    return L


def _torch_swiglu(x, Wg, Wu, Wd):
    F = torch.nn.functional
    return F.linear(F.silu(F.linear(x, Wg)) * F.linear(x, Wu), Wd)


def test_dense_reduction_matches_torch_fp64():
    """E = 1, k = 1: the layer is a dense SwiGLU FFN plus the gated shared
    expert plus the residual (alpha = 1 exactly)."""
    shape = _tiny_shape(E=1, k=1, d=16, I=8, Is=12)
    L = _tiny_layer(shape, T=5)
    res = orc.moe_layer_forward(L, shape)
    t = {k_: torch.from_numpy(v.astype(np.float64)) for k_, v in L.items()}
    routed = _torch_swiglu(t["x"], t["W_gate"][0], t["W_up"][0], t["W_down"][0])
    s = torch.sigmoid(t["x"] @ t["w_shared"])
    shared = s[:, None] * _torch_swiglu(t["x"], t["Ws_gate"], t["Ws_up"], t["Ws_down"])
    want = t["r_attn"] + routed + shared
    np.testing.assert_allclose(res["out"], want.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["s_shared"], s.numpy(), rtol=1e-14)
    assert np.all(res["weights"] == 1.0)


def test_identical_experts_make_routing_irrelevant():
    shape = _tiny_shape(E=6, k=3, d=12, I=5, Is=0)
    L = _tiny_layer(shape, T=4, seed=3)
    for b in ("W_gate", "W_up", "W_down"):
        L[b][:] = L[b][0]
    res = orc.moe_layer_forward(L, shape)
    t = {k_: torch.from_numpy(v.astype(np.float64)) for k_, v in L.items()}
    want = t["r_attn"] + _torch_swiglu(t["x"], t["W_gate"][0], t["W_up"][0], t["W_down"][0])
    np.testing.assert_allclose(res["out"], want.numpy(), rtol=1e-12, atol=1e-12)


def test_shared_gate_half_at_zero_and_branch_split():
    shape = _tiny_shape(E=4, k=2, d=10, I=6, Is=6)
    L = _tiny_layer(shape, T=3, seed=4)
    L["w_shared"][:] = 0
    res = orc.moe_layer_forward(L, shape)
    assert np.all(res["s_shared"] == 0.5)
    np.testing.assert_allclose(res["out"], L["r_attn"] + res["y_routed"] + res["y_shared"],
                               atol=1e-14)
    # zero routed banks: only the shared branch and the residual remain
    for b in ("W_gate", "W_up", "W_down"):
        L[b][:] = 0
    res0 = orc.moe_layer_forward(L, shape)
    np.testing.assert_allclose(res0["y_routed"], 0.0)
    np.testing.assert_allclose(res0["out"], L["r_attn"] + res0["y_shared"], atol=1e-14)


def test_token_permutation_equivariance():
    shape = _tiny_shape(E=8, k=3, d=12, I=5, Is=4)
    L = _tiny_layer(shape, T=7, seed=5)
    res = orc.moe_layer_forward(L, shape)
    perm = np.random.default_rng(1).permutation(7)
    L2 = dict(L)
    L2["x"] = L["x"][perm]
    L2["r_attn"] = L["r_attn"][perm]
    res2 = orc.moe_layer_forward(L2, shape)
    np.testing.assert_allclose(res2["out"], res["out"][perm], atol=1e-13)
    assert np.array_equal(res2["ids"], res["ids"][perm])


def test_expert_permutation_invariance():
    shape = _tiny_shape(E=8, k=3, d=12, I=5, Is=4)
    L = _tiny_layer(shape, T=6, seed=6)
    res = orc.moe_layer_forward(L, shape)
    pi = np.random.default_rng(2).permutation(8)   # new expert j = old expert pi[j]
    L2 = dict(L)
    for b in ("W_router", "W_gate", "W_up", "W_down"):
        L2[b] = L[b][pi]
    res2 = orc.moe_layer_forward(L2, shape)
    np.testing.assert_allclose(res2["out"], res["out"], atol=1e-13)
    assert np.array_equal(pi[res2["ids"]], res["ids"])


def test_token_sample_equals_full_rows():
    shape = _tiny_shape(E=8, k=2, d=12, I=5, Is=4)
    L = _tiny_layer(shape, T=9, seed=8)
    full = orc.moe_layer_forward(L, shape)
    part = orc.moe_layer_forward(L, shape, tokens=[7, 2])
    np.testing.assert_array_equal(part["out"], full["out"][[7, 2]])
    np.testing.assert_array_equal(part["ids"], full["ids"][[7, 2]])


def test_sigmoid_layer_weights_sum_to_scaling():
    shape = mi.DEEPSEEK_GROUP.with_(d_model=32, n_experts=16, n_group=4, topk_group=2,
                                    top_k=4, d_ff=8, d_ff_shared=8, act_dtype="f32",
                                    expert_dtype="f32")
    L = _tiny_layer(shape, T=5, seed=9)
    L["expert_bias"] = np.random.default_rng(3).uniform(-0.1, 0.1, 16).astype(np.float32)
    res = orc.moe_layer_forward(L, shape)
    np.testing.assert_allclose(res["weights"].sum(axis=1), 2.5, rtol=1e-14)


# ----------------------------------------------------------------------------
# bucketing ("Intel SYCL path" counting and packing)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("T,k,E", [(0, 4, 16), (1, 8, 256), (37, 4, 16), (300, 8, 64)])
def test_bucket_matches_stable_sort(T, k, E):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int32)
    b = orc.bucket(ids, E)
    flat = ids.reshape(-1)
    assert b["counts"].tolist() == np.bincount(flat, minlength=E).tolist()
    assert b["offsets"][0] == 0 and b["offsets"][-1] == T * k
    assert b["perm"].tolist() == np.argsort(flat, kind="stable").tolist()
    assert b["active"].tolist() == np.nonzero(np.bincount(flat, minlength=E))[0].tolist()
    if T:
        assert np.array_equal(b["perm"][b["pos"]], np.arange(T * k))


# ----------------------------------------------------------------------------
# the shapes on the pages
# ----------------------------------------------------------------------------
def test_presets_match_the_pages():
    g = _gold("model_constants.json")
    for name, preset in (("qwen36", mi.QWEN36), ("qwen36", mi.QWEN36_PREFILL_SKEW),
                         ("deepseek_group", mi.DEEPSEEK_GROUP), ("mixtral", mi.MIXTRAL)):
        for key, val in g[name].items():
            assert getattr(preset, key) == val, (preset.name, key)


def test_generator_is_deterministic_and_shaped():
    s = mi.TINY_F32
    a = mi.make_layer(s, 32)
    b = mi.make_layer(s, 32)
    for key in a:
        assert np.array_equal(a[key], b[key])
    x = a["x"].astype(np.float64)
    np.testing.assert_allclose(np.sqrt((x * x).mean(axis=1)), 1.0, rtol=1e-5)
    assert abs(a["W_gate"].std() - 0.02) < 1e-3
    assert a["W_gate"].shape == (16, 64, 256) and a["W_down"].shape == (16, 256, 64)


def test_skew_makes_imbalanced_histogram():
    s = mi.QWEN36_PREFILL_SKEW.with_(d_model=256, n_experts=64, d_ff=8, d_ff_shared=8)
    L = mi.make_layer(s, 512)
    res = orc.route_tokens(orc.router_logits(orc.to_f64(L["x"], "bf16"),
                                             orc.to_f64(L["W_router"], "bf16")), s)
    counts = np.bincount(res["ids"].reshape(-1), minlength=64)
    assert counts.max() > 3 * counts.mean()
