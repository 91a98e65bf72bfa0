"""The oracle's whole layer against a hand-worked example (CPU only).

tests/golden/tiny_layer_example.json writes out, by hand from the Treebeard
page's "Routing math", "Routed expert computation", "Shared expert
computation" and "Pseudocode", every intermediate of a 2-token layer with
3 experts, top-2, a shared expert and a residual: logits, softmax
probabilities, ids, renormalised weights, shared gate, routed and shared
outputs and the layer output. Its 4-bit twin stores the same routed banks as
4-bit affine group-64 codes (two groups per gate/up row, different scale and
min per group), so the oracle's bank lookup is pinned as well.

The planted-mistake tests show what the example tells apart: alpha paired
with the other slot, routing on r_attn instead of x, and a 4-bit bank read
with scale and min swapped each change the result beyond the tolerance.
"""
import json
import os

import numpy as np
import pytest

import moe_inputs as mi
import oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden", "tiny_layer_example.json")
TOL = 1e-12


@pytest.fixture(scope="module")
def g():
    with open(GOLD) as f:
        return json.load(f)


def _shape(g, **kw):
    base = dict(d_model=g["d_model"], n_experts=g["n_experts"], top_k=g["top_k"],
                d_ff=g["d_ff"], d_ff_shared=g["d_ff_shared"], renorm_clamp=g["renorm_clamp"],
                act_dtype="f32", expert_dtype="f32")
    base.update(kw)
    return mi.MoEShape("golden_tiny", 90, **base)


def _layer(g):
    return {k: np.asarray(v, np.float32) for k, v in g["inputs"].items()}


def _close(got, want):
    return np.max(np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))) <= TOL


def test_every_intermediate_matches_the_hand_worked_layer(g):
    ref = orc.moe_layer_forward(_layer(g), _shape(g))
    want = g["expected"]
    assert _close(ref["logits"], want["logits"])
    assert _close(ref["score"], want["p"])
    assert ref["ids"].tolist() == want["ids"]
    assert _close(ref["weights"], want["weights"])
    assert _close(ref["s_shared"], want["s_shared"])
    assert _close(ref["y_routed"], want["y_routed"])
    assert _close(ref["y_shared"], want["y_shared"])
    assert _close(ref["out"], want["out"])


def test_experts_half_alone_matches_the_hand_worked_layer(g):
    want = g["expected"]
    ids = np.asarray(want["ids"], np.int32)
    w = np.asarray(want["weights"])
    ref = orc.moe_experts_forward(_layer(g), _shape(g), ids, w)
    assert _close(ref["out"], want["out"])
    # the shared gate given instead of computed
    ref2 = orc.moe_experts_forward(_layer(g), _shape(g), ids, w, np.asarray(want["s_shared"]))
    assert _close(ref2["out"], want["out"])


def test_planted_mistakes_are_caught(g):
    want = g["expected"]
    L, shape = _layer(g), _shape(g)
    ids = np.asarray(want["ids"], np.int32)
    w = np.asarray(want["weights"])
    # alpha paired with the other slot's expert
    swapped = orc.moe_experts_forward(L, shape, ids, w[:, ::-1].copy())
    assert not _close(swapped["out"], want["out"])
    # the router fed the attention residual instead of x
    wrong_in = dict(L, x=L["r_attn"].copy())
    z = orc.router_logits(orc.to_f64(wrong_in["x"], "f32"), orc.to_f64(L["W_router"], "f32"))
    assert orc.route_tokens(z, shape)["ids"].tolist() != want["ids"]
    # a transposed router does not even have the stored shape
    with pytest.raises(ValueError):
        orc.router_logits(orc.to_f64(L["x"], "f32"), orc.to_f64(L["W_router"], "f32").T)


# ----------------------------------------------------------------------------
# 4-bit twin
# ----------------------------------------------------------------------------
def _bf16(v):
    bits = np.asarray(v, np.float32).view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value must be exact in bf16"
    return (bits >> 16).astype(np.uint16)


def _pack(codes):
    """codes uint8 [..., K] in 0..15 -> [..., K/2], even element low nibble."""
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _q4_layer(g):
    tw = g["q4_twin"]
    D, I = tw["d_model"], tw["d_ff"]
    pos = tw["pos"]
    d, i_n = g["d_model"], g["d_ff"]
    inp = g["inputs"]

    def pad_d(v):                      # [..., d] -> [..., D] at pos
        v = np.asarray(v, np.float64)
        out = np.zeros(v.shape[:-1] + (D,))
        out[..., pos] = v
        return out

    L = {"x": pad_d(inp["x"]).astype(np.float32),
         "r_attn": pad_d(inp["r_attn"]).astype(np.float32),
         "W_router": pad_d(inp["W_router"]).astype(np.float32),
         "w_shared": pad_d(inp["w_shared"]).astype(np.float32),
         "Ws_gate": pad_d(inp["Ws_gate"]).astype(np.float32),
         "Ws_up": pad_d(inp["Ws_up"]).astype(np.float32)}
    wsd = np.zeros((D, g["d_ff_shared"]))
    wsd[pos] = np.asarray(inp["Ws_down"], np.float64)
    L["Ws_down"] = wsd.astype(np.float32)
    g0, g1 = tw["gateup_groups"]
    for bank in ("W_gate", "W_up"):
        w = np.zeros((g["n_experts"], I, D))
        w[:, :i_n, :] = pad_d(inp[bank])
        sc = np.empty(w.shape[:-1] + (2,))
        mn = np.empty_like(sc)
        sc[..., 0], mn[..., 0] = g0["scale"], g0["min"]
        sc[..., 1], mn[..., 1] = g1["scale"], g1["min"]
        codes = (w - np.repeat(mn, 64, axis=-1)) / np.repeat(sc, 64, axis=-1)
        assert np.all(codes == np.round(codes)) and codes.min() >= 0 and codes.max() <= 15
        L[bank + "_q"] = _pack(codes.astype(np.uint8))
        L[bank + "_scale"], L[bank + "_min"] = _bf16(sc), _bf16(mn)
    dn = tw["down_group"]
    w = np.zeros((g["n_experts"], D, I))
    w[:, pos, :i_n] = np.asarray(inp["W_down"], np.float64)
    codes = (w - dn["min"]) / dn["scale"]
    assert np.all(codes == np.round(codes)) and codes.min() >= 0 and codes.max() <= 15
    L["W_down_q"] = _pack(codes.astype(np.uint8))
    L["W_down_scale"] = _bf16(np.full((g["n_experts"], D, 1), dn["scale"]))
    L["W_down_min"] = _bf16(np.full((g["n_experts"], D, 1), dn["min"]))
    return L


def _q4_shape(g):
    tw = g["q4_twin"]
    return _shape(g, d_model=tw["d_model"], d_ff=tw["d_ff"], expert_dtype="q4")


def test_q4_twin_bytes_match_the_hand_packed_ones(g):
    L = _q4_layer(g)
    ex = g["q4_twin"]["example_bytes"]
    assert int(L["W_up_q"][0][0][0]) == ex["W_up[0][0][0]"]
    assert int(L["W_up_q"][0][0][32]) == ex["W_up[0][0][32]"]
    assert int(L["W_gate_q"][1][1][32]) == ex["W_gate[1][1][32]"]
    assert int(L["W_gate_q"][1][1][0]) == ex["W_gate[1][1][0]"]


def test_q4_twin_matches_the_hand_worked_layer(g):
    tw = g["q4_twin"]
    ref = orc.moe_layer_forward(_q4_layer(g), _q4_shape(g))
    want = g["expected"]
    assert ref["ids"].tolist() == want["ids"]
    assert _close(ref["weights"], want["weights"])
    out = np.zeros((g["T"], tw["d_model"]))
    out[:, tw["pos"]] = np.asarray(want["out"])
    assert _close(ref["out"], out)


def test_q4_twin_scale_and_min_swapped_is_caught(g):
    L = _q4_layer(g)
    for bank in ("W_gate", "W_up", "W_down"):
        L[bank + "_scale"], L[bank + "_min"] = L[bank + "_min"], L[bank + "_scale"]
    ref = orc.moe_layer_forward(L, _q4_shape(g))
    tw = g["q4_twin"]
    out = np.zeros((g["T"], tw["d_model"]))
    out[:, tw["pos"]] = np.asarray(g["expected"]["out"])
    assert not _close(ref["out"], out)


def test_selection_weights_of_other_selections(g):
    """The weight step applied to a selection the rule did not make (how a
    near-tied token's alternative is weighted): token 0's logits (2, 1, 0)
    with experts {0, 2} give (e^2, 1)/(e^2 + 1) = (sig(2), sig(-2)), with
    {1, 2} (e, 1)/(e + 1) = (sig(1), sig(-1)); the rule's own selection gives
    the weights route_tokens returns."""
    shape = _shape(g)
    z = np.asarray(g["expected"]["logits"][0], np.float64)
    s1, sm1 = g["expected"]["weights"][0]
    s2, sm2 = g["expected"]["weights"][1]
    assert _close(orc.selection_weights(z, [0, 2], shape), [s2, sm2])
    assert _close(orc.selection_weights(z, [1, 2], shape), [s1, sm1])
    r = orc.route_tokens(np.asarray(g["expected"]["logits"], np.float64), shape)
    for t in range(2):
        assert _close(orc.selection_weights(r["logits"][t], r["ids"][t], shape), r["weights"][t])


def test_selection_weights_sigmoid_family():
    """Edge0 "Sigmoid group top-k": raw scores of the selection, no bias,
    normalised, times routed_scaling. Logits (ln 3, 0, -ln 3, 0) have sigmoid
    scores (3/4, 1/2, 1/4, 1/2); selecting {0, 1} gives (3/5, 2/5) * 2.5 =
    (1.5, 1.0), selecting {1, 2} gives (2/3, 1/3) * 2.5, whatever the bias."""
    shape = mi.TINY_F32.with_(router="sigmoid_group", n_experts=4, top_k=2, n_group=2,
                              topk_group=1, routed_scaling=2.5)
    z = np.array([np.log(3.0), 0.0, -np.log(3.0), 0.0])
    bias = np.array([0.0, 0.3, -0.2, 0.1])
    assert np.max(np.abs(orc.selection_weights(z, [0, 1], shape, bias) - [1.5, 1.0])) <= 1e-15
    assert np.max(np.abs(orc.selection_weights(z, [1, 2], shape) - [5 / 3, 5 / 6])) <= 1e-15
