"""fp64 CPU oracle for the sparse mixture-of-experts layer forward.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this module; the library itself never
does, and there is no CPU fallback through it.

It is a plain, slow, literal statement of what the layer computes, in float64,
from the exact values the GPU receives (bf16 and fp32 inputs upcast exactly,
4-bit affine weights dequantised exactly). It shares no code with the CUDA
path. Sources, by page and section:

  [P1] "How Treebeard routes Qwen3.6 MoE tokens": "The short version",
       "Routing math", "Routed expert computation", "Shared expert
       computation", "Pseudocode", "Implementation notes", and the SYCL
       counting/packing steps under "Intel SYCL path".
  [P2] Edge0 "MoE Routing and Experts": "Experts", the tier table,
       "Softmax top-k", "Sigmoid group top-k".
  [P3] Airframe MoE roadmap: "Top-K Expert Selection", "Expert Combine".

Readings adopted where the pages are silent (each is also listed with the
design notes):
  * ties in every top-k (experts and groups) go to the lower index;
  * selected ids are returned in descending score order;
  * softmax family: the renormalisation denominator is clamped below at 2^-14
    as [P1] "Routing math" states ([P2] states no clamp; for a true softmax the
    clamp can never bind since the selected mass is >= k/E);
  * sigmoid family: groups are contiguous blocks of E/n_group experts; a group
    scores the sum of its two largest selection scores (all of them when a
    group has fewer than two members); experts outside the kept groups cannot
    be selected; routed_scaling multiplies after normalisation; no clamp;
  * the shared expert's gate is the scalar sigmoid gate of [P1] "Shared expert
    computation" for every configuration that has a shared expert;
  * 4-bit affine group 64 ([P2] tier table gives only the name):
    w = scale * q + min, q in 0..15, 64 consecutive input-dim elements per
    group, the even element in the low nibble, bf16 scale and min.

Parity pins for every function live in the CPU test suite; the only part with
no external pin is absolute parity with a trained checkpoint (none exists
here).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "to_f64", "dequant_q4_affine_g64", "ExpertBanks",
    "router_logits", "softmax", "topk_desc", "renormalise_clamped",
    "softmax_topk_route", "sigmoid", "sigmoid_group_topk_route",
    "route_tokens", "selection_weights", "silu", "swiglu_expert", "shared_gate",
    "moe_layer_forward", "moe_experts_forward", "bucket",
]


# ----------------------------------------------------------------------------
# exact upcasts of the storage formats
# ----------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly: a bf16 value is the
    upper half of the fp32 value with the same bits."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array ('f32' float32 or 'bf16' uint16 bits) -> float64."""
    if dtype == "bf16":
        return bf16_bits_to_f64(a)
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def dequant_q4_affine_g64(q: np.ndarray, scale_bits: np.ndarray,
                          min_bits: np.ndarray) -> np.ndarray:
    """4-bit affine, group 64 ([P2] tier table): w = scale*q + min.

    q: uint8 [N][K/2], two codes per byte, even element in the low nibble.
    scale_bits, min_bits: bf16 bits [N][K/64]. Returns float64 [N][K].
    """
    q = np.asarray(q)
    N, half = q.shape
    K = 2 * half
    codes = np.empty((N, K), dtype=np.float64)
    codes[:, 0::2] = (q & 0x0F)
    codes[:, 1::2] = (q >> 4)
    scale = bf16_bits_to_f64(scale_bits)          # [N][K/64]
    mn = bf16_bits_to_f64(min_bits)
    group = np.arange(K) // 64                    # group of each column
    return scale[:, group] * codes + mn[:, group]


class ExpertBanks:
    """fp64 view of one layer's expert banks, converted one expert at a time.

    Banks are [E][I][d] (gate, up) and [E][d][I] (down) with the input
    dimension contiguous, as the Airframe roadmap's GGUF loader lists expert
    tensors ([n_experts, dim_out, dim_in]).
    """

    def __init__(self, layer: dict, expert_dtype: str, cache_bytes: int = 3 << 30):
        self.layer = layer
        self.dtype = expert_dtype
        self._cache = {}
        self._cache_bytes = cache_bytes

    def get(self, bank: str, e: int) -> np.ndarray:
        key = (bank, int(e))
        m = self._cache.get(key)
        if m is None:
            if self.dtype == "q4":
                m = dequant_q4_affine_g64(self.layer[bank + "_q"][e],
                                          self.layer[bank + "_scale"][e],
                                          self.layer[bank + "_min"][e])
            else:
                m = to_f64(self.layer[bank][e], self.dtype)
            held = sum(v.nbytes for v in self._cache.values())
            while self._cache and held + m.nbytes > self._cache_bytes:
                held -= self._cache.pop(next(iter(self._cache))).nbytes
            self._cache[key] = m
        return m


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------
def router_logits(x: np.ndarray, W_router: np.ndarray) -> np.ndarray:
    """[P1] "Routing math": z_t = W_router^T x_t, one logit per routed expert.
    x [T][d], W_router [E][d] (row e scores expert e) -> z [T][E]."""
    return x @ W_router.T


def softmax(z: np.ndarray) -> np.ndarray:
    """[P1] "Routing math" p_t = softmax(z_t); [P2] "computed exactly".
    The maximum is subtracted first (exact in real arithmetic)."""
    m = np.max(z)
    e = np.exp(z - m)
    return e / np.sum(e)


def topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    """TopK of [P1] "Routing math" / [P2] step 2: the indices of the k largest
    scores, largest first; equal scores are taken lower index first.
    A stable sort of the negated scores keeps equal keys in index order."""
    order = np.argsort(-np.asarray(scores, dtype=np.float64), kind="stable")
    return order[:k]


def renormalise_clamped(p_sel: np.ndarray, clamp: float) -> np.ndarray:
    """[P1] "Routing math": denom = max(sum of the selected p, 2^-14);
    alpha_i = p_i / denom."""
    denom = max(float(np.sum(p_sel)), float(clamp))
    return p_sel / denom


def softmax_topk_route(z: np.ndarray, k: int, clamp: float = 2.0 ** -14):
    """Softmax top-k rule for one token ([P1] "Routing math" and
    "Pseudocode"; [P2] "Softmax top-k"): softmax over all experts, the k
    largest probabilities, gathered and renormalised with the clamp.
    Returns (ids [k] int, alpha [k] float64, p [E] float64)."""
    p = softmax(z)
    ids = topk_desc(p, k)
    alpha = renormalise_clamped(p[ids], clamp)
    return ids, alpha, p


def sigmoid(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, dtype=np.float64)))


def sigmoid_group_topk_route(z: np.ndarray, bias, n_group: int, topk_group: int,
                             k: int, routed_scaling: float):
    """Sigmoid group top-k rule for one token ([P2] "Sigmoid group top-k"):
      1. scores = sigmoid(logits);
      2. selection score = scores + expert_bias;
      3. contiguous groups of E/n_group experts, each ranked by the sum of its
         two largest selection scores; the best topk_group groups are kept;
      4. the k largest selection scores inside the kept groups are selected;
      5. weights = the selected raw scores (no bias) normalised to sum to one,
         times routed_scaling.
    Returns (ids [k], weights [k], sel [E], group_scores [n_group],
    kept_groups [topk_group])."""
    E = z.shape[0]
    gsize = E // n_group
    s = sigmoid(z)
    b = np.zeros(E) if bias is None else np.asarray(bias, dtype=np.float64)
    sel = s + b
    group_scores = np.empty(n_group)
    for g in range(n_group):
        members = sel[g * gsize:(g + 1) * gsize]
        top2 = topk_desc(members, min(2, gsize))
        group_scores[g] = np.sum(members[top2])
    kept = topk_desc(group_scores, topk_group)
    masked = np.full(E, -np.inf)
    for g in kept:
        masked[g * gsize:(g + 1) * gsize] = sel[g * gsize:(g + 1) * gsize]
    ids = topk_desc(masked, k)
    raw = s[ids]
    weights = raw / np.sum(raw) * routed_scaling
    return ids, weights, sel, group_scores, kept


def selection_weights(z: np.ndarray, ids, shape, bias=None) -> np.ndarray:
    """The weight step of the shape's rule applied to a given selection `ids`
    of one token with logits z [E] (the last step of [P1] "Routing math" /
    [P2] "Softmax top-k": the selected probabilities renormalised with the
    clamp; of [P2] "Sigmoid group top-k": the selected raw sigmoid scores,
    no bias, normalised to one), times routed_scaling. For the oracle's own
    selection this is the weight route_tokens returns; for another valid
    selection of a near-tied token it is the weight that selection carries.
    `bias` is accepted for symmetry with the rules and never enters."""
    ids = np.asarray(ids, dtype=np.int64)
    if shape.router == "softmax":
        p = softmax(z)
        return renormalise_clamped(p[ids], shape.renorm_clamp) * shape.routed_scaling
    if shape.router == "sigmoid_group":
        raw = sigmoid(np.asarray(z, dtype=np.float64)[ids])
        return raw / np.sum(raw) * shape.routed_scaling
    raise ValueError(shape.router)


def route_tokens(z: np.ndarray, shape, bias=None) -> dict:
    """Routes every token of z [T][E] by the shape's rule. Returns ids [T][k]
    int32, weights [T][k] float64, and the per-token ranking scores used to
    classify near-ties: `score` [T][E] (softmax p, or the selection score with
    bias) and, for the sigmoid family, `group_score` [T][n_group]; `logits`
    and `bias` are the inputs, returned for selection_weights."""
    T, E = z.shape
    k = shape.top_k
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    score = np.zeros((T, E), dtype=np.float64)
    gsc = np.zeros((T, max(shape.n_group, 1)), dtype=np.float64)
    for t in range(T):
        if shape.router == "softmax":
            i, a, p = softmax_topk_route(z[t], k, shape.renorm_clamp)
            a = a * shape.routed_scaling
            score[t] = p
        elif shape.router == "sigmoid_group":
            i, a, sel, gs, _ = sigmoid_group_topk_route(
                z[t], bias, shape.n_group, shape.topk_group, k,
                shape.routed_scaling)
            score[t] = sel
            gsc[t] = gs
        else:
            raise ValueError(shape.router)
        ids[t] = i
        w[t] = a
    return {"ids": ids, "weights": w, "score": score, "group_score": gsc, "logits": z,
            "bias": bias}


# ----------------------------------------------------------------------------
# experts and the layer
# ----------------------------------------------------------------------------
def silu(v):
    """SiLU(g) = g * sigmoid(g)."""
    v = np.asarray(v, dtype=np.float64)
    return v * sigmoid(v)


def swiglu_expert(x: np.ndarray, Wg: np.ndarray, Wu: np.ndarray,
                  Wd: np.ndarray) -> np.ndarray:
    """[P1] "Routed expert computation", [P2] "Experts":
    g = W_gate x, u = W_up x, h = SiLU(g) * u, e = W_down h.
    Wg, Wu [I][d]; Wd [d][I]; x [d] -> e [d]."""
    g = Wg @ x
    u = Wu @ x
    h = silu(g) * u
    return Wd @ h


def shared_gate(x: np.ndarray, w_shared: np.ndarray) -> float:
    """[P1] "Shared expert computation": s_t = sigmoid(w_shared^T x_t)."""
    return float(sigmoid(np.dot(w_shared, x)))


def _layer_f64(layer: dict, shape):
    adt = shape.act_dtype
    L = {
        "x": to_f64(layer["x"], adt),
        "r_attn": np.asarray(layer["r_attn"], dtype=np.float32).astype(np.float64),
        "W_router": to_f64(layer["W_router"], adt),
        "expert_bias": None if "expert_bias" not in layer else
        np.asarray(layer["expert_bias"], dtype=np.float32).astype(np.float64),
    }
    if shape.d_ff_shared > 0:
        for key in ("w_shared", "Ws_gate", "Ws_up", "Ws_down"):
            L[key] = to_f64(layer[key], adt)
    return L


def moe_experts_forward(layer: dict, shape, ids: np.ndarray, weights: np.ndarray,
                        s_shared=None, tokens=None, banks: ExpertBanks = None,
                        L64: dict = None) -> dict:
    """Steps 5-8 of [P1] "The short version" for given routing artefacts:
    per token, y_routed = sum over slots of alpha * expert(x) in slot order,
    y_shared = s_t * shared(x) with s_t the shared gate (computed from
    w_shared when s_shared is None), out = r_attn + (y_routed + y_shared).
    `tokens` restricts the computation to those token rows (each is computed
    on its own, so a sample of rows gives exactly the full run's rows)."""
    L64 = L64 or _layer_f64(layer, shape)
    banks = banks or ExpertBanks(layer, shape.expert_dtype)
    T = L64["x"].shape[0]
    tokens = range(T) if tokens is None else [int(t) for t in tokens]
    d = shape.d_model
    n = len(tokens)
    y_routed = np.zeros((n, d))
    y_shared = np.zeros((n, d))
    s_out = np.zeros(n)
    out = np.zeros((n, d))
    for row, t in enumerate(tokens):
        x = L64["x"][t]
        routed = np.zeros(d)
        for slot in range(shape.top_k):
            e = int(ids[t][slot])
            down = swiglu_expert(x, banks.get("W_gate", e), banks.get("W_up", e),
                                 banks.get("W_down", e))
            routed = routed + float(weights[t][slot]) * down
        shared = np.zeros(d)
        s = 0.0
        if shape.d_ff_shared > 0:
            s = shared_gate(x, L64["w_shared"]) if s_shared is None else float(s_shared[t])
            shared = s * swiglu_expert(x, L64["Ws_gate"], L64["Ws_up"], L64["Ws_down"])
        y_routed[row] = routed
        y_shared[row] = shared
        s_out[row] = s
        out[row] = L64["r_attn"][t] + (routed + shared)
    return {"out": out, "y_routed": y_routed, "y_shared": y_shared,
            "s_shared": s_out, "tokens": np.asarray(list(tokens), dtype=np.int64)}


def moe_layer_forward(layer: dict, shape, tokens=None) -> dict:
    """The whole layer, [P1] "Pseudocode" (with x already RMS-normalised):
    router logits, routing by the shape's rule, the selected SwiGLU experts
    weighted by alpha, the sigmoid-gated shared expert, the residual add.
    Returns out, ids, weights, s_shared, y_routed, y_shared (rows of
    `tokens`, all rows by default) plus the ranking scores of route_tokens."""
    L64 = _layer_f64(layer, shape)
    T = L64["x"].shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    z = router_logits(L64["x"][tok], L64["W_router"])
    r = route_tokens(z, shape, L64["expert_bias"])
    ids_full = np.zeros((T, shape.top_k), dtype=np.int32)
    w_full = np.zeros((T, shape.top_k))
    ids_full[tok] = r["ids"]
    w_full[tok] = r["weights"]
    res = moe_experts_forward(layer, shape, ids_full, w_full, None, tok,
                              ExpertBanks(layer, shape.expert_dtype), L64)
    res.update({"ids": r["ids"], "weights": r["weights"], "score": r["score"],
                "group_score": r["group_score"], "logits": z})
    return res


# ----------------------------------------------------------------------------
# bucketing
# ----------------------------------------------------------------------------
def bucket(ids: np.ndarray, n_experts: int) -> dict:
    """Counting and packing pass of [P1] "Intel SYCL path" (steps 1-3): count
    the routed (token, slot) pairs per expert, exclusive-scan the counts into
    offsets, list the active experts in ascending id, and pack each pair id
    (t*k + slot) under its expert, pairs of one expert in ascending pair id.
    Returns counts [E], offsets [E+1], active [A], perm [T*k] int32 and
    pos [T*k] (pair id -> packed position)."""
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    P = len(flat)
    counts = [0] * n_experts
    for e in flat:
        counts[e] += 1
    offsets = [0] * (n_experts + 1)
    for e in range(n_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    active = [e for e in range(n_experts) if counts[e] > 0]
    cursor = list(offsets[:-1])
    perm = [0] * P
    pos = [0] * P
    for pair, e in enumerate(flat):
        perm[cursor[e]] = pair
        pos[pair] = cursor[e]
        cursor[e] += 1
    i32 = np.int32
    return {"counts": np.asarray(counts, i32), "offsets": np.asarray(offsets, i32),
            "active": np.asarray(active, i32), "perm": np.asarray(perm, i32),
            "pos": np.asarray(pos, i32)}
