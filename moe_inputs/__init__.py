"""Seeded synthetic inputs for the sparse MoE layer forward.

This module only *makes inputs*: layer shapes, random weights and activations,
their storage encodings (bf16 bit patterns, 4-bit affine group-64 packing) and
the seeds. It holds none of the layer's arithmetic (no router, no top-k, no
expert, no combine), so both the fp64 oracle and the CUDA path can consume the
same bytes without sharing any computation.

Shapes follow the pages this library implements:
  * Qwen3.6-35B-A3B layer: d_model 2048, 256 routed experts, top-8 softmax,
    expert and shared intermediate 512 ("How Treebeard routes Qwen3.6 MoE
    tokens", "Model constants" table and the packaged GGUF metadata).
  * DeepSeek-style sigmoid group top-k: n_group 8, topk_group 4, top-8,
    routed_scaling 2.5, 128 routed experts (Edge0 "MoE Routing and Experts",
    tier table and "Sigmoid group top-k").
  * Mixtral 8x7B style: 8 experts, top-2 (Airframe MoE roadmap, "MoE Models
    That Would Benefit"); d_model 4096 and intermediate 14336.
  * 4-bit affine, group 64 checkpoint quantisation (Edge0 tier table).

Recipe (every draw is seeded; the same call returns the same bytes):
  * weights ~ N(0, 0.02) (standard deviation 0.02), rounded to the storage
    dtype (bf16 round-to-nearest-even, or kept fp32);
  * x ~ N(0, 1) per row, then divided by its RMS (no gain, eps 1e-6) because
    the layer consumes the post-attention RMS-normalised state; stored in the
    activation dtype;
  * r_attn (the attention residual) ~ N(0, 1), fp32;
  * sigmoid-group configs: expert_bias ~ U(-bias_range, bias_range), fp32;
  * skewed configs: b_e ~ N(0, skew) and a seeded unit direction u; every
    token row gets a unit component along u (x <- x - (u.x)u + u, then RMS
    normalised) and router row e gets + b_e * u, so logit e is shifted by
    about b_e, giving an imbalanced token-per-expert histogram;
  * 4-bit affine group 64: per group of 64 consecutive input-dim weights,
    min = group minimum, scale = (max - min)/15 (both stored bf16), code
    q = clip(round_half_even((w - min_bf16)/scale_bf16), 0, 15); two codes per
    byte, the even element in the low nibble.

Seeds: weights from numpy default_rng(1000 + config_index); activations from
default_rng([1000 + config_index, T, 1]).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

__all__ = [
    "MoEShape", "PRESETS", "TINY_F32", "QWEN36", "QWEN36_PREFILL_SKEW",
    "DEEPSEEK_GROUP", "MIXTRAL", "MIXTRAL_Q4", "f32_to_bf16_bits",
    "make_layer", "make_activations", "make_weights", "quantize_q4_affine_g64",
    "random_router_outputs",
]

_CHUNK = 1 << 24  # elements per generation chunk (bounds host memory)


@dataclass(frozen=True)
class MoEShape:
    """One MoE layer shape plus its routing rule and storage dtypes."""
    name: str
    config_index: int
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    d_ff_shared: int            # 0: no shared expert
    router: str = "softmax"     # "softmax" | "sigmoid_group"
    n_group: int = 1
    topk_group: int = 1
    routed_scaling: float = 1.0
    renorm_clamp: float = 2.0 ** -14
    act_dtype: str = "bf16"     # "f32" | "bf16"  (x, router, shared weights)
    expert_dtype: str = "bf16"  # "f32" | "bf16" | "q4"
    logit_skew: float = 0.0     # std of the per-expert additive logit skew
    bias_range: float = 0.0     # expert_bias ~ U(-r, r) (sigmoid family)
    tokens: tuple = (1,)        # the token batch sizes this shape is run at

    def with_(self, **kw) -> "MoEShape":
        return dataclasses.replace(self, **kw)


TINY_F32 = MoEShape("tiny_f32", 0, d_model=256, n_experts=16, top_k=4, d_ff=64,
                    d_ff_shared=64, act_dtype="f32", expert_dtype="f32",
                    tokens=(32,))
QWEN36 = MoEShape("qwen36_decode", 1, d_model=2048, n_experts=256, top_k=8,
                  d_ff=512, d_ff_shared=512, tokens=(1, 8, 64))
QWEN36_PREFILL_SKEW = MoEShape("qwen36_prefill_skew", 2, d_model=2048,
                               n_experts=256, top_k=8, d_ff=512,
                               d_ff_shared=512, logit_skew=1.5,
                               tokens=(4096,))
DEEPSEEK_GROUP = MoEShape("deepseek_group", 3, d_model=2048, n_experts=128,
                          top_k=8, d_ff=512, d_ff_shared=512,
                          router="sigmoid_group", n_group=8, topk_group=4,
                          routed_scaling=2.5, bias_range=0.1,
                          tokens=(1, 4096))
MIXTRAL = MoEShape("mixtral_bf16", 4, d_model=4096, n_experts=8, top_k=2,
                   d_ff=14336, d_ff_shared=0, tokens=(2048,))
MIXTRAL_Q4 = MIXTRAL.with_(name="mixtral_q4", expert_dtype="q4")
# Further expert counts from the Airframe roadmap's model table (experts /
# top-k only; the widths are this generator's choice): DeepSeek-MoE 64/6 with
# one shared expert, Qwen MoE 60/4 with a shared expert four experts wide, and
# DeepSeek-V2 160/6, all softmax top-k.
DEEPSEEK_MOE_64 = MoEShape("deepseek_moe_64", 5, d_model=2048, n_experts=64, top_k=6,
                           d_ff=1408, d_ff_shared=1408, tokens=(1, 256))
QWEN_MOE_60 = MoEShape("qwen_moe_60", 6, d_model=2048, n_experts=60, top_k=4,
                       d_ff=1408, d_ff_shared=5632, tokens=(1, 5))
DEEPSEEK_V2_160 = MoEShape("deepseek_v2_160", 7, d_model=2048, n_experts=160, top_k=6,
                           d_ff=512, d_ff_shared=512, tokens=(64, 1024))

PRESETS = {s.name: s for s in (TINY_F32, QWEN36, QWEN36_PREFILL_SKEW,
                               DEEPSEEK_GROUP, MIXTRAL, MIXTRAL_Q4, DEEPSEEK_MOE_64,
                               QWEN_MOE_60, DEEPSEEK_V2_160)}


# ----------------------------------------------------------------------------
# storage encodings
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even:
    add 0x7FFF plus the lowest kept bit, keep the upper half. In 32-bit
    arithmetic the sum cannot wrap for any finite input (the largest,
    0xFF7FFFFF + 0x8000, stays below 2^32)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    flat_in = a.reshape(-1).view(np.uint32)
    flat_out = out.reshape(-1)
    for s in range(0, flat_in.size, _CHUNK):
        u = flat_in[s:s + _CHUNK]
        r = (u >> 16) & 1
        r += 0x7FFF
        r += u
        r >>= 16
        flat_out[s:s + _CHUNK] = r
    return out


def _bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def quantize_q4_affine_g64(w: np.ndarray):
    """Quantise fp32 weights [..., K] to 4-bit affine codes, groups of 64
    consecutive elements along the last axis.

    Returns (packed uint8 [..., K/2], scale bf16 bits [..., K/64],
    minv bf16 bits [..., K/64]); dequantised value = scale * q + minv.
    """
    K = w.shape[-1]
    if K % 64:
        raise ValueError("4-bit affine group-64 needs the input dim % 64 == 0")
    g = w.reshape(*w.shape[:-1], K // 64, 64).astype(np.float32)
    lo = g.min(axis=-1)
    hi = g.max(axis=-1)
    scale_bits = f32_to_bf16_bits((hi - lo) / np.float32(15.0))
    min_bits = f32_to_bf16_bits(lo)
    scale = _bf16_bits_to_f32(scale_bits)
    mn = _bf16_bits_to_f32(min_bits)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    q = np.rint((g - mn[..., None]) / safe[..., None])
    q = np.clip(q, 0, 15).astype(np.uint8).reshape(*w.shape[:-1], K)
    packed = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    return packed, scale_bits, min_bits


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------
def _normal(rng, shape, std, dtype):
    """N(0, std) of `shape` stored as `dtype` ('f32' -> float32,
    'bf16' -> uint16 bit patterns), generated in bounded chunks."""
    n = int(np.prod(shape))
    if dtype == "f32":
        out = np.empty(n, dtype=np.float32)
    else:
        out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        c = rng.standard_normal(min(_CHUNK, n - s), dtype=np.float32)
        c *= np.float32(std)
        out[s:s + c.size] = c if dtype == "f32" else f32_to_bf16_bits(c)
    return out.reshape(shape)


def _store(a32: np.ndarray, dtype: str) -> np.ndarray:
    return a32.astype(np.float32) if dtype == "f32" else f32_to_bf16_bits(a32)


def _skew_direction(shape: MoEShape):
    rng = np.random.default_rng([1000 + shape.config_index, 7])
    u = rng.standard_normal(shape.d_model).astype(np.float64)
    u /= np.linalg.norm(u)
    b = rng.normal(0.0, shape.logit_skew, size=shape.n_experts)
    return u, b


def make_weights(shape: MoEShape) -> dict:
    """All weights of one layer, in storage format.

    Keys: W_router [E][d], w_shared [d] (if shared), expert_bias [E] fp32
    (sigmoid family), W_gate/W_up [E][I][d], W_down [E][d][I] (or, for q4,
    `<bank>_q` uint8 [E][N][K/2], `<bank>_scale`/`<bank>_min` bf16 bits
    [E][N][K/64]), Ws_gate/Ws_up [I_s][d], Ws_down [d][I_s].
    """
    rng = np.random.default_rng(1000 + shape.config_index)
    d, E, I, Is = shape.d_model, shape.n_experts, shape.d_ff, shape.d_ff_shared
    adt = shape.act_dtype
    W = {}
    router = rng.standard_normal((E, d), dtype=np.float32) * np.float32(0.02)
    if shape.logit_skew > 0:
        u, b = _skew_direction(shape)
        router = (router.astype(np.float64) + b[:, None] * u[None, :]).astype(np.float32)
    W["W_router"] = _store(router, adt)
    if shape.router == "sigmoid_group":
        W["expert_bias"] = rng.uniform(-shape.bias_range, shape.bias_range,
                                       size=E).astype(np.float32)
    if Is > 0:
        W["w_shared"] = _normal(rng, (d,), 0.02, adt)
        W["Ws_gate"] = _normal(rng, (Is, d), 0.02, adt)
        W["Ws_up"] = _normal(rng, (Is, d), 0.02, adt)
        W["Ws_down"] = _normal(rng, (d, Is), 0.02, adt)
    for bank, (N, K) in (("W_gate", (I, d)), ("W_up", (I, d)), ("W_down", (d, I))):
        if shape.expert_dtype == "q4":
            qs, ss, ms = [], [], []
            for _ in range(E):
                w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
                q, s, m = quantize_q4_affine_g64(w)
                qs.append(q); ss.append(s); ms.append(m)
            W[bank + "_q"] = np.stack(qs)
            W[bank + "_scale"] = np.stack(ss)
            W[bank + "_min"] = np.stack(ms)
        else:
            W[bank] = _normal(rng, (E, N, K), 0.02, shape.expert_dtype)
    return W


def make_activations(shape: MoEShape, T: int) -> dict:
    """x [T][d] (act dtype, RMS-normalised rows) and r_attn [T][d] fp32."""
    rng = np.random.default_rng([1000 + shape.config_index, T, 1])
    d = shape.d_model
    x = rng.standard_normal((T, d)).astype(np.float64)
    if shape.logit_skew > 0 and T > 0:
        u, _ = _skew_direction(shape)
        x = x - (x @ u)[:, None] * u[None, :] + u[None, :]
    if T > 0:
        x = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + 1e-6)
    r = rng.standard_normal((T, d)).astype(np.float32)
    return {"x": _store(x.astype(np.float32), shape.act_dtype), "r_attn": r}


def make_layer(shape: MoEShape, T: int) -> dict:
    """Weights and activations of one layer at token batch T."""
    L = make_weights(shape)
    L.update(make_activations(shape, T))
    return L


def random_router_outputs(shape: MoEShape, T: int, seed: int = 0):
    """Arbitrary valid routing artefacts (distinct ids per token, positive
    weights) for exercising the expert path on its own: topk_ids int32 [T][k],
    weights fp32 [T][k], s_shared fp32 [T]."""
    rng = np.random.default_rng([1000 + shape.config_index, T, 2, seed])
    E, k = shape.n_experts, shape.top_k
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) \
        if T > 0 else np.zeros((0, k), np.int32)
    w = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    s = rng.uniform(0.0, 1.0, size=(T,)).astype(np.float32)
    return ids.reshape(T, k), w, s
