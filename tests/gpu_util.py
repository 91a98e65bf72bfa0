"""Helpers for the GPU parity tests: configs from shapes, device upload, the
near-tie routing comparison and the relative-to-RMS error."""
from __future__ import annotations

import functools

import numpy as np

import moe_inputs as mi
import sparse_moe_routing_gb300 as smr

GAP = 1e-4          # near-tie threshold on the oracle's ranking scores
W_TOL = 1e-5        # routing weights, absolute
OUT_TOL = {"bf16": 2e-2, "f32": 1e-4}   # max |out - ref| / rms(ref)


def cfg_for(shape: mi.MoEShape, T: int, path: int = smr.PATH_AUTO) -> smr.MoEConfig:
    dt = {"f32": smr.F32, "bf16": smr.BF16, "q4": smr.Q4_AFFINE_G64}
    return smr.MoEConfig(
        T=T, d_model=shape.d_model, n_experts=shape.n_experts, top_k=shape.top_k,
        d_ff=shape.d_ff, d_ff_shared=shape.d_ff_shared,
        router=smr.SOFTMAX_TOPK if shape.router == "softmax" else smr.SIGMOID_GROUP_TOPK,
        n_group=shape.n_group, topk_group=shape.topk_group,
        routed_scaling=shape.routed_scaling, renorm_clamp=shape.renorm_clamp,
        act_dtype=dt[shape.act_dtype], expert_dtype=dt[shape.expert_dtype], path=path)


def to_dev(a: np.ndarray):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@functools.lru_cache(maxsize=2)
def weights_host(name: str):
    return mi.make_weights(mi.PRESETS[name])


def layer_host(shape: mi.MoEShape, T: int) -> dict:
    L = dict(weights_host(shape.name)) if shape.name in mi.PRESETS and \
        mi.PRESETS[shape.name] == shape else mi.make_weights(shape)
    L.update(mi.make_activations(shape, T))
    return L


class DevLayer:
    """One layer's tensors on the GPU plus the output buffers."""

    def __init__(self, shape: mi.MoEShape, L: dict):
        import torch
        self.shape = shape
        self.T = L["x"].shape[0]
        self.t = {k: to_dev(v) for k, v in L.items()}
        k = shape.top_k
        self.out = torch.empty((self.T, shape.d_model), dtype=torch.float32, device="cuda")
        self.ids = torch.empty((self.T, k), dtype=torch.int32, device="cuda")
        self.w = torch.empty((self.T, k), dtype=torch.float32, device="cuda")

    def bank(self, name):
        if self.shape.expert_dtype == "q4":
            return (self.t[name + "_q"], self.t[name + "_scale"], self.t[name + "_min"])
        return self.t[name]

    def shared(self):
        if self.shape.d_ff_shared == 0:
            return dict(Ws_gate=None, Ws_up=None, Ws_down=None, w_shared=None)
        return dict(Ws_gate=self.t["Ws_gate"], Ws_up=self.t["Ws_up"],
                    Ws_down=self.t["Ws_down"], w_shared=self.t["w_shared"])

    def layer_forward(self, cfg, ws, stream=None):
        smr.layer_forward(cfg, ws, self.t["x"], self.t["r_attn"], self.t["W_router"],
                          self.bank("W_gate"), self.bank("W_up"), self.bank("W_down"),
                          self.out, self.ids, self.w, expert_bias=self.t.get("expert_bias"),
                          stream=stream, **self.shared())


def rel_rms_err(got: np.ndarray, ref: np.ndarray) -> float:
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref)) / max(rms, 1e-30))


def _candidate_scores(ref: dict, shape, t: int):
    """The oracle's ranking scores of token t among the experts it may pick
    (all experts; for the sigmoid family those of the kept groups), and the
    group-stage gap (inf without groups)."""
    score = ref["score"][t]
    ggap = np.inf
    if shape.router == "sigmoid_group":
        gs = ref["group_score"][t]
        order = np.argsort(-gs, kind="stable")
        if shape.topk_group < shape.n_group:
            ggap = gs[order[shape.topk_group - 1]] - gs[order[shape.topk_group]]
        G = shape.n_experts // shape.n_group
        kept = order[:shape.topk_group]
        mask = np.zeros(shape.n_experts, bool)
        for g in kept:
            mask[g * G:(g + 1) * G] = True
        return np.where(mask, score, -np.inf), ggap
    return score, ggap


def check_routing(gpu_ids: np.ndarray, gpu_w: np.ndarray, ref: dict, shape, rows=None):
    """North-star routing criteria. For every token whose oracle gap between
    the k-th and (k+1)-th ranking score (and, for groups, between the
    topk_group-th and next group score) exceeds GAP, the id sets must match
    exactly and the order must match wherever the oracle's neighbouring scores
    differ by more than GAP; weights must match per id within W_TOL. Tokens
    under the gap are near-ties: each GPU id must then be a valid choice
    (oracle score within GAP of the k-th). Returns the near-tie count."""
    k = shape.top_k
    rows = range(len(ref["ids"])) if rows is None else rows
    near = 0
    for r, t in enumerate(rows):
        cand, ggap = _candidate_scores(ref, shape, r)
        srt = np.sort(cand)[::-1]
        kgap = srt[k - 1] - srt[k] if k < np.isfinite(cand).sum() else np.inf
        want = [int(v) for v in ref["ids"][r]]
        got = [int(v) for v in gpu_ids[t]]
        wref = dict(zip(want, ref["weights"][r]))
        if min(kgap, ggap) > GAP:
            assert sorted(got) == sorted(want), (t, got, want, kgap)
            # slot order: the oracle's slots split into runs of near-equal
            # scores (neighbour gap <= GAP); each run must hold the same ids,
            # in any order (equal keys have no unique order)
            start = 0
            for s in range(k):
                if s == k - 1 or cand[want[s]] - cand[want[s + 1]] > GAP:
                    assert sorted(got[start:s + 1]) == sorted(want[start:s + 1]), (t, got, want)
                    start = s + 1
        else:
            near += 1
            if sorted(got) != sorted(want):
                score = ref["score"][r]
                floor = srt[k - 1] - GAP
                for e in got:
                    assert score[e] >= floor, (t, e, got, want)
                continue
        for e, w in zip(got, gpu_w[t]):
            assert abs(float(w) - wref[e]) <= W_TOL, (t, e, float(w), wref[e])
    return near
