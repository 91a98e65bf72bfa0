"""Helpers for the GPU parity tests: configs from shapes, device upload, the
near-tie routing comparison and the relative-to-RMS error."""
from __future__ import annotations

import functools
import itertools
import math

import numpy as np

import moe_inputs as mi
import oracle as orc
import sparse_moe_routing_gb300 as smr

GAP = 1e-4          # near-tie threshold on the oracle's ranking scores
W_TOL = 1e-5        # routing weights, absolute
OUT_TOL = {"bf16": 2e-2, "f32": 1e-4}   # max |out - ref| / rms(ref)
# the same metric on y_moe = out - r_attn, the layer's own contribution (out is
# dominated by the N(0, 1) residual, so its gate says little about y_moe)
Y_TOL = {"bf16": 3e-2, "f32": 1e-3}


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


def _valid_topk_sets(v: np.ndarray, k: int):
    """Every set of k indices that the near-tie rule accepts as the top k of
    the scores v (-inf marks an index that cannot be chosen): all indices
    scoring more than GAP above the k-th score, completed from those within
    GAP of it. One set when the k-th and (k+1)-th scores differ by more than
    GAP."""
    idx = np.flatnonzero(np.isfinite(v))
    if idx.size <= k:
        return {frozenset(int(i) for i in idx)}
    srt = np.sort(v[idx])[::-1]
    sk = srt[k - 1]
    forced = [int(i) for i in idx if v[i] > sk + GAP]
    opt = [int(i) for i in idx if sk - GAP <= v[i] <= sk + GAP]
    need = k - len(forced)
    if math.comb(len(opt), need) > 20000:
        raise ValueError("too many near-tied candidates to enumerate")
    return {frozenset(forced + list(c)) for c in itertools.combinations(opt, need)}


def routing_alternatives(ref: dict, shape, r: int):
    """The id sets the routing criteria accept for oracle row r. Softmax
    family: the valid top-k sets of the oracle's probabilities. Sigmoid group
    family: for every valid set of kept groups (the same rule on the group
    scores), the valid top-k sets of the selection scores inside those
    groups; experts of other groups cannot be chosen."""
    score = ref["score"][r]
    k = shape.top_k
    if shape.router != "sigmoid_group":
        return _valid_topk_sets(score, k)
    G = shape.n_experts // shape.n_group
    out = set()
    for kept in _valid_topk_sets(ref["group_score"][r], shape.topk_group):
        mask = np.zeros(shape.n_experts, bool)
        for g in kept:
            mask[g * G:(g + 1) * G] = True
        out |= _valid_topk_sets(np.where(mask, score, -np.inf), k)
    return out


def _clear_gaps(ref: dict, shape, r: int):
    """(k-th vs (k+1)-th gap among the choosable experts, group-stage gap) of
    oracle row r (inf where a stage has no (k+1)-th)."""
    score = ref["score"][r]
    ggap = np.inf
    cand = score
    if shape.router == "sigmoid_group":
        gs = ref["group_score"][r]
        order = np.argsort(-gs, kind="stable")
        if shape.topk_group < shape.n_group:
            ggap = gs[order[shape.topk_group - 1]] - gs[order[shape.topk_group]]
        G = shape.n_experts // shape.n_group
        mask = np.zeros(shape.n_experts, bool)
        for g in order[:shape.topk_group]:
            mask[g * G:(g + 1) * G] = True
        cand = np.where(mask, score, -np.inf)
    srt = np.sort(cand)[::-1]
    k = shape.top_k
    kgap = srt[k - 1] - srt[k] if k < np.isfinite(cand).sum() else np.inf
    return cand, kgap, ggap


def ordered(ids, score):
    """A selection in the oracle's slot order: descending score, ties to the
    lower id."""
    return sorted(ids, key=lambda e: (-score[e], e))


def check_routing(gpu_ids: np.ndarray, gpu_w: np.ndarray, ref: dict, shape, rows=None):
    """North-star routing criteria. Every token: k distinct ids in [0, E).
    Tokens whose oracle gap between the k-th and (k+1)-th ranking score (and,
    for groups, between the topk_group-th and next group score) exceeds GAP:
    the id sets match exactly and the order matches wherever the oracle's
    neighbouring scores differ by more than GAP. Near-tie tokens: the GPU's
    set must be one of the sets the criteria accept (routing_alternatives).
    Weights match, per id within W_TOL, the oracle's weight step applied to
    the GPU's own selection (for a matching set, the oracle's weights).

    Returns (near-tie count, {token: oracle-ordered alternative selection}
    for the tokens whose GPU set differs from the oracle's)."""
    k, E = shape.top_k, shape.n_experts
    rows = range(len(ref["ids"])) if rows is None else rows
    near = 0
    alts = {}
    for r, t in enumerate(rows):
        got = [int(v) for v in gpu_ids[t]]
        assert all(0 <= e < E for e in got), (t, got)
        assert len(set(got)) == k, (t, got, "duplicate id")
        cand, kgap, ggap = _clear_gaps(ref, shape, r)
        want = [int(v) for v in ref["ids"][r]]
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
            sel = want
            wsel = ref["weights"][r]
        else:
            near += 1
            if sorted(got) == sorted(want):
                sel = want
                wsel = ref["weights"][r]
            else:
                valid = routing_alternatives(ref, shape, r)
                assert frozenset(got) in valid, (t, got, want, "not a valid near-tie choice")
                sel = ordered(sorted(frozenset(got)), ref["score"][r])
                wsel = orc.selection_weights(ref["logits"][r], sel, shape, ref.get("bias"))
                alts[t] = sel
        wref = dict(zip(sel, wsel))
        for e, w in zip(got, gpu_w[t]):
            assert abs(float(w) - wref[e]) <= W_TOL, (t, e, float(w), wref[e])
    return near, alts


def oracle_routing(L: dict, shape) -> dict:
    """The oracle's routing of every token of layer L (logits from x)."""
    x = orc.to_f64(L["x"], shape.act_dtype)
    W = orc.to_f64(L["W_router"], shape.act_dtype)
    bias = None if "expert_bias" not in L else L["expert_bias"].astype(np.float64)
    return orc.route_tokens(orc.router_logits(x, W), shape, bias)


def oracle_outputs(L: dict, shape, ref_r: dict, rows, alts=None, banks=None) -> dict:
    """The oracle's layer output rows `rows` under its own routing ref_r,
    except that a near-tied token in `alts` takes that alternative selection
    (with the weights the oracle's rule gives it)."""
    ids = np.array(ref_r["ids"], dtype=np.int32)
    w = np.array(ref_r["weights"], dtype=np.float64)
    for t, sel in (alts or {}).items():
        ids[t] = sel
        w[t] = orc.selection_weights(ref_r["logits"][t], sel, shape, ref_r.get("bias"))
    return orc.moe_experts_forward(L, shape, ids, w, None, rows, banks)


def _host_mem_bytes() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 8 << 30


def oracle_banks(L: dict, shape):
    """The oracle's fp64 expert banks with a cache large enough for every
    expert of the layer when the host has the memory (the cache only saves
    repeated conversions; results do not depend on it)."""
    per = 8 * 3 * shape.d_ff * shape.d_model
    want = per * shape.n_experts + (64 << 20)
    return orc.ExpertBanks(L, shape.expert_dtype,
                           cache_bytes=int(min(want, max(3 << 30, _host_mem_bytes() // 4))))


def block_rows(ref_r: dict, shape, T: int, bm: int = 128, extra=(), seed=0):
    """Token rows that cover every work item of the grouped GEMMs: the oracle's
    own bucketing of its ids (the order the GPU packs rows in, wherever the
    ids agree) is cut into blocks of bm packed rows per expert, and the
    tokens of the first and last row of every block are taken; the shared
    expert's blocks are tokens [m*bm, (m+1)*bm). Returns (rows, number of
    blocks covered)."""
    k = shape.top_k
    b = orc.bucket(ref_r["ids"], shape.n_experts)
    toks = set(int(t) for t in extra)
    blocks = 0
    for e in range(shape.n_experts):
        lo, hi = int(b["offsets"][e]), int(b["offsets"][e + 1])
        for s in range(lo, hi, bm):
            last = min(s + bm, hi) - 1
            toks.add(int(b["perm"][s]) // k)
            toks.add(int(b["perm"][last]) // k)
            blocks += 1
    if shape.d_ff_shared > 0:
        for s in range(0, T, bm):
            toks.update((s, min(s + bm, T) - 1))
            blocks += 1
    return np.array(sorted(toks), dtype=np.int64), blocks


def check_layer(L: dict, shape, gpu_ids, gpu_w, out, rows, ref_r=None, banks=None):
    """Routing of every token (check_routing) and the output rows `rows`
    against the oracle (a near-tied token whose GPU selection differs from
    the oracle's is compared with the oracle's output for that selection).
    Returns (near-tie count, number of tokens routed differently, out error,
    y_moe error)."""
    ref_r = ref_r if ref_r is not None else oracle_routing(L, shape)
    near, alts = check_routing(gpu_ids, gpu_w, ref_r, shape)
    rows = np.asarray(rows, dtype=np.int64)
    ref = oracle_outputs(L, shape, ref_r, rows, alts, banks)
    o = np.asarray(out, np.float64)[rows]
    r = np.asarray(L["r_attn"], np.float64)[rows]
    err = rel_rms_err(o, ref["out"])
    y_err = rel_rms_err(o - r, ref["out"] - r)
    return near, len(alts), err, y_err
