#!/usr/bin/env python
"""Throughput of the sparse MoE layer forward on GB300 (tokens/s).

Default workload: the Qwen3.6-35B-A3B MoE layer shape (d_model 2048, 256
routed experts, top-8 softmax with renormalisation, expert and shared
intermediate 512, one sigmoid-gated shared expert), synthetic seeded weights
N(0, 0.02) in bf16 and RMS-normalised activations, at the decode batch T=64
(the sweep also runs T = 1 and 8, prefill, the sigmoid-group layer and the
Mixtral-shape layers). One step = one full layer forward (router, routing
rule, bucketing, routed experts, shared expert, combine, residual). Other
workloads (--workload prefill | deepseek | mixtral | mixtral_q4 |
deepseek_moe_64 | qwen_moe_60 | deepseek_v2_160) run the other shapes for
measurement; the default is the headline.

Timing: K steps are captured into one CUDA graph and replayed (W eager
warm-up steps first). Consecutive steps use distinct copies of the layer's
weights (rotating over enough copies that one pass touches >= 4x the L2), so
every step reads its weights from HBM. CUDA events on the capture/replay
stream bracket the replay; for the roofline figure the dominant kernel is
bracketed by events inside the graph (moe_trace_kernel) in a second replay, so
the event nodes do not add to the timed step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--tokens T]
                       [--workload decode|prefill|deepseek|mixtral|mixtral_q4|...]
                       [--path auto|gemv|tc|fused] [--impl ours|reference]
                       [--no-sweep] [--no-cpu-baseline] [--no-hot-l2] [--breakdown]
For N > 1 launch with torchrun (one rank per GPU, NCCL): every rank runs an
independent replica on its own token batch (the layer has no cross-token
exchange), so the job processes N*T tokens per step ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (Qwen3.6 shape, T=1..4096); % of HBM/tensor roofline"
L2_BYTES = 129 * 10 ** 6
TC_MIN_TOKENS = 6  # the library's MOE_PATH_AUTO switch away from the GEMV chain
FUSED_MAX_TOKENS = 16  # the single-launch decode kernel (--path fused) takes up to this many
FUSED_MIN_TOKENS = 4  # the library's MOE_PATH_AUTO takes it from this many (narrow bf16 shapes)

WORKLOADS = {
    # name: (preset, default T, description)
    "decode": ("qwen36_decode", 64, "qwen3.6-35b-a3b moe layer forward, decode batch T=%d"),
    "prefill": ("qwen36_prefill_skew", 4096,
                "qwen3.6-35b-a3b moe layer forward, prefill T=%d, skewed routing"),
    "deepseek": ("deepseek_group", 4096, "deepseek-style sigmoid group top-k layer, T=%d"),
    "mixtral": ("mixtral_bf16", 2048, "mixtral-style top-2 layer, bf16, T=%d"),
    "mixtral_q4": ("mixtral_q4", 2048,
                   "mixtral-style top-2 layer, 4-bit affine g64 experts, T=%d"),
    # further expert counts (experts / top-k of the Airframe model table; the
    # widths are the generator's choice), not part of the default sweep
    "deepseek_moe_64": ("deepseek_moe_64", 256,
                        "64-expert top-6 layer with a shared expert, width 1408, T=%d"),
    "qwen_moe_60": ("qwen_moe_60", 64,
                    "60-expert top-4 layer with a 5632-wide shared expert, width 1408, T=%d"),
    "deepseek_v2_160": ("deepseek_v2_160", 1024,
                        "160-expert top-6 layer with a shared expert, width 512, T=%d"),
}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _sustained_tflops():
    """bf16 dense rate measured as a seconds-long loop (the burst figure
    when only that one is known)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p.get("bf16_tflops_sustained", p["bf16_tflops"]))
    except Exception:
        return 1700.0


NOMINAL_HBM_GBS = 8000.0  # nominal HBM3e bandwidth of the part, for context
N_EXTRA_REPLAYS = 9       # timed replays after the first, for the median per step


# ----------------------------------------------------------------------------
# algorithmic work (what the layer must move / compute; intermediates excluded)
# ----------------------------------------------------------------------------
def _wbytes(shape):
    """Bytes per routed-expert weight: bf16 2, f32 4, 4-bit affine g64 0.5 plus
    a bf16 scale and min per 64 weights (0.5625)."""
    return {"bf16": 2, "f32": 4, "q4": 0.5 + 4 / 64}[shape.expert_dtype]


def _abytes(shape):
    return 2 if shape.act_dtype == "bf16" else 4


def layer_bytes(shape, T, n_active):
    d, E, I, Is, k = shape.d_model, shape.n_experts, shape.d_ff, shape.d_ff_shared, shape.top_k
    wb, ab = _wbytes(shape), _abytes(shape)
    b = E * d * ab + (d * ab if Is else 0)                 # router (+ shared gate)
    b += n_active * 3 * I * d * wb + 3 * Is * d * ab       # active experts + shared expert
    b += T * d * ab + 2 * T * d * 4 + T * k * 8            # x, r_attn, out, ids+weights
    return int(b)


def layer_flops(shape, T):
    d, E, I, Is, k = shape.d_model, shape.n_experts, shape.d_ff, shape.d_ff_shared, shape.top_k
    return 2 * T * d * (E + (1 if Is else 0)) + 2 * T * k * 3 * d * I + 2 * T * 3 * d * Is


def gateup_work(shape, T, n_active):
    """Per launch of a gate/up kernel: the gate and up rows of every active
    expert and of the shared expert (2*I*d*2 B each: 4,194,304 B at the Qwen
    shape) plus the activations x; flops 2*d*2*I per routed pair and per
    shared row."""
    d, I, Is, k = shape.d_model, shape.d_ff, shape.d_ff_shared, shape.top_k
    wb, ab = _wbytes(shape), _abytes(shape)
    b = n_active * 2 * I * d * wb + 2 * Is * d * ab + T * d * ab
    f = 2 * T * k * d * 2 * I + 2 * T * d * 2 * Is
    return int(b), f


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append((ts, parts))
        if not rows:
            return None
        inside = [r for r in rows if t0 <= r[0] <= t1 + 0.05]
        if not inside:  # region shorter than the sampling period: nearest sample
            inside = [min(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))]
        sm = sorted(float(p[1]) for _, p in inside if p[1].replace(".", "").isdigit())
        smax = max((float(p[2]) for _, p in inside if p[2].replace(".", "").isdigit()),
                   default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in inside for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(inside)}


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------
def _to_dev(a, device):
    import numpy as np
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def _traffic(kernel_name):
    """dram bytes per unit from the committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_name)
        src = os.path.join(ROOT, "sparse_moe_routing_gb300", "csrc", rec["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if h != rec["source_sha256_16"]:
            return None
        return rec
    except Exception:
        return None


class Weights:
    """One layer's weights generated once (host), uploaded once, and cloned on
    the device into as many distinct copies as a workload needs."""

    def __init__(self, shape, device, host=None):
        import moe_inputs as mi
        self.shape, self.device = shape, device
        self.host = mi.make_weights(shape) if host is None else host
        self.copies = [{k: _to_dev(v, device) for k, v in self.host.items()}]

    def get(self, n):
        while len(self.copies) < n:
            self.copies.append({k: v.clone() for k, v in self.copies[0].items()})
        return self.copies[:n]


def _cfg(shape, T, path):
    import sparse_moe_routing_gb300 as smr
    dt = {"f32": smr.F32, "bf16": smr.BF16, "q4": smr.Q4_AFFINE_G64}
    return smr.MoEConfig(
        T=T, d_model=shape.d_model, n_experts=shape.n_experts, top_k=shape.top_k,
        d_ff=shape.d_ff, d_ff_shared=shape.d_ff_shared,
        router=smr.SOFTMAX_TOPK if shape.router == "softmax" else smr.SIGMOID_GROUP_TOPK,
        n_group=shape.n_group, topk_group=shape.topk_group,
        routed_scaling=shape.routed_scaling, renorm_clamp=shape.renorm_clamp,
        act_dtype=dt[shape.act_dtype], expert_dtype=dt[shape.expert_dtype], path=path)


def _fused_auto(shape):
    """Whether the library's automatic choice takes the single-launch kernel
    for this shape (at 4-16 tokens): its tensor-core variant, d_model up to
    2048 and expert widths up to 1024."""
    return (shape.expert_dtype == "bf16" and shape.act_dtype == "bf16"
            and shape.d_model % 1024 == 0 and shape.d_ff % 128 == 0
            and shape.d_ff_shared % 128 == 0 and shape.d_model <= 2048
            and shape.d_ff <= 1024 and shape.d_ff_shared <= 1024)


def _uses_fused(shape, T, path):
    if shape.expert_dtype == "q4" or shape.expert_dtype != shape.act_dtype:
        return False
    if path == 0:  # the library's automatic choice
        return FUSED_MIN_TOKENS <= T <= FUSED_MAX_TOKENS and _fused_auto(shape)
    return path == 3 and T <= FUSED_MAX_TOKENS


def _tc_shape(shape):
    """The library's tensor-core path shapes: bf16 activations, d_model a
    multiple of 256, widths multiples of 128 (no shared expert for 4-bit
    banks)."""
    if shape.act_dtype != "bf16" or shape.d_model % 256 or shape.d_ff % 128:
        return False
    if shape.expert_dtype == "q4":
        return shape.d_ff_shared == 0
    return shape.expert_dtype == "bf16" and shape.d_ff_shared % 128 == 0


def _uses_tc(shape, T, path):
    if not _tc_shape(shape):
        return False
    if shape.expert_dtype == "q4":
        return True  # 4-bit banks are dequantised inside the tensor-core kernel
    if _uses_fused(shape, T, path):
        return False
    return path == 2 or (path == 0 and T >= TC_MIN_TOKENS)


def _expert_path(shape, T, path):
    if _uses_fused(shape, T, path):
        return "single-launch decode kernel"
    if _uses_tc(shape, T, path):
        return "tcgen05 grouped GEMM"
    return "CUDA-core direct-load GEMV" if T <= 8 else "CUDA-core streaming GEMV"


class Workload:
    """Device weight copies, activations and buffers of one token batch."""

    def __init__(self, weights, T, n_copies, path):
        import torch
        import moe_inputs as mi
        import sparse_moe_routing_gb300 as smr
        shape, device = weights.shape, weights.device
        self.shape, self.T, self.device, self.path = shape, T, device, path
        A = mi.make_activations(shape, T)
        self.host = dict(weights.host)
        self.host.update(A)
        self.copies = weights.get(n_copies)
        self.x = _to_dev(A["x"], device)
        self.r = _to_dev(A["r_attn"], device)
        self.cfg = _cfg(shape, T, path)
        layer = smr.MoELayer(self.cfg, self.copies[0], device)
        self.ws = layer.ws
        self.out = torch.empty((T, shape.d_model), dtype=torch.float32, device=device)
        self.ids = layer.ids
        self.wts = layer.weights

    def step(self, i):
        import sparse_moe_routing_gb300 as smr
        w = self.copies[i % len(self.copies)]
        smr.layer_forward(self.cfg, self.ws, self.x, self.r, w["W_router"], _bank(w, "W_gate"),
                          _bank(w, "W_up"), _bank(w, "W_down"), self.out, self.ids, self.wts,
                          expert_bias=w.get("expert_bias"), Ws_gate=w.get("Ws_gate"),
                          Ws_up=w.get("Ws_up"), Ws_down=w.get("Ws_down"),
                          w_shared=w.get("w_shared"))


def _bank(w, name):
    """A bank tensor, or the (codes, scale, min) tuple of a 4-bit bank."""
    return w[name] if name in w else (w[name + "_q"], w[name + "_scale"], w[name + "_min"])


def _n_copies(shape, T):
    E, k = shape.n_experts, shape.top_k
    a = E * (1 - (1 - k / E) ** T)
    touched = layer_bytes(shape, T, a)
    return int(min(16, max(2, math.ceil(4 * L2_BYTES / touched) + 1)))


class StepDurations(list):
    """Per-step durations (ms) of one traced kernel family: the sum of the
    family's launches within each step (`per` launches per step)."""
    per = 1


def time_graph(wl, K, W, trace_kernel=None, sampler=None, extra_replays=0):
    """Eager warm-up, then one CUDA graph of K steps replayed once (timed);
    extra_replays more timed replays after it (their ms in the last slot of
    the result). With trace_kernel, the third slot holds that family's
    duration per step (StepDurations: a family may launch more than once per
    step, e.g. a shared expert of another width has its own launches)."""
    import torch
    import sparse_moe_routing_gb300 as smr
    for i in range(W):
        wl.step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    tr = smr.KernelTrace(trace_kernel, 4 * K) if trace_kernel else None
    n0 = smr.launch_count()
    if tr:
        tr.__enter__()
    try:
        with torch.cuda.graph(g):
            for i in range(K):
                wl.step(i)
    finally:
        if tr:
            tr.__exit__(None, None, None)
    launches = smr.launch_count() - n0
    g.replay()  # untimed warm replay
    torch.cuda.synchronize()
    st, word = smr.read_device_status(wl.cfg, wl.ws)
    if st != 0:
        raise RuntimeError("device status %s (0x%x)" % (smr.status_string(st), word))
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    if sampler:
        sampler.start()
        time.sleep(0.15)
    s.record()
    g.replay()
    e.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if sampler:
        time.sleep(0.1)
        sampler.stop()
    ms = s.elapsed_time(e)
    durs = StepDurations()
    if tr:
        per = max(1, tr.count // K)
        one = tr.durations_ms()
        durs.per = per
        durs.extend(sum(one[i * per:(i + 1) * per]) for i in range(len(one) // per))
    extra = []
    for _ in range(extra_replays):
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        extra.append(s.elapsed_time(e))
    del g
    return ms, launches, durs, (t0, t1), extra


# The rest of the metric's range (T = 1..4096 and the other configurations),
# measured in the default run after the decode batches: (workload, tokens).
SWEEP_WORKLOADS = (("prefill", 4096), ("deepseek", 4096), ("mixtral", 2048),
                   ("mixtral_q4", 2048))


def start_host_weights(names):
    """Generates the host weights of the sweep's workloads in background
    threads (numpy's generators release the interpreter lock), so that they
    are ready when the decode measurements finish."""
    import concurrent.futures as cf
    import moe_inputs as mi
    ex = cf.ThreadPoolExecutor(max_workers=len(names))
    futs = {n: ex.submit(mi.make_weights, mi.PRESETS[WORKLOADS[n][0]]) for n in names}
    ex.shutdown(wait=False)
    return futs


def sweep_point(name, T, host, device, local, K, W, hbm, tflops):
    """One workload of the sweep: the layer timed as a CUDA graph of K steps
    (weights rotated beyond L2), the clocks during that replay, and the
    gate/up kernel's mean in-graph duration against its roofline."""
    import numpy as np
    import torch
    import moe_inputs as mi
    preset, _, desc = WORKLOADS[name]
    shape = mi.PRESETS[preset]
    weights = Weights(shape, device, host)
    wl = Workload(weights, T, _n_copies(shape, T), 0)
    sampler = ClockSampler(local)
    ms, _, _, (t0, t1), _ = time_graph(wl, K, W, None, sampler)
    durs = time_graph(wl, min(K, 100), 3, "tc_gateup")[2]
    n_act = int(np.unique(wl.ids.cpu().numpy()).size)
    ms_step = ms / K
    lb, lf = layer_bytes(shape, T, n_act), layer_flops(shape, T)
    floor_us = max(lb / (hbm * 1e9), lf / (tflops * 1e12)) * 1e6
    gb, gf = gateup_work(shape, T, n_act)
    hbm_bound = gb / (hbm * 1e9) >= gf / (tflops * 1e12)
    mean_k = sum(durs) / len(durs) if durs else None
    ach = (gb / (mean_k * 1e-3) / 1e9 if hbm_bound else gf / (mean_k * 1e-3) / 1e12) \
        if mean_k else None
    peak = hbm if hbm_bound else tflops
    out = {"workload": desc % T, "T": T, "us_per_layer": ms_step * 1e3,
           "tokens_per_s": T / (ms_step * 1e-3), "active_experts": n_act,
           "layer_floor_us": floor_us, "layer_floor_frac": floor_us / (ms_step * 1e3),
           "layer_hbm_frac": lb / (ms_step * 1e-3) / 1e9 / hbm,
           "layer_tensor_frac": lf / (ms_step * 1e-3) / 1e12 / tflops,
           "dominant": {"kernel": "tc_gateup", "bound": "hbm" if hbm_bound else "tensor",
                        "mean_launch_us": mean_k * 1e3 if mean_k else None,
                        "achieved": ach, "peak": peak,
                        "unit": "GB/s" if hbm_bound else "TFLOP/s",
                        "frac": ach / peak if ach else None},
           "clocks": sampler.summary(t0, t1)}
    del wl, weights
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def time_e2e(wl, K):
    """End to end through the public call with host buffers: every step, the
    pinned-host x and r_attn go to the device, the layer runs, and out,
    topk_ids and weights come back to pinned host memory. The copies run on
    an upload and a download stream with two buffer sets, so that a step's
    upload and the previous step's download overlap the layer between them;
    all of every step's bytes move inside the timed region. Returns the time,
    the bytes per step each way, and whether the last steps' host outputs
    equal the device-timed run's (same inputs, identical weight copies)."""
    import torch
    import sparse_moe_routing_gb300 as smr
    NB = 2
    xh = wl.x.cpu().pin_memory()
    rh = wl.r.cpu().pin_memory()
    xd = [torch.empty_like(wl.x) for _ in range(NB)]
    rd = [torch.empty_like(wl.r) for _ in range(NB)]
    od = [torch.empty_like(wl.out) for _ in range(NB)]
    oh = [torch.empty(wl.out.shape, dtype=torch.float32).pin_memory() for _ in range(NB)]
    ih = [torch.empty(wl.ids.shape, dtype=torch.int32).pin_memory() for _ in range(NB)]
    wh = [torch.empty(wl.wts.shape, dtype=torch.float32).pin_memory() for _ in range(NB)]
    layers = [smr.MoELayer(wl.cfg, w, wl.device) for w in wl.copies]
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    h2d = [torch.cuda.Event() for _ in range(NB)]
    done = [torch.cuda.Event() for _ in range(NB)]
    d2h = [torch.cuda.Event() for _ in range(NB)]
    for ev in h2d + done + d2h:
        ev.record(comp)

    def one(i):
        b, L = i % NB, layers[i % len(layers)]
        up.wait_event(done[b])          # the layer that last read xd[b], rd[b]
        with torch.cuda.stream(up):
            xd[b].copy_(xh, non_blocking=True)
            rd[b].copy_(rh, non_blocking=True)
        h2d[b].record(up)
        comp.wait_event(h2d[b])
        comp.wait_event(d2h[b])         # od[b] and this layer's ids/weights read out
        L.forward(xd[b], rd[b], out=od[b], stream=comp)
        done[b].record(comp)
        down.wait_event(done[b])
        with torch.cuda.stream(down):
            oh[b].copy_(od[b], non_blocking=True)
            ih[b].copy_(L.ids, non_blocking=True)
            wh[b].copy_(L.weights, non_blocking=True)
        d2h[b].record(down)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(comp)
    up.wait_event(s)
    for i in range(3, 3 + K):
        one(i)
    comp.wait_event(d2h[(2 + K) % NB])
    e.record(comp)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    ref_out, ref_ids = wl.out.cpu(), wl.ids.cpu()
    same = all(torch.equal(oh[b], ref_out) and torch.equal(ih[b], ref_ids) for b in range(NB))
    h2d_bytes = xh.numel() * xh.element_size() + rh.numel() * rh.element_size()
    d2h_bytes = sum(t.numel() * t.element_size() for t in (oh[0], ih[0], wh[0]))
    return ms, h2d_bytes, d2h_bytes, same


def _host_cores():
    cores = len(os.sched_getaffinity(0))
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        if info:
            cores = max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    return cores


def cpu_baseline(wl, budget_s=12.0):
    """The fp64 oracle as it stands on this host's cores, on a bounded sample
    of the same workload (successive chunks of tokens of the same batch)."""
    import oracle as orc
    L = wl.host
    done, t0 = 0, time.perf_counter()
    chunk = 4
    while time.perf_counter() - t0 < budget_s:
        start = done % wl.T
        toks = list(range(start, min(wl.T, start + chunk)))
        orc.moe_layer_forward(L, wl.shape, tokens=toks)
        done += len(toks)
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": "tokens/s", "cores": _host_cores(), "kind": "oracle",
            "sample": "%d token-rows cycling over the %d-token batch, %d per call "
                      "(fp64 numpy oracle, %.1f s)" % (done, wl.T, chunk, el)}


# ----------------------------------------------------------------------------
# ranks: one replica per GPU, no data exchange (the layer is independent per
# token); the process group only carries the barrier and the max of the times
# ----------------------------------------------------------------------------
def workload_config(shape, T, desc):
    """The workload's identity, the same in both arms' lines."""
    return {"workload": desc % T, "T": T, "d_model": shape.d_model,
            "n_experts": shape.n_experts, "top_k": shape.top_k, "d_ff": shape.d_ff,
            "d_ff_shared": shape.d_ff_shared, "router": shape.router,
            "weights": "%s, fp32 accumulate" % shape.expert_dtype}


def init_ranks(backend="nccl"):
    """(world, rank, local_rank) from the torchrun environment; joins the
    process group when there is more than one rank."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend)
    return world, rank, local


def max_over_ranks(value, device):
    """The largest of every rank's value (the job takes as long as its
    slowest replica)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if torch.distributed.is_initialized() and torch.distributed.get_world_size() > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, T, K, ms):
    """Whole-job throughput: every rank processes T tokens per step."""
    return world * T * K / (ms / 1e3)


def finish_ranks():
    import torch
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def run_ours(args):
    import numpy as np
    import torch
    import moe_inputs as mi
    import sparse_moe_routing_gb300 as smr

    world, rank, local = init_ranks("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if not os.path.exists(smr.lib_path):
        from sparse_moe_routing_gb300 import build
        build.build()
    hbm, tflops, peak_src = _peaks()
    preset, T_default, desc = WORKLOADS[args.workload]
    shape = mi.PRESETS[preset]
    path = {"auto": smr.PATH_AUTO, "gemv": smr.PATH_GEMV, "tc": smr.PATH_TC,
            "fused": smr.PATH_FUSED}[args.path]
    K, W = args.steps, args.warmup
    T = args.tokens or T_default
    full_sweep = (not args.no_sweep and args.workload == "decode" and world == 1
                  and not args.tokens and path == smr.PATH_AUTO)
    host_futs = start_host_weights([n for n, _ in SWEEP_WORKLOADS]) if full_sweep else {}
    weights = Weights(shape, device)

    load = {}

    replay_ms = []

    def hot_l2(T):
        """K steps that reuse one weight copy (no rotation): the weights are
        L2-resident only where the layer's bytes fit in L2."""
        wl1 = Workload(weights, T, 1, path)
        ms1 = time_graph(wl1, K, W)[0]
        del wl1
        return ms1 / K

    def measure(T, main, detail=None):
        """The timed replay (no event nodes inside the graph); for the main
        workload (and the sweep's decode points, detail) also the clocks
        during it and, from one more replay with the dominant kernel
        bracketed by in-graph events, that kernel's mean duration."""
        detail = main if detail is None else detail
        wl = Workload(weights, T, _n_copies(shape, T), path)
        tc = _uses_tc(shape, T, path)
        fused = _uses_fused(shape, T, path)
        kern = ("decode_fused" if fused else ("tc_gateup" if tc else "gemv_gateup")) \
            if detail else None
        sampler = ClockSampler(local) if detail else None
        ms, launches, _, (t0, t1), extra = time_graph(wl, K, W, None, sampler,
                                                     N_EXTRA_REPLAYS if main else 0)
        if main:
            replay_ms[:] = [ms] + extra
        durs = time_graph(wl, min(K, 100), 3, kern)[2] if detail else []
        ids = wl.ids.cpu().numpy().ravel()
        n_act = int(np.unique(ids).size)
        if main:
            # load histogram of the routed pairs over the experts
            cnt = np.bincount(ids, minlength=shape.n_experts)
            load["expert_rows_max"] = int(cnt.max())
            load["expert_rows_mean_active"] = float(cnt[cnt > 0].mean())
            load["idle_experts"] = int((cnt == 0).sum())
        clocks = sampler.summary(t0, t1) if sampler else None
        return wl, ms, launches, durs, n_act, clocks, kern

    wl, ms, launches, durs, n_act, clocks, kern = measure(T, True)
    ms = max_over_ranks(ms, device)
    ms_step = ms / K
    value = job_tokens_per_s(world, T, K, ms)

    # roofline of the dominant kernel: bytes and flops per launch, bound by
    # whichever floor is larger
    mean_k = sum(durs) / len(durs) if durs else None
    if kern == "decode_fused":
        # the single-launch kernel is the whole layer: its work is the layer's
        gb, gf = layer_bytes(shape, T, n_act), layer_flops(shape, T)
    else:
        gb, gf = gateup_work(shape, T, n_act)
    hbm_bound = gb / (hbm * 1e9) >= gf / (tflops * 1e12)
    if mean_k:
        sec = mean_k * 1e-3
        ach = gb / sec / 1e9 if hbm_bound else gf / sec / 1e12
    else:
        ach = None
    peak = hbm if hbm_bound else tflops
    tr = _traffic(kern)
    roofline = {"kernel": kern + (" (the whole layer in one launch)" if kern == "decode_fused"
                                  else " (routed + shared gate/up + SwiGLU)"),
                "bound": "hbm" if hbm_bound else "tensor", "achieved": ach, "peak": peak,
                "unit": "GB/s" if hbm_bound else "TFLOP/s",
                "frac": ach / peak if ach else None,
                "traffic": (tr["dram_bytes_per_unit"] * (n_act + (1 if shape.d_ff_shared else 0))
                            if tr and tr.get("unit") != "layer" else
                            (tr["dram_bytes_per_layer_per_byte"] * gb if tr else None)),
                "peak_source": peak_src, "algorithmic_bytes_per_launch": gb,
                "algorithmic_flops_per_launch": gf,
                "units_per_launch": (1 if kern == "decode_fused" else
                                     n_act + (1 if shape.d_ff_shared else 0)),
                "mean_launch_us": mean_k * 1e3 if mean_k else None,
                # launches of the family per step (2 when a shared expert of
                # another width has its own launch): the figures above are
                # per step, all of them together
                "launches_per_step": getattr(durs, "per", 1)}
    lb, lf = layer_bytes(shape, T, n_act), layer_flops(shape, T)
    config = dict(workload_config(shape, T, desc))
    config.update({
              "expert_path": _expert_path(shape, T, path),
              "l2": "weights rotate over %d distinct layer copies (>= 4x L2 per pass)"
                    % len(wl.copies),
              "timing": "one CUDA graph of K steps, replayed once; CUDA events; the dominant "
                        "kernel's mean duration from a second replay with it bracketed by "
                        "in-graph events",
              "parallelism": "replicas" if world == 1 else "dp%d (independent replicas)" % world,
              "active_experts": n_act, **load, "layer_alg_bytes": lb, "layer_alg_flops": lf,
              "layer_hbm_frac": lb / (ms_step * 1e-3) / 1e9 / hbm,
              "layer_tensor_frac": lf / (ms_step * 1e-3) / 1e12 / tflops})
    # the layer's floor: the larger of its bytes at the measured copy rate
    # and its flops at the measured bf16 rate; fractions also against the
    # nominal HBM rate and the sustained bf16 rate
    floor_us = max(lb / (hbm * 1e9), lf / (tflops * 1e12)) * 1e6
    config.update({
        "layer_floor_us": floor_us,
        "layer_floor_frac": floor_us / (ms_step * 1e3),
        "layer_hbm_frac_nominal_8tbs": lb / (ms_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
        "layer_tensor_frac_sustained": lf / (ms_step * 1e-3) / 1e12 / _sustained_tflops(),
        "replays": {"n": len(replay_ms), "steps_each": K,
                    "ms_per_step_median": float(np.median(replay_ms)) / K,
                    "ms_per_step_min": min(replay_ms) / K,
                    "ms_per_step_max": max(replay_ms) / K},
    })
    if not args.no_hot_l2:
        hot = hot_l2(T)
        config["hot_l2"] = {"ms_per_step": hot, "tokens_per_s": T / (hot * 1e-3),
                            "note": "one weight copy reused every step (L2-hot where the "
                                    "layer's bytes fit in L2), not the headline"}
    if not args.no_sweep and args.workload == "decode":
        sweep = {}
        for Ts in (1, 8, 64):
            if Ts == T:
                sweep[str(Ts)] = {"T": T, "us_per_layer": ms_step * 1e3,
                                  "tokens_per_s": T * K / (ms / 1e3), "ms_per_step": ms_step,
                                  "expert_path": config["expert_path"],
                                  "layer_floor_us": floor_us,
                                  "layer_floor_frac": config["layer_floor_frac"],
                                  "layer_hbm_frac": config["layer_hbm_frac"],
                                  "dominant": {k_: roofline[k_] for k_ in
                                               ("kernel", "bound", "mean_launch_us", "achieved",
                                                "peak", "unit", "frac")},
                                  "clocks": clocks}
                continue
            wls, mss, _, dus, na, cls, kn = measure(Ts, False, True)
            b, f = layer_bytes(shape, Ts, na), layer_flops(shape, Ts)
            us = mss / K * 1e3
            fl = max(b / (hbm * 1e9), f / (tflops * 1e12)) * 1e6
            if kn == "decode_fused":
                kb_, kf_ = b, f
            else:
                kb_, kf_ = gateup_work(shape, Ts, na)
            mk = sum(dus) / len(dus) if dus else None
            kach = kb_ / (mk * 1e-3) / 1e9 if mk else None
            sweep[str(Ts)] = {"T": Ts, "us_per_layer": us, "tokens_per_s": Ts * K / (mss / 1e3),
                              "ms_per_step": mss / K, "active_experts": na,
                              "expert_path": _expert_path(shape, Ts, path),
                              "layer_floor_us": fl, "layer_floor_frac": fl / us,
                              "layer_hbm_frac": b / (mss / K * 1e-3) / 1e9 / hbm,
                              "dominant": {"kernel": kn, "bound": "hbm",
                                           "mean_launch_us": mk * 1e3 if mk else None,
                                           "achieved": kach, "peak": hbm, "unit": "GB/s",
                                           "frac": kach / hbm if kach else None},
                              "clocks": cls}
            del wls
            if not args.no_hot_l2:
                sweep[str(Ts)]["hot_l2_ms_per_step"] = hot_l2(Ts)
        config["sweep"] = sweep
    if full_sweep:
        # the rest of the metric's range: prefill, the sigmoid-group layer and
        # the Mixtral-shape layers at their configured batch sizes
        for name, Tw in SWEEP_WORKLOADS:
            sweep[name] = sweep_point(name, Tw, host_futs[name].result(), device, local, K, W,
                                      hbm, tflops)
            host_futs[name] = None
    if args.breakdown:
        # one more graph replay per kernel family, that family bracketed by
        # events: mean in-graph duration per launch (us)
        bd = {}
        kb = min(K, 50)
        for fam in smr.KERNELS:
            durs_f = time_graph(wl, kb, 3, fam)[2]
            if durs_f:
                bd[fam] = round(sum(durs_f) / len(durs_f) * 1e3, 2)
        config["breakdown_us"] = bd
    k_e2e = min(K, 200)
    e2e_ms, h2d, d2h, same = time_e2e(wl, k_e2e)
    e2e_ms = max_over_ranks(e2e_ms, device)
    e2e = {"value": job_tokens_per_s(world, T, k_e2e, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "copies": "upload and download streams, double-buffered, overlapping the layer",
           "host_outputs_match_device_run": bool(same)}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": shape.expert_dtype, "data": "synthetic",
            "config": config, "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line))
    finish_ranks()


def run_eager(args):
    """N plain layer calls in a row (for ncu captures of single launches: with
    K kernels per call, skip K*c launches to capture the (c+1)-th call)."""
    import torch
    import moe_inputs as mi
    import sparse_moe_routing_gb300 as smr
    device = torch.device("cuda", 0)
    preset, T_default, desc = WORKLOADS[args.workload]
    shape = mi.PRESETS[preset]
    path = {"auto": smr.PATH_AUTO, "gemv": smr.PATH_GEMV, "tc": smr.PATH_TC,
            "fused": smr.PATH_FUSED}[args.path]
    T = args.tokens or T_default
    wl = Workload(Weights(shape, device), T, 1, path)
    for _ in range(args.eager):
        wl.step(0)
    torch.cuda.synchronize()
    st, word = smr.read_device_status(wl.cfg, wl.ws)
    print(json.dumps({"eager_calls": args.eager, "workload": desc % T, "status": st}))
    if st != 0:
        sys.exit(1)


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on this host's
    cores, on the same workload; each step is a bounded sample of tokens."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import moe_inputs as mi
    import oracle as orc
    preset, T_default, desc = WORKLOADS[args.workload]
    shape = mi.PRESETS[preset]
    T = args.tokens or T_default
    L = mi.make_layer(shape, T)
    t0 = time.perf_counter()
    orc.moe_layer_forward(L, shape, tokens=[0])
    t_tok = time.perf_counter() - t0
    K, W = args.steps, args.warmup
    per_step = max(1, min(T, int(150.0 / max(1, K + W) / max(t_tok, 1e-6))))
    cur = 0

    def step():
        nonlocal cur
        toks = [(cur + j) % T for j in range(per_step)]
        cur = (cur + per_step) % T
        orc.moe_layer_forward(L, shape, tokens=toks)

    for _ in range(W):
        step()
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    el = time.perf_counter() - t0
    value = K * per_step / el
    sample = "%d token(s) of the T=%d batch per step (fp64 numpy oracle)" % (per_step, T)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": K, "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape, T, desc),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _host_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--tokens", type=int, default=0, help="token batch (default: workload's)")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--path", choices=["auto", "gemv", "tc", "fused"], default="auto")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-hot-l2", action="store_true",
                    help="skip the extra timing with one reused weight copy")
    ap.add_argument("--breakdown", action="store_true",
                    help="also report the mean in-graph time of every kernel family")
    ap.add_argument("--eager", type=int, default=0, metavar="N",
                    help="profiling aid: run N untimed eager layer calls on the workload "
                         "(one weight copy, no graph) and exit; prints no bench line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.eager:
        run_eager(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
