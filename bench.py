#!/usr/bin/env python
"""Throughput of the sparse MoE layer forward on GB300 (tokens/s).

Workload: the Qwen3.6-35B-A3B MoE layer shape (d_model 2048, 256 routed
experts, top-8 softmax with renormalisation, expert and shared intermediate
512, one sigmoid-gated shared expert), synthetic seeded weights N(0, 0.02)
in bf16 and RMS-normalised activations, at the decode batch T (default 64;
the sweep also runs T = 1 and 8). One step = one full layer forward (router,
routing rule, bucketing, routed experts, shared expert, combine, residual).

Timing: K steps are captured into one CUDA graph and replayed (W eager
warm-up steps first). Consecutive steps use distinct copies of the layer's
weights (rotating over enough copies that one pass touches >= 4x the L2), so
every step reads its weights from HBM. CUDA events on the capture/replay
stream bracket the replay; the dominant kernel is additionally bracketed by
events inside the graph (moe_trace_kernel) for the roofline figure.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--tokens T]
                       [--impl ours|reference] [--no-sweep] [--no-cpu-baseline]
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


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------
# algorithmic work (what the layer must move; intermediates excluded)
# ----------------------------------------------------------------------------
def layer_bytes(shape, T, n_active):
    d, E, I, Is, k = shape.d_model, shape.n_experts, shape.d_ff, shape.d_ff_shared, shape.top_k
    wb = 2  # bf16
    b = E * d * wb + (d * wb if Is else 0)                 # router (+ shared gate)
    b += n_active * 3 * I * d * wb + 3 * Is * d * wb       # active experts + shared expert
    b += T * d * wb + 2 * T * d * 4 + T * k * 8            # x, r_attn, out, ids+weights
    return b


def layer_flops(shape, T):
    d, E, I, Is, k = shape.d_model, shape.n_experts, shape.d_ff, shape.d_ff_shared, shape.top_k
    return 2 * T * d * (E + (1 if Is else 0)) + 2 * T * k * 3 * d * I + 2 * T * 3 * d * Is


def gateup_bytes(shape, T, n_active):
    """Per launch of the gate/up kernel: the gate and up rows of every active
    expert and of the shared expert (4,194,304 B each at this shape), plus the
    activations x."""
    d, I, Is = shape.d_model, shape.d_ff, shape.d_ff_shared
    return n_active * 2 * I * d * 2 + 2 * Is * d * 2 + T * d * 2


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
            if len(parts) < 9:
                continue
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
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel (else None)."""
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

    def __init__(self, shape, device):
        import moe_inputs as mi
        self.shape, self.device = shape, device
        self.host = mi.make_weights(shape)
        self.copies = [{k: _to_dev(v, device) for k, v in self.host.items()}]

    def get(self, n):
        while len(self.copies) < n:
            self.copies.append({k: v.clone() for k, v in self.copies[0].items()})
        return self.copies[:n]


class Workload:
    """Device weight copies, activations and buffers of one token batch."""

    def __init__(self, weights, T, n_copies):
        import torch
        import moe_inputs as mi
        import sparse_moe_routing_gb300 as smr
        shape, device = weights.shape, weights.device
        self.shape, self.T, self.device = shape, T, device
        A = mi.make_activations(shape, T)
        self.host = dict(weights.host)
        self.host.update(A)
        self.copies = weights.get(n_copies)
        self.x = _to_dev(A["x"], device)
        self.r = _to_dev(A["r_attn"], device)
        self.cfg = smr.MoEConfig(T=T, d_model=shape.d_model, n_experts=shape.n_experts,
                                 top_k=shape.top_k, d_ff=shape.d_ff,
                                 d_ff_shared=shape.d_ff_shared,
                                 routed_scaling=shape.routed_scaling,
                                 renorm_clamp=shape.renorm_clamp)
        layer = smr.MoELayer(self.cfg, self.copies[0], device)
        self.ws = layer.ws
        self.out = torch.empty((T, shape.d_model), dtype=torch.float32, device=device)
        self.ids = layer.ids
        self.wts = layer.weights

    def step(self, i):
        import sparse_moe_routing_gb300 as smr
        w = self.copies[i % len(self.copies)]
        smr.layer_forward(self.cfg, self.ws, self.x, self.r, w["W_router"], w["W_gate"],
                          w["W_up"], w["W_down"], self.out, self.ids, self.wts,
                          Ws_gate=w["Ws_gate"], Ws_up=w["Ws_up"], Ws_down=w["Ws_down"],
                          w_shared=w["w_shared"])


def _n_copies(shape, T):
    import moe_inputs  # noqa: F401
    E, k = shape.n_experts, shape.top_k
    a = E * (1 - (1 - k / E) ** T)
    touched = layer_bytes(shape, T, a)
    return int(min(16, max(2, math.ceil(4 * L2_BYTES / touched) + 1)))


def time_graph(wl, K, W, trace_kernel=None, sampler=None):
    """Eager warm-up, then one CUDA graph of K steps replayed once (timed)."""
    import torch
    import sparse_moe_routing_gb300 as smr
    for i in range(W):
        wl.step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    tr = smr.KernelTrace(trace_kernel, K) if trace_kernel else None
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
    durs = tr.durations_ms() if tr else []
    del g
    return ms, launches, durs, (t0, t1)


def time_e2e(wl, K):
    """End to end through the public call with host buffers: per step, the
    pinned-host x and r_attn go to the device, the layer runs, and out,
    topk_ids and weights come back to pinned host memory."""
    import torch
    xh = wl.x.cpu().pin_memory()
    rh = wl.r.cpu().pin_memory()
    oh = torch.empty(wl.out.shape, dtype=torch.float32).pin_memory()
    ih = torch.empty(wl.ids.shape, dtype=torch.int32).pin_memory()
    wh = torch.empty(wl.wts.shape, dtype=torch.float32).pin_memory()
    x = torch.empty_like(wl.x)
    r = torch.empty_like(wl.r)
    import sparse_moe_routing_gb300 as smr
    layers = [smr.MoELayer(wl.cfg, w, wl.device) for w in wl.copies]

    def one(i):
        x.copy_(xh, non_blocking=True)
        r.copy_(rh, non_blocking=True)
        out, ids, wts = layers[i % len(layers)].forward(x, r)
        oh.copy_(out, non_blocking=True)
        ih.copy_(ids, non_blocking=True)
        wh.copy_(wts, non_blocking=True)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for i in range(K):
        one(i)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    h2d = xh.numel() * xh.element_size() + rh.numel() * rh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in (oh, ih, wh))
    return ms, h2d, d2h


def cpu_baseline(wl, budget_s=12.0):
    """The fp64 oracle as it stands on this host's cores, on a bounded sample
    of the same workload (successive chunks of tokens of the same batch)."""
    import oracle as orc
    cores = len(os.sched_getaffinity(0))
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        if info:
            cores = max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    L = wl.host
    done, t0 = 0, time.perf_counter()
    chunk = 4
    while time.perf_counter() - t0 < budget_s:
        start = done % wl.T
        toks = list(range(start, min(wl.T, start + chunk)))
        orc.moe_layer_forward(L, wl.shape, tokens=toks)
        done += len(toks)
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d token-rows cycling over the %d-token batch, %d per call "
                      "(fp64 numpy oracle, %.1f s)" % (done, wl.T, chunk, el)}


def run_ours(args):
    import numpy as np
    import torch
    import moe_inputs as mi
    import sparse_moe_routing_gb300 as smr

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if not os.path.exists(smr.lib_path):
        from sparse_moe_routing_gb300 import build
        build.build()
    hbm, tflops, peak_src = _peaks()
    shape = mi.QWEN36
    K, W, T = args.steps, args.warmup, args.tokens

    weights = Weights(shape, device)

    def measure(T, trace):
        wl = Workload(weights, T, _n_copies(shape, T))
        sampler = ClockSampler(local) if trace else None
        ms, launches, durs, (t0, t1) = time_graph(wl, K, W, "gemv_gateup" if trace else None,
                                                  sampler)
        n_act = int(np.unique(wl.ids.cpu().numpy()).size)
        return wl, ms, launches, durs, n_act, (sampler.summary(t0, t1) if sampler else None)

    wl, ms, launches, durs, n_act, clocks = measure(T, True)
    t_max = torch.tensor([ms], device=device)
    if world > 1:
        torch.distributed.all_reduce(t_max, op=torch.distributed.ReduceOp.MAX)
    ms = float(t_max.item())
    ms_step = ms / K
    value = world * T * K / (ms / 1e3)

    mean_k = sum(durs) / len(durs) if durs else None
    ach = gateup_bytes(shape, T, n_act) / (mean_k * 1e-3) / 1e9 if mean_k else None
    tr = _traffic("gemv_gateup")
    roofline = {"kernel": "gemv_gateup (routed + shared gate/up + SwiGLU)", "bound": "hbm",
                "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm if ach else None,
                "traffic": (tr["dram_bytes_per_unit"] * (n_act + 1) if tr else None),
                "peak_source": peak_src,
                "algorithmic_bytes_per_launch": gateup_bytes(shape, T, n_act),
                "units_per_launch": n_act + 1, "mean_launch_us": mean_k * 1e3 if mean_k else None}
    lb = layer_bytes(shape, T, n_act)
    config = {"workload": "qwen3.6-35b-a3b moe layer forward, decode batch T=%d" % T,
              "T": T, "d_model": shape.d_model, "n_experts": shape.n_experts,
              "top_k": shape.top_k, "d_ff": shape.d_ff, "d_ff_shared": shape.d_ff_shared,
              "router": "softmax top-8, renorm clamp 2^-14", "weights": "bf16, fp32 accumulate",
              "l2": "weights rotate over %d distinct layer copies (>= 4x L2 per pass)"
                    % len(wl.copies),
              "timing": "one CUDA graph of K steps, replayed once; CUDA events",
              "parallelism": "replicas" if world == 1 else "dp%d (independent replicas)" % world,
              "active_experts": n_act,
              "layer_alg_bytes": lb, "layer_hbm_frac": lb / (ms_step * 1e-3) / 1e9 / hbm}
    sweep = {}
    if not args.no_sweep:
        for Ts in (1, 8, 64):
            if Ts == T:
                sweep[str(Ts)] = {"tokens_per_s": T * K / (ms / 1e3), "ms_per_step": ms_step,
                                  "layer_hbm_frac": config["layer_hbm_frac"]}
                continue
            wls, mss, _, _, na, _ = measure(Ts, False)
            b = layer_bytes(shape, Ts, na)
            sweep[str(Ts)] = {"tokens_per_s": Ts * K / (mss / 1e3), "ms_per_step": mss / K,
                              "active_experts": na,
                              "layer_hbm_frac": b / (mss / K * 1e-3) / 1e9 / hbm}
            del wls
        config["sweep"] = sweep
    e2e_ms, h2d, d2h = time_e2e(wl, min(K, 200))
    e2e = {"value": world * T * min(K, 200) / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches, "clocks": clocks}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on this host's
    cores, on the same workload; each step is a bounded sample of tokens."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import moe_inputs as mi
    import oracle as orc
    shape, T = mi.QWEN36, args.tokens
    L = mi.make_layer(shape, T)
    cores = len(os.sched_getaffinity(0))
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
        "config": {"workload": "qwen3.6-35b-a3b moe layer forward, decode batch T=%d" % T,
                   "T": T},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
