"""moe_route_static: routing for callers that cannot allocate device memory.

A caller that cannot call cudaMalloc (a plugin whose host framework owns all
device memory, or a serving loop that must not allocate once running) cannot
provide moe_route's workspace. moe_route_static keeps the router logits in a
fixed array inside the library instead. These tests call it through the C ABI
on two calls in a row (the second call runs on different inputs over the
first call's leftovers) and check it against the fp64 oracle by the routing
criteria of the parity tests, and against moe_route on the same inputs: bit
for bit below 128 tokens (the same kernels), by the same criteria above
(moe_route then contracts on the tensor cores). This file is collected last
so that a run stopping at its first failure has already run every other
test.
"""
import ctypes

import numpy as np
import pytest

import moe_inputs as mi
import oracle as orc
from gpu_util import W_TOL, cfg_for, check_routing, oracle_routing, to_dev

pytestmark = pytest.mark.gpu

import torch  # noqa: E402

import sparse_moe_routing_gb300 as smr  # noqa: E402


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_routing_gb300 import build
    build.build()
    lib = smr.lib()
    fn = lib.moe_route_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.POINTER(smr._Cfg)] + [ctypes.c_void_p] * 4
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _inputs(shape, T, salt):
    """(host arrays, device tensors) of the routing inputs; the activations
    differ between salts."""
    W = mi.make_weights(shape)
    A = mi.make_activations(shape.with_(config_index=shape.config_index + 100 * salt), T)
    host = {k: v for k, v in list(W.items()) + list(A.items())
            if k in ("x", "W_router", "expert_bias", "w_shared")}
    return host, {k: to_dev(v) for k, v in host.items()}


CASES = [(mi.QWEN36, 64), (mi.DEEPSEEK_GROUP, 37), (mi.QWEN36, 256), (mi.DEEPSEEK_GROUP, 1024)]


@pytest.mark.parametrize("shape,T", CASES, ids=["%s-T%d" % (c[0].name, c[1]) for c in CASES])
def test_static_scratch_route_matches_oracle_and_workspace_route(L, shape, T):
    cfg = cfg_for(shape, T)
    ws = smr.alloc_workspace(cfg)
    c_static = cfg._c()  # no workspace at all
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    k = shape.top_k
    for call in range(2):
        host, t = _inputs(shape, T, call)
        outs = []
        for use_static in (False, True):
            ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
            w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
            s = torch.full((T,), -1.0, dtype=torch.float32, device="cuda")
            if use_static:
                st = L.moe_route_static(_p(t["x"]), _p(t["W_router"]), _p(t.get("expert_bias")),
                                        _p(t["w_shared"]), ctypes.byref(c_static), _p(ids),
                                        _p(w), _p(s), stream)
                assert st == 0, smr.status_string(st)
            else:
                smr.route(cfg, ws, t["x"], t["W_router"], ids, w,
                          expert_bias=t.get("expert_bias"), w_shared=t["w_shared"], s_shared=s)
            torch.cuda.synchronize()
            outs.append((ids.cpu().numpy(), w.cpu().numpy(), s.cpu().numpy()))
        (i0, w0, s0), (i1, w1, s1) = outs
        ref = oracle_routing(host, shape)
        near, moved = check_routing(i1, w1, ref, shape)
        check_routing(i0, w0, ref, shape)
        x = orc.to_f64(host["x"], shape.act_dtype)
        ws_ = orc.to_f64(host["w_shared"], shape.act_dtype)
        gate = np.array([orc.shared_gate(x[r], ws_) for r in range(T)])
        assert np.max(np.abs(s1 - gate)) <= W_TOL, call
        print("%s T=%d call %d: near-ties %d, rerouted %d" % (shape.name, T, call, near, len(moved)))
        if T < 128:
            assert np.array_equal(i0, i1), call
            assert np.array_equal(w0, w1), call
            assert np.array_equal(s0, s1), call


def test_static_scratch_rejects_oversized_batches(L):
    shape = mi.QWEN36
    T = (1 << 20) // (shape.n_experts + 1) + 1      # T * (E + 1) above the array
    cfg = cfg_for(shape, T)
    st = L.moe_route_static(ctypes.c_void_p(16), ctypes.c_void_p(16), None, None,
                            ctypes.byref(cfg._c()), ctypes.c_void_p(16), ctypes.c_void_p(16),
                            None, None)
    assert st == smr._STATUS.index("MOE_ERR_UNSUPPORTED")
