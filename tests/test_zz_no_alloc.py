"""moe_route_static: routing for callers that cannot allocate device memory.

A caller that cannot call cudaMalloc (a plugin whose host framework owns all
device memory, or a serving loop that must not allocate once running) cannot
provide moe_route's workspace. moe_route_static keeps the router logits in a
fixed array inside the library instead. These tests call it through the C ABI
and check it against moe_route on the same inputs, on two calls in a row
(the second call runs on different inputs over the first call's leftovers).
This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import moe_inputs as mi
from gpu_util import W_TOL, cfg_for, to_dev

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
    W = mi.make_weights(shape)
    A = mi.make_activations(shape.with_(config_index=shape.config_index + 100 * salt), T)
    return {k: to_dev(v) for k, v in list(W.items()) + list(A.items())
            if k in ("x", "W_router", "expert_bias", "w_shared")}


@pytest.mark.parametrize("shape,T", [(mi.QWEN36, 64), (mi.DEEPSEEK_GROUP, 37)],
                         ids=["qwen36-T64", "deepseek-T37"])
def test_static_scratch_route_matches_workspace_route(L, shape, T):
    cfg = cfg_for(shape, T)
    ws = smr.alloc_workspace(cfg)
    c_static = cfg._c()  # no workspace at all
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    k = shape.top_k
    for call in range(2):
        t = _inputs(shape, T, call)
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
        assert np.array_equal(i0, i1), call
        assert np.max(np.abs(w0 - w1)) <= W_TOL, call
        assert np.max(np.abs(s0 - s1)) <= W_TOL, call


def test_static_scratch_rejects_oversized_batches(L):
    shape = mi.QWEN36
    T = (1 << 20) // (shape.n_experts + 1) + 1      # T * (E + 1) above the array
    cfg = cfg_for(shape, T)
    st = L.moe_route_static(ctypes.c_void_p(16), ctypes.c_void_p(16), None, None,
                            ctypes.byref(cfg._c()), ctypes.c_void_p(16), ctypes.c_void_p(16),
                            None, None)
    assert st == smr._STATUS.index("MOE_ERR_UNSUPPORTED")
