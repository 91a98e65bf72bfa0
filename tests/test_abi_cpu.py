"""The C-ABI library on the host (no GPU): it builds, loads, exports every
function include/moe_route.h declares, and its host-only paths (status
strings, workspace sizing, argument validation) behave as documented.
Nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

import moe_inputs as mi
import sparse_moe_routing_gb300 as smr
from sparse_moe_routing_gb300 import build as smr_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    smr_build.build()
    return smr.lib()


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names += re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n


def test_abi_version_and_status_strings(L):
    assert smr.abi_version() == 1
    for s in range(7):
        assert smr.status_string(s).startswith(smr._STATUS[s])
    assert "unknown" in smr.status_string(99)


def _cfg(**kw):
    base = dict(T=64, d_model=2048, n_experts=256, top_k=8, d_ff=512, d_ff_shared=512)
    base.update(kw)
    return smr.MoEConfig(**base)


def test_workspace_bytes_grows_with_T(L):
    a = smr.workspace_bytes(_cfg(T=1))
    b = smr.workspace_bytes(_cfg(T=64))
    c = smr.workspace_bytes(_cfg(T=4096))
    assert 0 < a < b < c
    assert a % 256 == 0 and c % 256 == 0


@pytest.mark.parametrize("bad", [
    dict(d_model=100), dict(n_experts=0), dict(top_k=0), dict(top_k=300),
    dict(d_ff=0), dict(d_ff_shared=4), dict(T=-1), dict(router=7),
    dict(router=1, n_group=3), dict(router=1, n_group=8, topk_group=0),
    dict(router=1, n_group=8, topk_group=9),
    dict(act_dtype=5), dict(renorm_clamp=-1.0), dict(routed_scaling=float("nan")),
    dict(path=9),
])
def test_invalid_configs_are_rejected_on_the_host(L, bad):
    cfg = _cfg(**bad)
    c = cfg._c()
    assert L.moe_workspace_bytes(ctypes.byref(c)) == 0
    # every entry point returns before touching the device
    st = L.moe_layer_forward(None, None, None, None, smr._Bank(), smr._Bank(), smr._Bank(),
                             None, None, None, None, ctypes.byref(c), None, None, None, None)
    assert st in (1, 2), st


def test_outside_build_limits_is_unsupported(L):
    for kw in (dict(router=1, n_group=64, topk_group=1, top_k=2), dict(n_experts=1024)):
        c = _cfg(**kw)._c()
        st = L.moe_layer_forward(None, None, None, None, smr._Bank(), smr._Bank(), smr._Bank(),
                                 None, None, None, None, ctypes.byref(c), None, None, None, None)
        assert st == 2, kw


def test_group_rule_needs_enough_candidates(L):
    # topk_group * E / n_group < k: the rule could not pick k experts
    c = _cfg(router=1, n_experts=128, n_group=8, topk_group=1, top_k=17)._c()
    assert L.moe_workspace_bytes(ctypes.byref(c)) == 0


def test_workspace_checks(L):
    cfg = _cfg()
    c = cfg._c()
    # no workspace
    st = L.moe_route(None, None, None, None, ctypes.byref(c), None, None, None, None)
    assert st == 3
    # misaligned workspace pointer
    c.workspace = 0x1001
    c.workspace_bytes = 1 << 40
    assert L.moe_workspace_init(ctypes.byref(c), None) == 3
    # too small
    c.workspace = 0x100000
    c.workspace_bytes = 1024
    st = L.moe_bucket(None, ctypes.byref(c), None, None, None, None, None, None, None)
    assert st == 3


def test_null_and_misaligned_tensors_rejected(L):
    cfg = _cfg(T=4)
    c = cfg._c()
    c.workspace = 0x100000
    c.workspace_bytes = smr.workspace_bytes(cfg)
    st = L.moe_route(None, 0x2000, None, None, ctypes.byref(c), 0x3000, 0x4000, None, None)
    assert st == 1
    st = L.moe_route(0x2008, 0x2000, None, None, ctypes.byref(c), 0x3000, 0x4000, None, None)
    assert st == 1


def test_zero_tokens_enqueue_nothing(L):
    cfg = _cfg(T=0)
    c = cfg._c()
    c.workspace = 0x100000
    c.workspace_bytes = smr.workspace_bytes(cfg)
    # T = 0 returns MOE_OK before any pointer or device use
    assert L.moe_route(None, None, None, None, ctypes.byref(c), None, None, None, None) == 0
    assert L.moe_bucket(None, ctypes.byref(c), None, None, None, None, None, None, None) == 0


def test_gpu_util_configs_are_valid(L):
    import gpu_util
    for shape in mi.PRESETS.values():
        for T in shape.tokens:
            cfg = gpu_util.cfg_for(shape, T)
            c = cfg._c()
            assert L.moe_workspace_bytes(ctypes.byref(c)) > 0, shape.name


def test_static_route_checks_match_moe_route(L):
    """moe_route_static returns moe_route's codes for every host-side check
    (the workspace check aside), and UNSUPPORTED when the logits would not
    fit its fixed array; none of these touch the device."""
    fn = L.moe_route_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.POINTER(smr._Cfg)] + [ctypes.c_void_p] * 4
    cases = [dict(top_k=300), dict(router=1, n_group=3), dict(n_experts=1024),
             dict(n_group=64), dict(router=1, n_group=64, topk_group=1, top_k=2),
             dict(expert_dtype=7), dict(d_model=100)]
    for kw in cases:
        cfg = _cfg(**kw)
        c = cfg._c()
        c.workspace = 0x100000
        c.workspace_bytes = 1 << 40
        want = L.moe_route(None, None, None, None, ctypes.byref(c), None, None, None, None)
        got = fn(None, None, None, None, ctypes.byref(cfg._c()), None, None, None, None)
        assert got == want and got in (1, 2), (kw, got, want)
    # null and misaligned tensors
    c = _cfg(T=4)._c()
    assert fn(None, 0x2000, None, None, ctypes.byref(c), 0x3000, 0x4000, None, None) == 1
    assert fn(0x2008, 0x2000, None, None, ctypes.byref(c), 0x3000, 0x4000, None, None) == 1
    # T = 0: nothing to do
    assert fn(None, None, None, None, ctypes.byref(_cfg(T=0)._c()), None, None, None, None) == 0
    # T * (E + 1) beyond the fixed array
    T = (1 << 20) // 257 + 1
    assert fn(0x2000, 0x2000, None, None, ctypes.byref(_cfg(T=T)._c()), 0x3000, 0x4000,
              None, None) == 2


def test_inject_stall_accepts_only_kernels_with_bounded_waits(L):
    assert L.moe_inject_stall(0, 0) == 0
    for bad in (1, 2, 4, 7, 11, 99):
        assert L.moe_inject_stall(bad, 100) == 1
    for ok in (8, 9, 12):
        assert L.moe_inject_stall(ok, 100) == 0
    assert L.moe_inject_stall(0, 0) == 0
