"""Layer parity on seeded random shapes: expert counts, top-k, widths, token
counts, both routing rules, with and without a shared expert, on every
expert path the shape allows. Every output row is compared with the fp64
oracle (the shapes are small enough for the oracle to do all of them)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import sparse_moe_routing_gb300 as smr
from gpu_util import DevLayer, OUT_TOL, Y_TOL, cfg_for, check_layer

pytestmark = pytest.mark.gpu


def _shapes(n=10, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([8, 16, 24, 32, 64, 96]))
        k = int(rng.integers(1, min(E, 8) + 1))
        d = int(rng.choice([256, 512]))
        I = int(rng.choice([128, 256]))
        Is = int(rng.choice([0, I]))
        sigmoid = bool(rng.integers(0, 2)) and E % 8 == 0
        kw = {}
        if sigmoid:
            n_group = int(rng.choice([g for g in (2, 4, 8) if E % g == 0]))
            G = E // n_group
            topk_group = int(rng.integers(max(1, -(-k // G)), n_group + 1))
            kw = dict(router="sigmoid_group", n_group=n_group, topk_group=topk_group,
                      routed_scaling=float(rng.choice([1.0, 2.5])), bias_range=0.1)
        T = int(rng.choice([1, 3, 5, 8, 37, 130, 300]))
        shape = mi.MoEShape("rand%d" % i, 20 + i, d_model=d, n_experts=E, top_k=k, d_ff=I,
                            d_ff_shared=Is, tokens=(T,), **kw)
        out.append((shape, T))
    return out


CASES = [(s, T, p) for s, T in _shapes() for p in (smr.PATH_AUTO, smr.PATH_GEMV, smr.PATH_TC)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_routing_gb300 import build
    build.build()


@pytest.mark.parametrize("shape,T,path", CASES,
                         ids=["%s-E%d-k%d-T%d-%s" % (c[0].name, c[0].n_experts, c[0].top_k, c[1],
                                                     {0: "auto", 1: "gemv", 2: "tc"}[c[2]])
                              for c in CASES])
def test_random_shape_layer_parity(shape, T, path):
    cfg = cfg_for(shape, T, path)
    if smr.lib().moe_workspace_bytes(__import__("ctypes").byref(cfg._c())) == 0:
        pytest.skip("invalid shape")
    L = mi.make_layer(shape, T)
    dev = DevLayer(shape, L)
    ws = None
    try:
        ws = smr.alloc_workspace(cfg)
        dev.layer_forward(cfg, ws)
    except smr.MoEError as e:
        if "UNSUPPORTED" in str(e):
            pytest.skip("shape outside this path's limits")
        raise
    st, word = smr.read_device_status(cfg, ws)
    assert st == 0, hex(word)
    near, moved, err, y_err = check_layer(L, shape, dev.ids.cpu().numpy(), dev.w.cpu().numpy(),
                                          dev.out.cpu().numpy(), np.arange(T))
    assert err <= OUT_TOL[shape.act_dtype], err
    assert y_err <= Y_TOL[shape.act_dtype], y_err
