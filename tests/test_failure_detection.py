"""Failure detection on the GPU without a fault: a bounded on-device wait is
made to run out, and the kernel must report it and leave the context usable.

moe_inject_stall arms a one-shot self-test: the next launch of the chosen
kernel family waits on a flag that nothing sets, with that launch's wait
limit cut to a few milliseconds. The tensor-core kernel's MMA warp then waits
on an accumulator barrier only it would complete; in the single-launch decode
kernel, block 0 never arrives at the first grid barrier. Either way the wait
gives up, the kernel records MOE_ERR_DEVICE_TIMEOUT in the workspace's status
word, lets its copies in flight land, frees its tensor memory and returns.
moe_read_device_status reports the timeout and resets the workspace's control
words; the next call on the same workspace must then match the oracle.
"""
import numpy as np
import pytest

import moe_inputs as mi
from gpu_util import DevLayer, cfg_for, check_layer, layer_host, OUT_TOL

pytestmark = pytest.mark.gpu

import torch  # noqa: E402

import sparse_moe_routing_gb300 as smr  # noqa: E402

TIMEOUT = 5  # MOE_ERR_DEVICE_TIMEOUT

TC_SMALL = mi.MoEShape("tc_small", 7, d_model=512, n_experts=4, top_k=2, d_ff=256,
                       d_ff_shared=256, tokens=(400,))


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_routing_gb300 import build
    build.build()
    smr.lib()
    yield
    smr.inject_stall(None, 0)


CASES = [("decode_fused", mi.QWEN36, 4, smr.PATH_FUSED, 9),
         ("tc_gateup", TC_SMALL, 400, smr.PATH_TC, 5),
         ("tc_down", TC_SMALL, 400, smr.PATH_TC, 6)]


@pytest.mark.parametrize("kernel,shape,T,path,site", CASES, ids=[c[0] for c in CASES])
def test_wait_runs_out_then_workspace_is_usable(kernel, shape, T, path, site):
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    cfg = cfg_for(shape, T, path)
    ws = smr.alloc_workspace(cfg)
    smr.inject_stall(kernel, 2000)
    dev.layer_forward(cfg, ws)
    st, word = smr.read_device_status(cfg, ws)
    assert st == TIMEOUT, (st, hex(word))
    assert (word >> 16) == site, hex(word)
    # the self-test is one-shot and the control words were reset: the same
    # workspace now gives the oracle's layer
    dev.out.zero_()
    dev.layer_forward(cfg, ws)
    st, word = smr.read_device_status(cfg, ws)
    assert st == 0, (st, hex(word))
    near, moved, err, y_err = check_layer(L, shape, dev.ids.cpu().numpy(), dev.w.cpu().numpy(),
                                          dev.out.cpu().numpy(), np.arange(T))
    assert err <= OUT_TOL[shape.act_dtype], err


def test_disarmed_stall_does_not_fire():
    shape, T = mi.QWEN36, 2
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    cfg = cfg_for(shape, T, smr.PATH_FUSED)
    ws = smr.alloc_workspace(cfg)
    smr.inject_stall("decode_fused", 2000)
    smr.inject_stall(None, 0)
    dev.layer_forward(cfg, ws)
    assert smr.read_device_status(cfg, ws)[0] == 0
