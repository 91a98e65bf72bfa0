"""GPU parity of the CUDA path with the fp64 oracle, through the C ABI.

Criteria (stated once here, applied throughout):
  * routing ids: bit-exact wherever the oracle's gap between the k-th and
    (k+1)-th ranking score (and for groups, between the topk_group-th and next
    group score) exceeds 1e-4; near-ties are counted and must be valid choices;
  * routing weights: within 1e-5 absolute;
  * bucketing: bit-exact (integers);
  * layer output: max |out - ref| / rms(ref) <= 2e-2 (bf16) or 1e-4 (fp32).
  * the layer's own contribution y_moe = out - r_attn: the same metric
    <= 3e-2 (bf16) or 1e-3 (fp32);
  * near-tie tokens: the GPU's selection must be one the criteria accept,
    with the weights the oracle's rule gives it, and its output row is
    compared with the oracle's output for that selection.
Small cases compare every element; full-size cases compare the routing of
every token and the output rows that cover every work item of the grouped
GEMMs (the first and last packed row of every 128-row block of every expert
and of the shared expert), plus a seeded sample (each output row depends
only on its own token, so the oracle computes those rows exactly).
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle as orc
from gpu_util import (OUT_TOL, Y_TOL, DevLayer, block_rows, cfg_for, check_layer,
                      check_routing, layer_host, oracle_banks, oracle_routing, rel_rms_err,
                      to_dev)

pytestmark = pytest.mark.gpu

import torch  # noqa: E402

import sparse_moe_routing_gb300 as smr  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_routing_gb300 import build
    build.build()
    smr.lib()


def _sample(T, n, seed=0):
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    s = np.sort(rng.choice(T, size=n - 2, replace=False))
    return np.unique(np.concatenate([[0, T - 1], s]))


def _run_layer(shape, T, path=smr.PATH_AUTO):
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    cfg = cfg_for(shape, T, path)
    ws = smr.alloc_workspace(cfg)
    dev.layer_forward(cfg, ws)
    st, word = smr.read_device_status(cfg, ws)
    assert st == 0, (st, hex(word))
    return L, dev, cfg, ws


# (shape, T, output rows the oracle checks: "all", or "blocks" for the rows
# covering every 128-row block of every group plus a seeded sample)
CASES = [
    (mi.TINY_F32, 32, "all"),
    (mi.TINY_F32.with_(name="tiny_f32_ragged"), 37, "all"),
    (mi.TINY_F32.with_(name="tiny_f32_t4"), 4, "all"),
    (mi.QWEN36, 1, "all"),
    (mi.QWEN36, 2, "all"),
    (mi.QWEN36, 3, "all"),
    (mi.QWEN36, 8, "all"),
    (mi.QWEN36, 16, "all"),
    (mi.QWEN36, 17, "all"),
    (mi.QWEN36, 64, "all"),
    (mi.QWEN36, 65, "all"),
    (mi.QWEN36, 37, "all"),
    (mi.DEEPSEEK_GROUP, 1, "all"),
    (mi.DEEPSEEK_GROUP, 64, "all"),
    (mi.QWEN36_PREFILL_SKEW, 4096, "blocks"),
    (mi.DEEPSEEK_GROUP, 4096, "blocks"),
    (mi.MIXTRAL, 2048, "blocks"),
    # decode batches of 6-16 tokens: the single-launch kernel where it is the
    # automatic choice (160 experts: router tiles past E), the tensor-core
    # path on the wider shapes
    (mi.MIXTRAL, 8, "all"),
    (mi.DEEPSEEK_MOE_64, 1, "all"),
    (mi.DEEPSEEK_MOE_64, 8, "all"),
    (mi.DEEPSEEK_MOE_64, 256, "blocks"),
    (mi.QWEN_MOE_60, 1, "all"),
    (mi.QWEN_MOE_60, 5, "all"),
    (mi.QWEN_MOE_60, 12, "all"),
    (mi.QWEN_MOE_60, 64, "all"),
    (mi.QWEN_MOE_60, 300, "blocks"),
    (mi.DEEPSEEK_V2_160, 16, "all"),
    (mi.DEEPSEEK_V2_160, 64, "all"),
    (mi.DEEPSEEK_V2_160, 1024, "blocks"),
]


def _check_rows(L, shape, T, dev, mode, seed=0):
    """Routing of every token and the chosen output rows against the oracle;
    prints and returns (near-ties, rerouted tokens, out error, y_moe error)."""
    ref_r = oracle_routing(L, shape)
    if mode == "all":
        rows, blocks = np.arange(T), None
    else:
        rows, blocks = block_rows(ref_r, shape, T, extra=_sample(T, 16, seed))
    res = check_layer(L, shape, dev.ids.cpu().numpy(), dev.w.cpu().numpy(),
                      dev.out.cpu().numpy(), rows, ref_r, oracle_banks(L, shape))
    near, moved, err, y_err = res
    print("%s T=%d rows=%d%s near-ties=%d rerouted=%d out_err=%.3e y_moe_err=%.3e" % (
        shape.name, T, len(rows), "" if blocks is None else " blocks=%d/%d" % (blocks, blocks),
        near, moved, err, y_err))
    assert err <= OUT_TOL[shape.act_dtype], err
    assert y_err <= Y_TOL[shape.act_dtype], y_err
    return res


@pytest.mark.parametrize("shape,T,mode", CASES,
                         ids=["%s-T%d" % (c[0].name, c[1]) for c in CASES])
def test_layer_forward_parity(shape, T, mode):
    L, dev, cfg, ws = _run_layer(shape, T)
    _check_rows(L, shape, T, dev, mode)


# The single-launch kernel forced on the shapes the automatic choice leaves
# to the tensor-core path: d_model 4096 (four K segments per warp, token
# fragments loaded per stage), expert widths of 1408 and 14336 and a 5632-wide
# shared expert (h chunks too wide to stage in shared memory).
FORCED_FUSED = [(mi.MIXTRAL, 3), (mi.MIXTRAL, 8), (mi.DEEPSEEK_MOE_64, 8), (mi.QWEN_MOE_60, 12)]


@pytest.mark.parametrize("shape,T", FORCED_FUSED,
                         ids=["%s-T%d" % (c[0].name, c[1]) for c in FORCED_FUSED])
def test_single_launch_forced_on_wide_shapes(shape, T):
    L, dev, cfg, ws = _run_layer(shape, T, smr.PATH_FUSED)
    _check_rows(L, shape, T, dev, "all")


ROUTE_CASES = [(mi.TINY_F32, 32), (mi.QWEN36, 64), (mi.QWEN36_PREFILL_SKEW, 4096),
               (mi.DEEPSEEK_GROUP, 4096), (mi.MIXTRAL, 2048)]


@pytest.mark.parametrize("shape,T", ROUTE_CASES,
                         ids=["%s-T%d" % (c[0].name, c[1]) for c in ROUTE_CASES])
def test_route_parity_and_shared_gate(shape, T):
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    cfg = cfg_for(shape, T)
    ws = smr.alloc_workspace(cfg)
    s_sh = torch.empty(T, dtype=torch.float32, device="cuda") if shape.d_ff_shared else None
    smr.route(cfg, ws, dev.t["x"], dev.t["W_router"], dev.ids, dev.w,
              expert_bias=dev.t.get("expert_bias"), w_shared=dev.t.get("w_shared"),
              s_shared=s_sh)
    assert smr.read_device_status(cfg, ws)[0] == 0
    ref = oracle_routing(L, shape)
    check_routing(dev.ids.cpu().numpy(), dev.w.cpu().numpy(), ref, shape)
    if s_sh is not None:
        x = orc.to_f64(L["x"], shape.act_dtype)
        ws_ = orc.to_f64(L["w_shared"], shape.act_dtype)
        want = np.array([orc.shared_gate(x[t], ws_) for t in range(T)])
        np.testing.assert_allclose(s_sh.cpu().numpy(), want, atol=1e-5)


BUCKET_CASES = [(1, 8, 256), (8, 8, 256), (64, 8, 256), (32, 4, 16), (37, 4, 16),
                (4096, 8, 256), (4096, 8, 128), (2048, 2, 8), (5000, 3, 60), (1000, 32, 512)]


@pytest.mark.parametrize("T,k,E", BUCKET_CASES)
def test_bucket_parity(T, k, E):
    rng = np.random.default_rng(T * 7 + k + E)
    # skewed but valid ids (distinct per token)
    p = rng.zipf(1.5, size=E).astype(np.float64)
    p /= p.sum()
    ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    ref = orc.bucket(ids, E)
    cfg = smr.MoEConfig(T=T, d_model=64, n_experts=E, top_k=k, d_ff=64, d_ff_shared=0)
    ws = smr.alloc_workspace(cfg)
    i32 = lambda n: torch.full((n,), -7, dtype=torch.int32, device="cuda")
    counts, offsets, active, n_active = i32(E), i32(E + 1), i32(E), i32(4)
    perm, pos = i32(T * k), i32(T * k)
    smr.bucket(cfg, ws, to_dev(ids), counts, offsets, active, n_active, perm, pos)
    assert smr.read_device_status(cfg, ws)[0] == 0
    na = int(n_active[0])
    assert na == len(ref["active"])
    assert counts.cpu().numpy().tolist() == ref["counts"].tolist()
    assert offsets.cpu().numpy().tolist() == ref["offsets"].tolist()
    assert active.cpu().numpy()[:na].tolist() == ref["active"].tolist()
    assert perm.cpu().numpy().tolist() == ref["perm"].tolist()
    assert pos.cpu().numpy().tolist() == ref["pos"].tolist()


@pytest.mark.parametrize("T", [16, 3000], ids=["one-cta", "multi-cta"])
def test_bucket_flags_out_of_range_ids(T):
    k, E = 4, 16
    ids = np.arange(T * k, dtype=np.int32).reshape(T, k) % E
    ids[3, 1] = E + 5
    ids[7, 0] = -1
    ids[T - 1, 3] = 1 << 30
    cfg = smr.MoEConfig(T=T, d_model=64, n_experts=E, top_k=k, d_ff=64, d_ff_shared=0)
    ws = smr.alloc_workspace(cfg)
    i32 = lambda n: torch.zeros((n,), dtype=torch.int32, device="cuda")
    perm = i32(T * k)
    smr.bucket(cfg, ws, to_dev(ids), i32(E), i32(E + 1), i32(E), i32(4), perm, i32(T * k))
    st, word = smr.read_device_status(cfg, ws)
    assert st == smr._STATUS.index("MOE_ERR_DEVICE_CHECK")
    assert word & 1 and (word >> 16) == 1
    # every access stayed in bounds: perm is still a permutation of the pairs
    assert sorted(perm.cpu().numpy().tolist()) == list(range(T * k))
    # the word was cleared by the read
    assert smr.read_device_status(cfg, ws)[0] == 0


EXPERT_CASES = [(mi.TINY_F32, 32, 32), (mi.QWEN36, 64, 64), (mi.DEEPSEEK_GROUP, 4096, 16),
                (mi.QWEN36, 8, 8), (mi.TINY_F32.with_(name="tiny_f32_t3"), 3, 3)]


@pytest.mark.parametrize("shape,T,n_check", EXPERT_CASES,
                         ids=["%s-T%d" % (c[0].name, c[1]) for c in EXPERT_CASES])
def test_experts_forward_parity_given_routing(shape, T, n_check):
    """The expert half on its own, fed routing artefacts that do not come
    from the GPU router (no near-tie can interfere)."""
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    ids, w, s = mi.random_router_outputs(shape, T)
    cfg = cfg_for(shape, T)
    ws = smr.alloc_workspace(cfg)
    for gate_given in (False, True):
        sh = dev.shared()
        smr.experts_forward(cfg, ws, dev.t["x"], dev.t["r_attn"], to_dev(ids), to_dev(w),
                            dev.bank("W_gate"), dev.bank("W_up"), dev.bank("W_down"), dev.out,
                            s_shared=to_dev(s) if gate_given else None, **sh)
        assert smr.read_device_status(cfg, ws)[0] == 0
        rows = _sample(T, n_check, seed=3)
        ref = orc.moe_experts_forward(L, shape, ids, w.astype(np.float64),
                                      s.astype(np.float64) if gate_given else None, rows)
        err = rel_rms_err(dev.out.cpu().numpy()[rows], ref["out"])
        assert err <= OUT_TOL[shape.act_dtype], err


@pytest.mark.parametrize("path", [smr.PATH_GEMV, smr.PATH_FUSED], ids=["gemv", "fused"])
@pytest.mark.parametrize("shape,T", [(mi.QWEN36, 2), (mi.TINY_F32, 3), (mi.QWEN36, 16)],
                         ids=["qwen-T2", "tiny-T3", "qwen-T16"])
def test_small_batch_with_an_expert_repeated_within_a_token(shape, T, path):
    """Caller-given ids may name one expert in several slots of a token, so an
    expert's group can hold more pairs than the batch has tokens; the
    direct-load GEMV and the single-launch decode kernel then walk the group
    in chunks of tokens."""
    if path == smr.PATH_GEMV and T > 8:
        pytest.skip("the direct-load GEMV takes up to 8 tokens")
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    ids, w, s = mi.random_router_outputs(shape, T)
    ids[:, : shape.top_k // 2] = 3          # expert 3 in half the slots of every token
    cfg = cfg_for(shape, T, path)
    ws = smr.alloc_workspace(cfg)
    sh = dev.shared()
    smr.experts_forward(cfg, ws, dev.t["x"], dev.t["r_attn"], to_dev(ids), to_dev(w),
                        dev.bank("W_gate"), dev.bank("W_up"), dev.bank("W_down"), dev.out,
                        s_shared=to_dev(s), **sh)
    assert smr.read_device_status(cfg, ws)[0] == 0
    ref = orc.moe_experts_forward(L, shape, ids, w.astype(np.float64), s.astype(np.float64),
                                  np.arange(T))
    assert rel_rms_err(dev.out.cpu().numpy(), ref["out"]) <= OUT_TOL[shape.act_dtype]


@pytest.mark.parametrize("path,site", [(smr.PATH_GEMV, 2), (smr.PATH_FUSED, 9)],
                         ids=["gemv", "fused"])
def test_few_token_paths_flag_out_of_range_ids(path, site):
    """Batches of a few tokens skip the bucketing pass (the direct-load GEMV
    treats each pair as its own group; the single-launch decode kernel groups
    pairs itself), so these kernels check the ids themselves: a bad id is
    flagged in the status word and its pair is skipped, with every access in
    bounds."""
    shape, T = mi.QWEN36, 2
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    ids, w, s = mi.random_router_outputs(shape, T)
    ids[1, 3] = shape.n_experts + 7
    cfg = cfg_for(shape, T, path)
    ws = smr.alloc_workspace(cfg)
    smr.experts_forward(cfg, ws, dev.t["x"], dev.t["r_attn"], to_dev(ids), to_dev(w),
                        dev.bank("W_gate"), dev.bank("W_up"), dev.bank("W_down"), dev.out,
                        s_shared=to_dev(s), **dev.shared())
    st, word = smr.read_device_status(cfg, ws)
    assert st == smr._STATUS.index("MOE_ERR_DEVICE_CHECK")
    assert word & 1 and (word >> 16) == site
    # token 0 does not involve the bad pair and is still exact
    ref = orc.moe_experts_forward(L, shape, ids[:1], w[:1].astype(np.float64),
                                  s[:1].astype(np.float64), np.arange(1))
    assert rel_rms_err(dev.out.cpu().numpy()[:1], ref["out"]) <= OUT_TOL[shape.act_dtype]


def test_in_place_residual_update():
    shape, T = mi.QWEN36, 8
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    cfg = cfg_for(shape, T)
    ws = smr.alloc_workspace(cfg)
    dev.layer_forward(cfg, ws)
    want = dev.out.clone()
    dev.out = dev.t["r_attn"]          # out aliases r_attn
    dev.layer_forward(cfg, ws)
    assert torch.equal(dev.t["r_attn"], want)


@pytest.mark.parametrize("T", [4, 64])
def test_repeat_calls_are_deterministic(T):
    shape = mi.QWEN36
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    cfg = cfg_for(shape, T)
    ws = smr.alloc_workspace(cfg)
    dev.layer_forward(cfg, ws)
    a = dev.out.clone()
    ids = dev.ids.clone()
    for _ in range(3):
        dev.layer_forward(cfg, ws)
        assert torch.equal(dev.out, a)
        assert torch.equal(dev.ids, ids)


CONSISTENCY_CASES = [(mi.QWEN36, 1), (mi.QWEN36, 37), (mi.QWEN36, 64), (mi.DEEPSEEK_GROUP, 8),
                     (mi.TINY_F32, 32), (mi.QWEN36, 600)]


FUSED_CONSISTENCY = [(mi.QWEN36, 1, smr.PATH_FUSED), (mi.QWEN36, 16, smr.PATH_FUSED),
                     (mi.DEEPSEEK_GROUP, 8, smr.PATH_FUSED),
                     (mi.TINY_F32.with_(name="tiny_f32_t5"), 5, smr.PATH_FUSED)]


@pytest.mark.parametrize("shape,T,path", [c + (smr.PATH_AUTO,) for c in CONSISTENCY_CASES] +
                         FUSED_CONSISTENCY,
                         ids=["%s-T%d" % (c[0].name, c[1]) for c in CONSISTENCY_CASES] +
                         ["%s-T%d-fused" % (c[0].name, c[1]) for c in FUSED_CONSISTENCY])
def test_layer_matches_route_then_experts(shape, T, path):
    """moe_layer_forward against moe_route followed by moe_experts_forward on
    the same inputs: the same kernels in the same order, so ids, weights and
    the layer output must agree bit for bit."""
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    cfg = cfg_for(shape, T, path)
    ws = smr.alloc_workspace(cfg)
    dev.layer_forward(cfg, ws)
    assert smr.read_device_status(cfg, ws)[0] == 0
    ids2, w2 = torch.empty_like(dev.ids), torch.empty_like(dev.w)
    sh = dev.shared()
    s2 = torch.empty(T, dtype=torch.float32, device="cuda") if shape.d_ff_shared else None
    ws2 = smr.alloc_workspace(cfg)
    smr.route(cfg, ws2, dev.t["x"], dev.t["W_router"], ids2, w2,
              expert_bias=dev.t.get("expert_bias"), w_shared=sh["w_shared"], s_shared=s2)
    assert torch.equal(ids2, dev.ids)
    assert torch.equal(w2, dev.w)
    out2 = torch.empty_like(dev.out)
    smr.experts_forward(cfg, ws2, dev.t["x"], dev.t["r_attn"], ids2, w2, dev.bank("W_gate"),
                        dev.bank("W_up"), dev.bank("W_down"), out2, s_shared=s2, **sh)
    assert smr.read_device_status(cfg, ws2)[0] == 0
    assert torch.equal(out2, dev.out)


def test_workspace_reuse_across_batch_sizes():
    """The multi-CTA bucketing pass hands work between CTAs with a
    self-resetting arrival counter in the workspace: alternating batch sizes
    (one-CTA and multi-CTA bucketing) on one workspace must give the same
    results as fresh workspaces."""
    shape = mi.QWEN36
    big = cfg_for(shape, 600)
    ws = smr.alloc_workspace(big)
    outs = {}
    for T in (600, 5, 1, 600, 64, 5):
        L = layer_host(shape, T)
        dev = DevLayer(shape, L)
        dev.layer_forward(cfg_for(shape, T), ws)
        if T in outs:
            assert torch.equal(outs[T][0], dev.out) and torch.equal(outs[T][1], dev.ids)
        else:
            fresh = smr.alloc_workspace(cfg_for(shape, T))
            ref = DevLayer(shape, L)
            ref.layer_forward(cfg_for(shape, T), fresh)
            assert torch.equal(ref.out, dev.out) and torch.equal(ref.ids, dev.ids)
            outs[T] = (dev.out.clone(), dev.ids.clone())
    assert smr.read_device_status(big, ws)[0] == 0


def test_degenerate_shapes():
    """k = E (every expert selected), E = 1 (dense), k = 1."""
    for E, k in ((4, 4), (1, 1), (16, 1)):
        shape = mi.TINY_F32.with_(name="deg", n_experts=E, top_k=k)
        T = 9
        L = mi.make_layer(shape, T)
        dev = DevLayer(shape, L)
        cfg = cfg_for(shape, T)
        ws = smr.alloc_workspace(cfg)
        dev.layer_forward(cfg, ws)
        assert smr.read_device_status(cfg, ws)[0] == 0
        ref = orc.moe_layer_forward(L, shape)
        ids = dev.ids.cpu().numpy()
        assert [sorted(r) for r in ids.tolist()] == [sorted(r) for r in ref["ids"].tolist()]
        assert rel_rms_err(dev.out.cpu().numpy(), ref["out"]) <= OUT_TOL["f32"]


def test_zero_tokens_is_a_no_op():
    shape = mi.QWEN36
    cfg = cfg_for(shape, 0)
    ws = smr.alloc_workspace(cfg)
    L = layer_host(shape, 1)
    dev = DevLayer(shape, L)
    empty = torch.empty((0, shape.d_model), dtype=torch.bfloat16, device="cuda")
    smr.layer_forward(cfg, ws, empty, dev.t["r_attn"][:0], dev.t["W_router"],
                      dev.bank("W_gate"), dev.bank("W_up"), dev.bank("W_down"),
                      dev.out[:0], dev.ids[:0], dev.w[:0], **dev.shared())
    assert smr.read_device_status(cfg, ws)[0] == 0


# A small shape whose experts each hold several 128-row tiles with a ragged
# tail (E = 4, k = 2, T = 400: ~200 rows per expert), two N tiles of gate/up
# (I = 256) and two of down (d = 512), with a full fp64 oracle.
TC_SMALL = mi.MoEShape("tc_small", 7, d_model=512, n_experts=4, top_k=2, d_ff=256,
                       d_ff_shared=256, tokens=(400,))
# Qwen3.6 at T = 16, 17, 64, 65: the A tiles of routed batches are 16 rows
# tall up to T = 16 and 64 rows up to T = 64 (the shared expert's group holds
# all T rows), so these sit at and just past each box edge.
PATH_CASES = [(TC_SMALL, 400), (TC_SMALL, 700), (TC_SMALL, 37), (TC_SMALL, 1), (mi.QWEN36, 64),
              (mi.QWEN36, 16), (mi.QWEN36, 17), (mi.QWEN36, 65),
              (mi.QWEN36, 8), (mi.QWEN36, 5), (mi.DEEPSEEK_GROUP, 6),
              (mi.DEEPSEEK_GROUP, 37)]


@pytest.mark.parametrize("path", [smr.PATH_GEMV, smr.PATH_TC, smr.PATH_FUSED],
                         ids=["gemv", "tc", "fused"])
@pytest.mark.parametrize("shape,T", PATH_CASES,
                         ids=["%s-T%d" % (c[0].name, c[1]) for c in PATH_CASES])
def test_every_expert_path_matches_oracle(shape, T, path):
    """The CUDA-core streaming path, the tcgen05 grouped-GEMM path and the
    single-launch decode kernel (batches of up to 16 tokens), each forced,
    against the oracle on every output row."""
    if path == smr.PATH_FUSED and T > 16:
        pytest.skip("the single-launch decode kernel takes up to 16 tokens")
    L, dev, cfg, ws = _run_layer(shape, T, path)
    _check_rows(L, shape, T, dev, "all")


# 4-bit affine group-64 experts (dequantised inside the tensor-core kernel):
# a small full-oracle shape and the Mixtral-style layer at T=2048.
Q4_SMALL = mi.MoEShape("q4_small", 8, d_model=512, n_experts=4, top_k=2, d_ff=256,
                       d_ff_shared=0, expert_dtype="q4", tokens=(300,))
# T=700: 350 rows per expert on average, so the 4-bit items pair row blocks
# (with ragged pairs at every group's end)
Q4_CASES = [(Q4_SMALL, 300, "all"), (Q4_SMALL, 700, "all"), (Q4_SMALL, 37, "all"),
            (Q4_SMALL, 1, "all"), (mi.MIXTRAL_Q4, 2048, "blocks")]


@pytest.mark.parametrize("shape,T,mode", Q4_CASES,
                         ids=["%s-T%d" % (c[0].name, c[1]) for c in Q4_CASES])
def test_q4_layer_forward_parity(shape, T, mode):
    L, dev, cfg, ws = _run_layer(shape, T)
    _check_rows(L, shape, T, dev, mode, seed=5)


def test_q4_experts_forward_given_routing():
    shape, T = Q4_SMALL, 300
    L = layer_host(shape, T)
    dev = DevLayer(shape, L)
    ids, w, s = mi.random_router_outputs(shape, T, seed=4)
    cfg = cfg_for(shape, T)
    ws = smr.alloc_workspace(cfg)
    smr.experts_forward(cfg, ws, dev.t["x"], dev.t["r_attn"], to_dev(ids), to_dev(w),
                        dev.bank("W_gate"), dev.bank("W_up"), dev.bank("W_down"), dev.out)
    assert smr.read_device_status(cfg, ws)[0] == 0
    ref = orc.moe_experts_forward(L, shape, ids, w.astype(np.float64))
    assert rel_rms_err(dev.out.cpu().numpy(), ref["out"]) <= OUT_TOL["bf16"]
