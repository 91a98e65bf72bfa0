"""The algorithmic work bench.py divides by: bytes and flops of one layer and of
one gate/up launch, checked against figures worked out by hand from the
shapes the pages give (Treebeard "Model constants": d 2048, 256 experts, top-8,
expert and shared width 512; Airframe model table: Mixtral 8 experts, top-2,
d 4096, width 14336; Edge0 tier table: 4-bit affine, group 64). No GPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_inputs as mi  # noqa: E402

QWEN = mi.PRESETS["qwen36_decode"]
MIX = mi.PRESETS["mixtral_bf16"]
MIX_Q4 = mi.PRESETS["mixtral_q4"]


def test_bytes_per_active_expert():
    # gate + up + down of one expert: 3 x 512 x 2048 bf16 = 6,291,456 B
    assert bench.layer_bytes(QWEN, 1, 9) - bench.layer_bytes(QWEN, 1, 8) == 6_291_456
    # Mixtral: 3 x 14336 x 4096 bf16 = 352,321,536 B
    assert bench.layer_bytes(MIX, 1, 2) - bench.layer_bytes(MIX, 1, 1) == 352_321_536
    # 4-bit: half a byte per weight plus a bf16 scale and min per 64 weights
    # = 0.5625 B per weight: 176,160,768 x 0.5625 = 99,090,432 B
    assert bench.layer_bytes(MIX_Q4, 1, 2) - bench.layer_bytes(MIX_Q4, 1, 1) == 99_090_432


def test_qwen_decode_t1_layer():
    # router 256 x 2048 x 2 + w_shared 2048 x 2 + 8 experts + shared expert
    # + x (2048 x 2) + r_attn and out (2 x 2048 x 4) + ids and weights (8 x 8)
    expect = 1_048_576 + 4_096 + 8 * 6_291_456 + 6_291_456 + 4_096 + 16_384 + 64
    assert expect == 57_696_320
    assert bench.layer_bytes(QWEN, 1, 8) == expect
    # flops: router 2 x 2048 x 257, 8 routed pairs x 3 x 2 x 2048 x 512, shared
    assert bench.layer_flops(QWEN, 1) == 1_052_672 + 50_331_648 + 6_291_456
    # floor at the measured copy rate used in the tables: 8.65 us
    assert bench.layer_bytes(QWEN, 1, 8) / 6668.9e9 * 1e6 == pytest.approx(8.652, abs=1e-3)


def test_prefill_and_mixtral_flops():
    # Qwen T=4096: 2*4096*2048*257 + 2*4096*8*3*2048*512 + 2*4096*3*2048*512
    assert bench.layer_flops(QWEN, 4096) == 4_311_744_512 + 206_158_430_208 + 25_769_803_776
    # Mixtral T=2048, no shared expert: 2*2048*4096*8 + 2*2048*2*3*4096*14336
    f = bench.layer_flops(MIX, 2048)
    assert f == 134_217_728 + 1_443_109_011_456
    # tensor floor at the measured bf16 rate: about 756 us
    assert f / 1909.9e12 * 1e6 == pytest.approx(755.65, abs=0.05)


def test_gateup_launch_unit():
    # one unit = gate + up rows of one expert: 2 x 512 x 2048 x 2 = 4,194,304 B
    b1, f1 = bench.gateup_work(QWEN, 64, 1)
    b2, f2 = bench.gateup_work(QWEN, 64, 2)
    assert b2 - b1 == 4_194_304
    assert f1 == f2  # flops follow the routed pairs, not the active count
    # T=64 with 223 active experts: 223 units + the shared expert + x
    b, f = bench.gateup_work(QWEN, 64, 223)
    assert b == 224 * 4_194_304 + 64 * 2048 * 2
    # 2 x 2048 x 1024 per routed pair (512 pairs) and per shared row (64)
    assert f == (512 + 64) * 2 * 2048 * 1024


def test_expert_path_labels_follow_the_automatic_choice():
    # MOE_PATH_AUTO (path 0): GEMV chain up to 3 tokens, the single launch for
    # 4-16 tokens on the narrow bf16 shapes (d_model <= 2048, widths <= 1024),
    # the tensor-core path above 16 tokens and on the wider shapes from 6
    auto = 0
    assert bench._expert_path(QWEN, 3, auto) == "CUDA-core direct-load GEMV"
    for T in (4, 8, 16):
        assert bench._expert_path(QWEN, T, auto) == "single-launch decode kernel"
    assert bench._expert_path(QWEN, 17, auto) == "tcgen05 grouped GEMM"
    assert bench._expert_path(MIX, 5, auto) == "CUDA-core direct-load GEMV"
    assert bench._expert_path(MIX, 8, auto) == "tcgen05 grouped GEMM"
    assert bench._expert_path(MIX_Q4, 8, auto) == "tcgen05 grouped GEMM"
    # forced single launch (path 3) up to 16 tokens, on any shape
    assert bench._expert_path(MIX, 3, 3) == "single-launch decode kernel"
    assert bench._expert_path(QWEN, 17, 3) != "single-launch decode kernel"


def test_expert_path_labels_of_other_shapes():
    # a shared expert wider than the routed ones (5632 against 1408) runs as
    # its own tensor-core launches; widths above 1024 leave the single launch
    q60 = mi.PRESETS["qwen_moe_60"]
    assert bench._expert_path(q60, 64, 0) == "tcgen05 grouped GEMM"
    assert bench._expert_path(q60, 8, 0) == "tcgen05 grouped GEMM"
    assert bench._expert_path(q60, 5, 0) == "CUDA-core direct-load GEMV"
    tiny = mi.PRESETS["tiny_f32"]
    assert bench._expert_path(tiny, 32, 0) == "CUDA-core streaming GEMV"
