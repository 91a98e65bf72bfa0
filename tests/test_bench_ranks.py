"""Multi-rank plumbing of bench.py on CPU: two gloo ranks, as torchrun would
start them (replicas only: the process group carries the barrier and the max
of the times, no layer data)."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    w, r, local = bench.init_ranks("gloo")
    ms = bench.max_over_ranks(10.0 + 5.0 * r, torch.device("cpu"))    # rank 1 is slower
    value = bench.job_tokens_per_s(w, 64, 100, ms)
    with open(os.path.join(out_dir, "rank%d.json" % r), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "ms": ms, "value": value}, f)
    bench.finish_ranks()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    for r, d in enumerate(res):
        assert d["world"] == 2 and d["rank"] == r and d["local"] == r
        assert d["ms"] == 15.0                       # max over ranks, on every rank
        # whole-job tokens/s: 2 replicas x 64 tokens x 100 steps in 15 ms
        assert d["value"] == pytest.approx(2 * 64 * 100 / 15e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""             # non-zero ranks exit without work


def test_single_rank_needs_no_process_group():
    torch = pytest.importorskip("torch")
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.init_ranks("gloo") == (1, 0, 0)
    assert not torch.distributed.is_initialized()
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
