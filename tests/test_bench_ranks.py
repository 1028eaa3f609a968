"""The replica path of bench.py on CPU with two gloo ranks: the timed region
is the maximum over ranks, the whole-job rate counts every replica's work,
the reference arm runs on rank 0 only, and the per-token cost model
matches the pages' worked example."""
import json
import os
import pathlib
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    local_ms = 100.0 + 50.0 * rank  # rank 1 is the slower replica
    ms = bench.reduce_max(local_ms, world)
    value, verified = bench.job_rates(world, 1, 10, ms, 3.0)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, value, verified))


def test_two_ranks_take_the_slowest_replica():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value, verified in out:
        assert ms == 150.0                          # max over ranks
        assert value == pytest.approx(2 * 1 * 10 / 0.150)   # both replicas' draft blocks
        assert verified == pytest.approx(2 * 3.0 * 10 / 0.150)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(12.5, 1) == 12.5
    value, verified = bench.job_rates(1, 32, 4, 200.0, 64.0)
    assert value == pytest.approx(32 * 4 / 0.2) and verified == pytest.approx(64 * 4 / 0.2)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"workload": "qwen3-8b-b1", "steps": 1, "warmup": 0, "gpus": 2})()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""


def test_cost_model_matches_the_worked_example():
    """The bench's per-token cost against the pages' worked example: a 3 ms
    draft and a 20 ms verification (a 23 ms cycle) cost about 3.8 ms a token
    at 6 tokens per round and 11.5 ms at 2."""
    import bench
    g = json.loads((pathlib.Path(__file__).parent / "golden" / "cost_model_example.json").read_text())
    cycle = g["t_draft_ms"] + g["t_verify_ms"]
    for case in g["cases"]:
        c = bench.cost_model(g["t_draft_ms"], cycle, case["accepted"])
        assert abs(c["per_token_ms"] - case["ms_per_token"]) <= case["abs_tol"]
        assert c["verify_and_fusion_ms"] == g["t_verify_ms"]
    sp = g["baseline_ms_per_token"] / bench.cost_model(g["t_draft_ms"], cycle, 6)["per_token_ms"]
    assert abs(sp - g["speedup_at_6"]) <= g["speedup_tol"]


def test_gemm_flops_of_the_32_sequence_cycle():
    """The tensor roofline's algorithmic flops: 2 per multiply-add of every
    projection weight with every row it multiplies (41 layers of 512 block
    rows; the fusion projections over the committed rows), written out from
    the Qwen3-8B layer shape (32 query heads, 8 KV heads, head dim 128,
    hidden 4096, MLP 12288)."""
    sys.path.insert(0, ROOT)
    import bench
    from block_diffusion_speculative_step_gb300 import synth

    w = synth.WORKLOADS["qwen3-8b-b32"]
    layer = (32 + 2 * 8) * 128 * 4096 + 4096 * 32 * 128 + 3 * 4096 * 12288  # 192,937,984 weights
    assert layer == 192_937_984
    rows = 32 * 16
    fuse = 4096 * 5 * 4096 + 5 * 2 * 8 * 128 * 4096  # FC over 5 taps + K/V injection of 5 draft layers
    assert bench.gemm_flops_per_cycle(w, 0) == 2.0 * rows * 41 * layer
    assert bench.gemm_flops_per_cycle(w, 183) == 2.0 * (rows * 41 * layer + 183 * fuse)
