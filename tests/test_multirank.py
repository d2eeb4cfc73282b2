"""Host logic of multi-rank runs, on two gloo ranks on the CPU.

The verify step shards by sequence: each rank verifies its own batch, and the
only collective is the max-over-ranks of the timings.  These tests check that
logic (seeds per rank, the MAX reduction, whole-job throughput, rank-0-only
reference arm) and that a rank's result does not depend on the other rank.
"""
import json
import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as bm
    import oracle
    import workloads as wl
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_max = bm.max_over_ranks(1.5 + rank, world, "cpu")
        seed = bm.rank_seed("tiny", rank)
        inp = wl.make("tiny", "cpu", seed=seed, B=3, plant="hash")
        res = oracle.verify_step(wl.to_numpy(inp))
        args = types.SimpleNamespace(steps=1, warmup=0, workload="tiny", batch=None)
        ref_line = bm.bench_reference(args, rank, world) if rank != 0 else "rank0-skipped"
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"t_max": t_max, "seed": seed,
                       "out_tokens": res["out_tokens"].tolist(),
                       "n_emit": res["n_emit"].tolist(),
                       "ref_line": ref_line}, f)
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks(tmp_path_factory, oracle_mod):
    out = tmp_path_factory.mktemp("ranks")
    mp.start_processes(_rank_main, args=(2, _free_port(), str(out)), nprocs=2,
                       start_method="spawn", join=True)
    return [json.load(open(out / f"rank{r}.json")) for r in range(2)]


def test_max_over_ranks_is_max_on_every_rank(two_ranks):
    assert [r["t_max"] for r in two_ranks] == [2.5, 2.5]


def test_each_rank_has_its_own_batch(two_ranks):
    s0, s1 = two_ranks[0]["seed"], two_ranks[1]["seed"]
    assert s0 == workloads.get("tiny").seed and s1 == s0 + 1


def test_rank_results_equal_single_process(two_ranks, oracle_mod):
    """No data-path collective: a rank's step equals the same batch run alone."""
    import oracle
    for r, got in enumerate(two_ranks):
        inp = workloads.make("tiny", "cpu", seed=workloads.get("tiny").seed + r, B=3,
                             plant="hash")
        res = oracle.verify_step(workloads.to_numpy(inp))
        assert got["out_tokens"] == res["out_tokens"].tolist()
        assert got["n_emit"] == res["n_emit"].tolist()
    assert two_ranks[0]["out_tokens"] != two_ranks[1]["out_tokens"]


def test_reference_arm_runs_on_rank0_only(two_ranks):
    assert two_ranks[1]["ref_line"] is None


def test_job_throughput():
    # 2 ranks x 100 steps, slowest rank 50 ms -> 4000 steps/s for the job
    assert bench.job_throughput(2, 100, 50.0) == pytest.approx(4000.0)
    assert bench.job_throughput(1, 1, 1000.0) == pytest.approx(1.0)
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_reference_plan_fits_budget():
    # all heads fit: 300 steps x (0.2 + 0.01) s < 150 s? no -> fewer heads
    h = bench.reference_plan(0.2, 0.01, 32, 300, 5, budget_s=150.0)
    assert 1 <= h <= 32
    assert (300 + 5) * (0.2 * h / 32 + 0.01) <= 150.0
    assert bench.reference_plan(0.2, 0.01, 32, 10, 1, budget_s=150.0) == 32
    assert bench.reference_plan(100.0, 0.0, 32, 300, 5, budget_s=150.0) == 1


def test_reference_arm_line_single_rank(oracle_mod):
    args = types.SimpleNamespace(steps=2, warmup=1, workload="tiny", batch=None)
    line = bench.bench_reference(args, 0, 1)
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the same workload as the GPU arm's line; only the L2 statement differs
    ours = bench.workload_config("tiny")
    assert {k: v for k, v in line["config"].items() if k != "l2"} == \
        {k: v for k, v in ours.items() if k != "l2"}
    sf = line["scaled_from"]
    assert sf["sequences_timed_per_step"] == 1 and sf["steps_timed"] == 2
    assert sf["factor"] == sf["batch"] * sf["query_heads"] / sf["query_heads_timed"]
