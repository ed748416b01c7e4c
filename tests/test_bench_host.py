"""Host-side logic of bench.py: byte accounting, replica seeding and the
multi-rank timing reduction (two gloo ranks on CPU, no GPU)."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from synth import CONFIGS


def test_algorithmic_bytes_per_block():
    # W2 + U + gathered W1 rows per step, plus h for the confidence head / gate, plus Wg
    assert bench.algorithmic_bytes(0, CONFIGS[0]) == 8_456_192
    assert bench.algorithmic_bytes(1, CONFIGS[1]) == 1_254_391_808
    assert bench.algorithmic_bytes(2, CONFIGS[2]) == 2_498_756_608
    assert bench.algorithmic_bytes(3, CONFIGS[3]) == 1_877_999_616
    assert bench.algorithmic_bytes(4, CONFIGS[4]) == 2_596_536_320
    assert bench.algorithmic_bytes(5, CONFIGS[5]) == 1_880_096_768  # gated + the decay gate


def test_verify_and_label_bytes():
    B, K, V, r = 128, 16, 151936, 256
    c = CONFIGS[2]
    # every verified target row (window and bonus), W2, and the base-logit, embedding and
    # target rows at the draw position
    assert bench.verify_bytes(c) == (B * (K + 1) * V * 4 + r * V * 2 + B * V * 4 + B * r * 2
                                     + B * V * 4)
    # U and the target rows of the K positions once, W2 once, the gathered embeddings
    assert bench.label_bytes(c) == 2 * B * K * V * 4 + r * V * 2 + B * K * r * 2
    assert bench.metric_of("label") == bench.LABEL_METRIC
    assert bench.metric_of("verify") == bench.VERIFY_METRIC
    assert bench.metric_of("serving") == bench.METRIC


def test_single_cta_kernel_op_counts():
    # 2048 candidates: a bitonic network of 11 * 12 / 2 = 66 stages over every element,
    # then the prefix sum and the cut
    assert bench.schedule_ops(128, 16) == 2048 * 66 + 2 * 2048
    assert bench.schedule_ops(7, 3) == 32 * 15 + 2 * 21  # 21 candidates padded to 32
    # every row x position x round (8) x grid point (32)
    assert bench.sts_ops(8192, 16) == 4 * 8192 * 16 * 8 * 32  # four SFU results per evaluation
    assert bench.metric_of("schedule") == bench.SCHEDULE_METRIC
    assert bench.metric_of("sts") == bench.STS_METRIC


def test_replica_seeds_are_distinct_per_rank_and_step():
    seeds = {bench.replica_seed(r, s) for r in range(8) for s in range(100)}
    assert len(seeds) == 800
    assert bench.replica_seed(0, 7) == 7


def test_job_throughput_is_weak_scaling():
    one = bench.job_throughput(2048, 10, 1, 5.0)
    assert bench.job_throughput(2048, 10, 4, 5.0) == pytest.approx(4 * one)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    bench.barrier(world)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    value = bench.job_throughput(128 * 16, 20, world, slowest)
    q.put((rank, slowest, value))
    dist.destroy_process_group()


def test_two_rank_timing_reduction_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time and the same whole-job throughput
    assert res[0][1] == res[1][1] == 15.0
    assert res[0][2] == res[1][2] == pytest.approx(2 * 128 * 16 * 20 / 0.015)


def test_profile_hash_ignores_comments_but_not_code():
    """A committed ncu summary stays valid across comment edits of the kernel
    sources and is retired by any change to their code."""
    src = "int f(int x) {  // doubles x\n  /* body */ return 2 * x;\n}\n"
    assert bench._code_only(src) == bench._code_only(
        "// header comment\nint f(int x) {\n  return 2 * x;   /* changed note */\n}\n")
    assert bench._code_only(src) != bench._code_only("int f(int x) {\n  return 3 * x;\n}\n")
    assert len(bench.kernel_source_hash("serving")) == 16


def test_profiles_name_existing_sources_and_carry_their_figures():
    """Every workload with a committed ncu summary names kernel sources that exist, and the
    summary carries the source hash and the per-launch DRAM bytes the bench reads."""
    import re
    for workload, (summary, sources) in bench.PROFILES.items():
        for name in sources:
            assert os.path.exists(os.path.join(bench.ROOT, "rank_markov_draft_gb300", "csrc", name)), name
        text = open(os.path.join(bench.ROOT, "profiles", summary)).read()
        assert re.search(r"kernel source hash:\s*`[0-9a-f]{16}`", text), summary
        assert re.search(r"dram bytes per launch:\s*`[0-9]+`", text), summary
