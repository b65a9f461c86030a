"""Multi-rank host logic on CPU with two gloo ranks (no GPU): expert shards chosen by
group_offset add up to the full grouped matmul, and the benchmark's time is the slowest
rank's."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from moe_grouped_matrix_gb300.sharding import expert_shard, max_over_ranks


def test_expert_shard_covers_every_expert_once():
    for G in (1, 7, 8, 64, 128):
        for world in range(1, min(G, 9) + 1):
            seen = []
            for r in range(world):
                go, L = expert_shard(G, r, world)
                assert L >= 1
                seen.extend(range(go, go + L))
            assert seen == list(range(G))
    with pytest.raises(ValueError):
        expert_shard(3, 0, 4)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from moe_grouped_matrix_gb300 import workloads as W

        G, m, k, n = 6, 40, 32, 16
        sizes = np.array([7, 0, 12, 5, 9, 4], np.int32)
        lhs = W.stored_bits(W.normal((m, k), 1.0, 1))
        rhs = W.stored_bits(W.normal((G, n, k), 0.1, 2))
        go, L = expert_shard(G, rank, world)
        part, _ = oracle.gmm(lhs, rhs[go:go + L], sizes, group_offset=go)
        t = torch.from_numpy(part)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        full, _ = oracle.gmm(lhs, rhs, sizes)
        ok_sum = bool(np.array_equal(t.numpy(), full))
        slowest = max_over_ranks(10.0 + rank)
        with open(os.path.join(result_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{int(ok_sum)} {slowest}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_expert_parallel_sum_and_max_time(tmp_path, oracle_lib):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        ok, slowest = open(tmp_path / f"rank{r}.txt").read().split()
        assert ok == "1", "expert shards do not add up to the full result"
        assert float(slowest) == 11.0

