"""The multi-process (N>1) path of the benchmark on the CPU: two gloo ranks
run the replica helpers that bench.py uses under torchrun with one GPU per
rank -- rank environment, barrier, max over ranks, whole-job throughput and
per-rank token streams -- and the reference arm's rank != 0 exit."""
import os
import socket
import sys
import time

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from autograd_arena_allocated_gb300 import replicas, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        info = replicas.rank_env()
        g = replicas.Group(dist, device="cpu")
        g.barrier()
        # ranks take different times; the job is as slow as its slowest rank
        t0 = time.perf_counter()
        time.sleep(0.05 * (rank + 1))
        mine = time.perf_counter() - t0
        slowest = g.max(mine)
        tok, _ = synth.token_stream(2, 16, 50257, "zipf", seed=replicas.token_seed(synth.TOKEN_SEED, rank))
        sys.path.insert(0, ROOT)
        import bench

        class Args:
            workload, ref_tokens, warmup, steps = "tiny_fp32", 8, 0, 1

        ref_rc = bench.run_reference(Args, world, rank) if rank != 0 else 0
        out[rank] = dict(world=info.world, rank=info.rank, local=info.local, group_world=g.world,
                         mine=mine, slowest=slowest, tok=tok.tolist(), ref_rc=ref_rc)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in range(world):
        assert (res[r]["world"], res[r]["rank"], res[r]["local"], res[r]["group_world"]) == (world, r, r, world)
        assert res[r]["ref_rc"] == 0
    # both ranks agree on the max, and it is the slower rank's own time
    assert res[0]["slowest"] == res[1]["slowest"] == max(res[0]["mine"], res[1]["mine"])
    assert res[1]["mine"] > res[0]["mine"]
    # rank 0 draws the single-GPU token stream, rank 1 an independent one
    single, _ = synth.token_stream(2, 16, 50257, "zipf")
    assert np.array_equal(np.array(res[0]["tok"]), single)
    assert not np.array_equal(np.array(res[1]["tok"]), single)


def test_single_process_group_is_noop():
    calls = []
    g = replicas.Group(None, sync=lambda: calls.append(1))
    g.barrier()
    assert calls == [1] and g.world == 1 and g.max(3.5) == 3.5


def test_rank_env_and_throughput():
    r = replicas.rank_env({"WORLD_SIZE": "4", "RANK": "3", "LOCAL_RANK": "1"})
    assert (r.world, r.rank, r.local) == (4, 3, 1)
    assert replicas.rank_env({}) == replicas.RankInfo(1, 0, 0)
    # 4 ranks x 32768 tokens x 10 steps in 2 s
    assert replicas.job_throughput(4, 32768, 10, 2.0) == pytest.approx(655360.0)
    with pytest.raises(ValueError):
        replicas.job_throughput(1, 1, 1, 0.0)
    assert replicas.token_seed(42, 0) == 42 and replicas.token_seed(42, 1) != 42
