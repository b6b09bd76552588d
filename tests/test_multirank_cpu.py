"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

Under weak scaling each rank draws its own shard of the global batch (no
exchange of data), the oracle runs on each shard independently, and the
job's time is the maximum over ranks."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from log_linear_attention_chunkwise_gb300 import workloads as W


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = W.small_fwd_config(1, 2, 64, 16, 16, 16, torch.float32, seed=5)
        shard = bench.rank_shard(cfg, rank, world)
        x = W.make_fwd_inputs(shard)
        out = oracle.fenwick(x["q"], x["k"], x["v"], x["g"], x["lam"])
        t = bench.max_over_ranks(1.5 + rank, torch.device("cpu"))
        np.save(os.path.join(result_dir, f"out{rank}.npy"), out)
        np.save(os.path.join(result_dir, f"q{rank}.npy"), x["q"].numpy())
        np.save(os.path.join(result_dir, f"t{rank}.npy"), np.array([t]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_take_the_max(tmp_path):
    world = 2
    mp.start_processes(worker, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    q0, q1 = np.load(tmp_path / "q0.npy"), np.load(tmp_path / "q1.npy")
    assert not np.allclose(q0, q1)  # disjoint units, not replicas
    for r in range(world):
        assert float(np.load(tmp_path / f"t{r}.npy")[0]) == 2.5
        # each rank's result is what one process computes for that shard alone
        cfg = bench.rank_shard(W.small_fwd_config(1, 2, 64, 16, 16, 16, torch.float32, seed=5), r, world)
        x = W.make_fwd_inputs(cfg)
        ref = oracle.fenwick(x["q"], x["k"], x["v"], x["g"], x["lam"])
        np.testing.assert_array_equal(np.load(tmp_path / f"out{r}.npy"), ref)


def test_single_rank_is_unchanged():
    cfg = W.FWD_CONFIGS["fp32_T256"]
    assert bench.rank_shard(cfg, 0, 1) == cfg
    assert bench.max_over_ranks(3.25, torch.device("cpu")) == 3.25
