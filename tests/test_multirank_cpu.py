"""The multi-rank path on CPU: two gloo ranks shard independent sequences
(each its own seeded batch, no data exchange) and agree on the slowest
rank's time, which sets the whole-job rate."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_gqa_pkv_gb300 import sharding
from paged_kv_gqa_pkv_gb300 import workloads as W


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = W.qwen3_b64_decode(sharding.shard_seed(rank), permute=False)
        my_time = 1.0 + 0.5 * rank
        slowest = sharding.max_over_ranks(my_time)
        lens = case.seq_lens.tolist()
        gathered = [None] * world
        dist.all_gather_object(gathered, lens)
        results[rank] = (slowest, gathered)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, join=True,
                       start_method="spawn")
    assert set(results.keys()) == {0, 1}
    for r in range(world):
        slowest, lens = results[r]
        assert slowest == pytest.approx(1.5)      # max over ranks, on every rank
        assert lens[0] != lens[1]                 # distinct shards
        assert lens[r] == W.qwen3_b64_decode(r).seq_lens.tolist()


def test_single_process_reduction_is_identity():
    assert sharding.max_over_ranks(3.25) == 3.25
    assert sharding.whole_job_rate(100.0, 4, 2.0) == 200.0
    assert sharding.shard_seed(3, 10) == 13
    with pytest.raises(ValueError):
        sharding.shard_seed(-1)
