"""The data-parallel (N > 1) path of bench.py on the CPU: two gloo ranks, each
with its own shard of a workload, reduce their step times to the slowest
rank's, and the job value counts the keys of every rank.  No GPU, no
collective on the data path (the path shards by batch)."""
import json
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from sparse_attention_indexer_mxfp4_gb300 import synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = bench._case(1, shard=rank)
        ms = 1.0 + 0.5 * rank  # the slower rank must set the job time
        reduced = bench.max_over_ranks([ms, 10.0 * (world - rank)], "cpu", world)
        res = {"rank": rank, "reduced": reduced, "keys": int(case.keys_scored),
               "q_sum": int(np.asarray(case.q, dtype=np.int64).sum()),
               "ke": [int(v) for v in case.ke]}
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_and_count_every_rank(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["reduced"] == [1.5, 20.0]  # element-wise max over ranks
    # each rank runs its own shard: same shape and lengths, different values
    assert res[0]["keys"] == res[1]["keys"] and res[0]["ke"] == res[1]["ke"]
    assert res[0]["q_sum"] != res[1]["q_sum"]
    value = bench.job_value(world, res[0]["keys"], res[0]["reduced"][0])
    assert value == pytest.approx(world * res[0]["keys"] / 1.5e-3 / 1e9)


def test_shard_zero_is_the_workload_itself():
    a, b = synth.config1(), synth.config1(0)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.k, b.k)
    c = synth.config1(1)
    assert not np.array_equal(a.q, c.q) and np.array_equal(a.ke, c.ke)
