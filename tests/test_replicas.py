"""The N>1 path (independent replicas, max-over-ranks timing) on CPU with two
gloo ranks.  No GPU and no kernel: only the host logic bench.py runs under
torchrun is exercised here."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from fp8_hybrid_granularity_gb300 import replicas, workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ri = replicas.rank_info()
        ms = 10.0 + 5.0 * ri.rank                  # rank 1 is the slow one
        ms_max = replicas.max_over_ranks(ms, dist)
        # each replica draws its own batch from the shifted seed
        x = workloads.make_tensor("act", 8, 256, replicas.replica_seed(2, ri.rank), "X")
        fp = workloads.bf16_bits(x).astype("int64").sum()
        t = torch.tensor([float(fp)], dtype=torch.float64)
        gathered = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(gathered, t)
        out[rank] = (ri.world, ri.rank, ri.is_root, ms_max, [float(g.item()) for g in gathered])
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_replicas():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r, (w, rank, root, ms_max, fps) in res.items():
        assert (w, rank, root) == (2, r, r == 0)
        assert ms_max == 15.0                       # the slowest rank sets the step time
        assert fps[0] != fps[1]                     # replicas do not share inputs
    # rank 0 of a multi-rank job sees exactly the single-process inputs
    x0 = workloads.make_tensor("act", 8, 256, 2, "X")
    assert res[0][4][0] == float(workloads.bf16_bits(x0).astype("int64").sum())


def test_world_of_one_needs_no_process_group():
    assert replicas.max_over_ranks(3.5) == 3.5
    ri = replicas.rank_info({})
    assert (ri.world, ri.rank, ri.local, ri.is_root) == (1, 0, 0, True)


def test_job_throughput_counts_every_rank():
    # 2 ranks x 1 TFLOP per step in 10 ms -> 200 TFLOP/s for the job
    assert replicas.job_throughput(2, 1e12, 10.0) == pytest.approx(200.0)
    with pytest.raises(ValueError):
        replicas.job_throughput(1, 1.0, 0.0)


def test_bad_rank_layout_rejected():
    with pytest.raises(ValueError):
        replicas.rank_info({"WORLD_SIZE": "2", "RANK": "2"})
