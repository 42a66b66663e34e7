"""Host-side bookkeeping for running the hot path as independent replicas,
one process per GPU.

Quantizing a tensor and the scaled GEMM's forward and data-gradient products
split over tokens with no exchange, so N processes each run the whole step
on their own slice of tokens (here: their own seeded batch).  No data moves
between ranks.  The only cross-rank traffic is the timing reduction: the job
is as slow as its slowest rank, so the step time is the maximum over ranks,
and the job's throughput is the work of all ranks divided by that time.
"""
import os

__all__ = ["RankInfo", "rank_info", "replica_seed", "max_over_ranks", "job_throughput"]


class RankInfo:
    def __init__(self, world, rank, local):
        if world < 1 or not 0 <= rank < world or local < 0:
            raise ValueError(f"bad rank layout: world={world} rank={rank} local={local}")
        self.world, self.rank, self.local = world, rank, local

    @property
    def is_root(self):
        return self.rank == 0

    def __repr__(self):
        return f"RankInfo(world={self.world}, rank={self.rank}, local={self.local})"


def rank_info(env=None):
    """World size, global rank and local rank as torch.distributed.run exports
    them; a plain launch is a world of one."""
    env = os.environ if env is None else env
    return RankInfo(int(env.get("WORLD_SIZE", "1")), int(env.get("RANK", "0")),
                    int(env.get("LOCAL_RANK", "0")))


def replica_seed(base_seed, rank):
    """Each replica draws its own batch: the workload seed shifted by the rank,
    so rank 0 of any world sees exactly the single-process inputs."""
    return base_seed + rank


def max_over_ranks(value, dist=None, device=None):
    """Maximum of a per-rank float over the process group (the value itself in
    a world of one).  `device` is where the reduction tensor lives: the rank's
    GPU under NCCL, the CPU under gloo."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, work_per_rank_step, ms_per_step, scale=1e12):
    """Whole-job rate: every rank's work in one step over the slowest rank's
    step time, in units of `scale` per second (TFLOP/s by default)."""
    if ms_per_step <= 0:
        raise ValueError("step time must be positive")
    return world * work_per_rank_step / (ms_per_step * 1e-3) / scale
