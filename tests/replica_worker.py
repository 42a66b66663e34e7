"""A stand-in rank for the replica-launcher test: joins the gloo process
group from the environment bench.spawn_replicas sets, reports a per-rank
step time, and rank 0 prints one JSON line with the job's figures, as
bench.py's GPU arm does after its max-over-ranks reduction."""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch.distributed as dist  # noqa: E402

from fp8_hybrid_granularity_gb300 import replicas  # noqa: E402

ri = replicas.rank_info()
dist.init_process_group("gloo")
ms = replicas.max_over_ranks(10.0 + 5.0 * ri.rank, dist)
if ri.is_root:
    print(json.dumps({"n_gpus": ri.world, "ms_per_step": ms,
                      "value": replicas.job_throughput(ri.world, 1e12, ms),
                      "local_ranks_seen": dist.get_world_size(), "argv": sys.argv[1:],
                      "master": os.environ["MASTER_ADDR"]}), flush=True)
dist.destroy_process_group()
