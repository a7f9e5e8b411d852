"""A stand-in rank for the launch test: bench.py's own rank set-up, timing
reduction and whole-job rate, with the codec step replaced by a fixed time
(no GPU).  Run by torch.distributed.run, never collected by pytest."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402

world, rank, local = bench.init_ranks()
ms = bench.dist_max(10.0 + 5.0 * rank)  # the slower rank decides the job time
if rank == 0:
    print(json.dumps({"n_gpus": world, "ms_per_step": ms, "value": bench.whole_job_gbs(world, 1e9, ms),
                      "local_ranks_seen": local}), flush=True)
if world > 1:
    dist.barrier()
    dist.destroy_process_group()
