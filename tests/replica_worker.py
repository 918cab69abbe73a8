"""One rank of the replica path, run under torch.distributed.run with the gloo backend.

Each rank reports a different step time (2 + rank ms) and one unit per step; rank 0 alone
prints the aggregate as one JSON line, the way the benchmark does.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    world, rank, local = bench.init_replicas(dist, "gloo")
    dist.barrier()
    ms, units, value = bench.aggregate_replicas(torch, dist, 2.0 + rank, 1)
    dist.barrier()
    if rank == 0:
        print(json.dumps({"world": world, "ms": ms, "units": units, "value": value,
                          "local": local}))
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
