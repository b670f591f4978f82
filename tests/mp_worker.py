"""One rank of the world-size-2 gloo test of bench.py's multi-process helpers
(run by tests/test_multiprocess.py; reads RANK / WORLD_SIZE / MASTER_* from
the environment like a torchrun rank)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def main():
    rank, world, local = bench.dist_setup(int(os.environ["WORLD_SIZE"]))
    bench.barrier(world)
    # each rank reports a different step time; the job time is the slowest
    t = bench.max_over_ranks(1.5 * (rank + 1), world)
    bench.barrier(world)
    import torch.distributed as dist
    dist.destroy_process_group()
    print(json.dumps({"rank": rank, "world": world, "max_ms": t}), flush=True)


if __name__ == "__main__":
    main()
