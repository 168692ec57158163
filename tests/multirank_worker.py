"""Child process of the two-rank CPU test of the replica aggregation in bench.py (gloo)."""
import os
import sys


def run(rank, world, port, q):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    step_ms = [3.0, 5.0][rank]
    value, agg_ms = bench.aggregate_ranks(step_ms, 1000, world, "cpu")
    dist.barrier()
    q.put((rank, value, agg_ms))
    dist.destroy_process_group()
