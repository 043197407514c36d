"""Worker of the multi-rank bench test (a module of its own so that spawned
processes can import it)."""
import os


def max_over_ranks_worker(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.0 + 0.5 * rank, dist, "cpu")
        dist.barrier()
        queue.put((rank, slowest))
    finally:
        dist.destroy_process_group()
