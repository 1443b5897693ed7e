"""Process bodies for the multi-process tests (spawned children import this
module by name): the bench's rank logic over a gloo process group on CPU."""
import os


def bench_rank(rank, world, port, ms, queue):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(torch, world)
        m = bench.allreduce_max(torch, world, ms[rank])
        queue.put((rank, m, bench.whole_job_gbs(world, 1e9, m)))
        bench.barrier(torch, world)
    finally:
        dist.destroy_process_group()
