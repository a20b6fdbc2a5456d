"""Worker of the two-rank CPU test of bench.py's cross-rank timing (gloo)."""
import os


def max_over_ranks_worker(rank, world, port, out_dir):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (10 + r) ms for the steps and (20 - r) ms end to end
        got = bench.max_over_ranks([10.0 + rank, 20.0 - rank], world)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(" ".join(repr(v) for v in got))
    finally:
        dist.destroy_process_group()
