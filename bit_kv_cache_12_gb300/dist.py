"""Replica plumbing for running the decode on several GPUs of one node.

The decode shards without any exchange: sequences are independent, so each
rank owns a contiguous slice of the batch (or, for the benchmark, a full
replica of the workload) and no collective touches the data path.  The only
collectives are host-side: a barrier around timed regions and the maximum of
the per-rank step times.  Everything here works on any torch.distributed
backend (NCCL on GPUs, gloo on CPUs for tests)."""

import os


def rank_world():
    """(rank, world_size, local_rank) from the launcher's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend):
    """Join the process group when launched with more than one rank.
    Returns (rank, world_size, local_rank)."""
    rank, world, local = rank_world()
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if not dist.is_initialized():
            dist.init_process_group(backend)
    return rank, world, local


def shutdown():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of a list of floats over all ranks."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def shard(n, rank, world):
    """Contiguous [begin, end) slice of n independent units owned by a rank;
    the slices of all ranks partition [0, n) and differ in size by at most 1."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("rank out of range")
    base, extra = divmod(n, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)
