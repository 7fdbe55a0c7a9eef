"""Host logic for running the step on several GPUs, one process per GPU.

The sequences of a batch are independent at every stage of the step (each
draws its own tree, attends to its own KV prefix and walks its own target
rows), so several GPUs share a job by splitting the batch into contiguous
ranges of sequences, one per rank, with no exchange on the data path.  The
only collective is the max-over-ranks of a measured time.
"""


def shard(B, rank, world):
    """Contiguous range [b0, b1) of the B sequences that `rank` of `world`
    processes; ranges of consecutive ranks differ in size by at most one and
    together cover 0..B-1 exactly once."""
    if world < 1 or not 0 <= rank < world or B < 0:
        raise ValueError(f"bad shard request B={B} rank={rank} world={world}")
    q, r = divmod(B, world)
    b0 = rank * q + min(rank, r)
    return b0, b0 + q + (1 if rank < r else 0)


def max_over_ranks(value, device="cpu"):
    """Largest `value` over all ranks of the default process group (the
    value itself when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
