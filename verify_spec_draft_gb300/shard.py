"""A batch split across processes, one per GPU.

Requests (draft, verify) and branches (E2E-TV) are independent of one another, so each
rank takes a contiguous shard and the data path needs no exchange.  The one quantity of
the whole batch is the E2E-TV loss, L = 1 - (mean survival over all branches and
positions): every rank's spec_e2etv_shard returns its part of that mean, and one scalar
all-reduce (sum) completes it.  Timings are combined by the slowest rank.
"""


def shard_range(n, rank, world):
    """(start, count) of rank's contiguous shard of n units: the first n % world ranks
    take one unit more than the others."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must lie in [0, world)")
    base, extra = divmod(int(n), int(world))
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def e2etv_loss_from_shares(msum, group=None):
    """The loss of the whole batch from this rank's share ``msum`` (a 1-element float
    tensor on the process group's device): sums the shares over the group in place and
    returns 1 - sum as a new tensor."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(msum, op=dist.ReduceOp.SUM, group=group)
    return 1.0 - msum


def max_over_ranks(value, device, group=None):
    """The largest of a per-rank float over the group (the slowest rank's time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def e2etv_rank(target, draft, n_local, Wb, total_branches, ws=None, out=None, group=None, stream=None):
    """spec_e2etv_shard on this rank's rows, then the loss of the whole batch by one
    all-reduce.  Returns the shard's outputs with ``loss`` added."""
    from . import e2etv_shard
    out = e2etv_shard(target, draft, n_local, Wb, total_branches, ws=ws, out=out, stream=stream)
    out["loss"] = e2etv_loss_from_shares(out["msum"].clone(), group)
    return out
