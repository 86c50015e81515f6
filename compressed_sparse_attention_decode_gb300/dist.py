"""Multi-GPU layout of the decode path: replicas, batch-sharded.

Sequences are independent (each has its own cache, indices and attention), so
N ranks (one process per GPU) split the batch and exchange nothing on the data
path.  The only collectives are the benchmark's timing barrier and a max over
ranks of the elapsed time.  Rank r of N with `per_rank` sequences owns global
sequence ids [r*per_rank, (r+1)*per_rank) of a workload of N*per_rank.
"""
import os

import torch


def env():
    """(rank, world, local_rank) from the launcher's environment (torchrun)"""
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def shard(per_rank, rank, world):
    """global sequence ids of this rank"""
    assert 0 <= rank < world and per_rank > 0
    return list(range(rank * per_rank, (rank + 1) * per_rank))


def reduce_max(x, device=None):
    """max of a float over all ranks (identity when not distributed)"""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()
