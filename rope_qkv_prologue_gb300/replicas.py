"""Running the prologue on several GPUs: replicas, no exchange on the data path.

Tokens are independent in every step of the prologue, so a job on N GPUs
gives each rank its own tokens (a contiguous shard of one batch, or a whole
per-GPU batch in weak scaling) and nothing crosses ranks in the forward. The
one cross-token result is the backward's RMSNorm weight gradient, a sum over
tokens: the sum of the ranks' gradients over their shards is the gradient
over all tokens, and in data-parallel training it rides the model's own
gradient all-reduce. These helpers hold that bookkeeping; they launch no
kernel.
"""

import torch
import torch.distributed as dist


def token_shard(T, rank, world):
    """The contiguous token range [start, stop) of `rank` out of `world` for a
    batch of T tokens (sizes differ by at most one)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    return rank * T // world, (rank + 1) * T // world


def sum_over_ranks(t):
    """All-reduce (sum) of a per-rank partial result in place, e.g. the weight
    gradients of a token shard; a no-op without a process group."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings over the process group (any
    backend); the values themselves without one."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_gbs(bytes_per_rank_step, world, ms_per_step):
    """Whole-job throughput: the bytes all ranks moved / the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9
