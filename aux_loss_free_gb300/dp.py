"""Data-parallel glue for the aux-loss-free balancing step.

Replicas route their own tokens; the method's only cross-replica exchange is the sum
of the per-expert loads before the bias update, so that every replica applies the
same update computed from the global load (relay article, architecture paragraph:
the bias moves by gamma times the sign of target minus load).  The target is the
global mean load, so it needs the global T*k: the sum of the summed loads, since every
token adds exactly k pairs.  That holds whatever the shards' sizes (a batch that does
not divide evenly, ragged batches), where world * (local T*k) would not.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _lib


def allreduce_load(load: torch.Tensor, group=None) -> int:
    """Sum the int32 per-expert loads of all replicas in place; returns the replica count."""
    dist.all_reduce(load, op=dist.ReduceOp.SUM, group=group)
    return dist.get_world_size(group)


def global_tokens_times_k(summed_load: torch.Tensor) -> int:
    """The global T*k from the loads summed over replicas (a host integer; reading a
    device tensor synchronises with it)."""
    return int(summed_load.sum(dtype=torch.int64).item())


def dp_bias_update(load: torch.Tensor, bias: torch.Tensor, gamma: float, group=None, stream=None) -> None:
    """All-reduce the loads, then apply the bias update with the global T*k (device
    tensors).  The update kernel takes the global T*k as the sum of the summed loads
    itself, so nothing is read back to the host."""
    allreduce_load(load, group)
    _lib.moe_bias_update(bias.numel(), _lib.MOE_TK_FROM_LOAD, load, gamma, bias, stream)
