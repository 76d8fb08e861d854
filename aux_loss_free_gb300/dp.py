"""Data-parallel glue for the aux-loss-free balancing step.

Replicas route their own tokens; the method's only cross-replica exchange is the sum
of the per-expert loads before the bias update, so that every replica applies the
same update computed from the global load (relay article, architecture paragraph:
the bias moves by gamma times the sign of target minus load).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _lib


def allreduce_load(load: torch.Tensor, group=None) -> int:
    """Sum the int32 per-expert loads of all replicas in place; returns the replica count."""
    dist.all_reduce(load, op=dist.ReduceOp.SUM, group=group)
    return dist.get_world_size(group)


def dp_bias_update(load: torch.Tensor, bias: torch.Tensor, tokens_times_k_local: int, gamma: float,
                   group=None, stream=None) -> None:
    """All-reduce the loads, then apply the bias update with the global T*k (device tensors)."""
    world = allreduce_load(load, group)
    _lib.moe_bias_update(bias.numel(), world * tokens_times_k_local, load, gamma, bias, stream)
