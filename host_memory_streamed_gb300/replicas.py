"""Data-parallel replicas with a host-side gradient sum.

One process per GPU, each with its own ``StreamedDecoder`` and its own share of
the global batch (equal token counts).  A replica step is

  1. ``train_step_grads``: forward and backward of the local batch; every host
     tile's G section holds the BF16 gradient of the local mean loss;
  2. the gradients of all replicas are averaged on the host, tile by tile
     (``torch.distributed`` all-reduce of FP32 copies over the given process
     group, gloo on the host), and written back into each tile's G;
  3. ``apply_adam``: every replica applies the same Adam step to the same
     averaged gradient, so the replicas' weights stay identical.

The mean over replicas of the local mean losses' gradients is the gradient of
the mean loss over the global batch.  This is the host-side gradient sum that
the MegaTrain pages leave as future work for several GPUs (one GPU per
process; no device-side collective, no peer access between GPUs).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from ._lib import MT_PART_G


def allreduce_mean_bf16_(raw: torch.Tensor, group=None) -> None:
    """In place: the BF16 values held in the uint8 buffer ``raw`` become the
    mean over the group's ranks, summed in FP32 and rounded to BF16 once."""
    bf = raw.view(torch.bfloat16)
    acc = bf.to(torch.float32)
    dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    acc /= dist.get_world_size(group)
    bf.copy_(acc.to(torch.bfloat16))


def replica_step(model, tokens: torch.Tensor, group=None) -> float:
    """One data-parallel step of this replica on its local ``tokens``; returns
    the mean loss over all replicas' tokens (the same value on every rank)."""
    loss = model.train_step_grads(tokens)
    for i in range(model.n_tiles):
        g = model.get_tile(i, MT_PART_G)
        allreduce_mean_bf16_(g, group)
        model.load_tile(i, MT_PART_G, g)
    model.apply_adam()
    t = torch.tensor([loss], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t) / dist.get_world_size(group)
