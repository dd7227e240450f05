"""Data-parallel replicas of one model, one process per GPU, summed on the host.

The MegaTrain pages leave several GPUs as future work (author's blog, planned
projects).  Here every replica is a ``StreamedDecoder`` opened with
``replica_group=(name, rank, n)``: the n processes map one shared-memory
segment that holds the host tiles (W, G, M, V exist once), each streams the
weights from it and trains on its own batch, and the runtime's accumulator
adds each replica's gradient chunks into the shared G in rank order, the last
replica running Adam on every chunk as soon as its sum is complete, while the
backward goes on (paperlayer.ai summary §A.3, background accumulator over the
gradient slabs).  No collective runs on the data path, and no GPU reads
another's memory.

A group step is one ``train_step`` on every replica; it returns the loss of
the global batch (the mean over every replica's tokens) on each.  The result
equals ``train_step_micro`` of one model over the replicas' batches stacked in
rank order, bit for bit.

    name = replicas.group_name()      # made once, handed to every process
    m = replicas.open_replica(shape, name, rank, n)
    if rank == 0:
        m.load_weights(params)        # the tiles are shared: one replica writes
    m.barrier()
    loss = m.train_step(local_tokens)
"""
from __future__ import annotations

import os
import secrets

from . import StreamedDecoder


def group_name(prefix: str = "mt-group") -> str:
    """A shared-memory name for a new group (unique per call); pass it to
    every replica.  Replica 0 removes the name once all have attached."""
    return f"{prefix}-{os.getpid()}-{secrets.token_hex(6)}"


def shared_group_name(prefix: str = "mt-group", group=None) -> str:
    """``group_name`` made on rank 0 of an initialised torch.distributed
    process group and broadcast to its ranks (host-side agreement only)."""
    import torch.distributed as dist
    obj = [group_name(prefix) if dist.get_rank(group) == 0 else None]
    dist.broadcast_object_list(obj, src=0, group=group)
    return obj[0]


def open_replica(shape, name: str, rank: int, n: int, **kw) -> StreamedDecoder:
    """Replica ``rank`` of ``n`` of the model ``shape``; returns once all n
    replicas have attached to the group ``name``."""
    return StreamedDecoder.from_shape(shape, replica_group=(name, rank, n), **kw)


def replica_step(model: StreamedDecoder, tokens) -> float:
    """One group step on this replica's ``tokens``; the global batch's loss."""
    return model.train_step(tokens)
