"""Rows sharded by batch entry across ranks: the split and the sink gradient's exchange.

Rows are independent, so the forward and backward of a shard need nothing from the other
ranks.  The one cross-shard step is d_sink: every rank computes the chunk partials of its batch
entries (``fos_sink_grad_partials``), the partials are all-gathered in rank order and added left
to right (``fos_sink_grad_merge``), which gives the bits of ``fos_sink_grad`` on the whole batch
("[ROCm] Jax Add softmax sink (learnable off-by-one) support": d_sink is one sum per head over
batch and query rows).  A gather keeps the order fixed; an all-reduce would not.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from .binding import fos_sink_grad_merge


def batch_shards(batch: int, q_len: int, parts: int) -> list[tuple[int, int]]:
    """Split batch entries into ``parts`` contiguous ranges whose starts fall on the
    256-position chunk grid of each head (start * q_len a multiple of 256), as evenly as the
    grid allows; some ranges may be empty when the batch is small."""
    step = 256 // math.gcd(int(q_len), 256) if q_len > 0 else 1
    units = -(-int(batch) // step)  # aligned blocks of `step` entries
    bounds = [min(int(batch), (units * k // parts) * step) for k in range(parts + 1)]
    bounds[-1] = int(batch)
    return [(bounds[k], bounds[k + 1]) for k in range(parts)]


def sharded_sink_grad(local_partials: torch.Tensor, group=None) -> torch.Tensor:
    """d_sink [heads] (CPU) from this rank's chunk partials [heads, n_local]: all-gathered in
    rank order (ranks hold consecutive batch ranges) and merged left to right."""
    import torch.distributed as dist

    mine = local_partials.detach().to("cpu", torch.float32).contiguous().numpy()
    world = dist.get_world_size(group)
    parts = [None] * world
    dist.all_gather_object(parts, mine, group=group)
    merged = np.concatenate([np.asarray(p, dtype=np.float32).reshape(mine.shape[0], -1)
                             for p in parts], axis=1)
    return fos_sink_grad_merge(torch.from_numpy(np.ascontiguousarray(merged)))
