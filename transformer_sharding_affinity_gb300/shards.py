"""Token-sharded calibration over several processes (one GPU each).

Every affinity entry is a token mean times a per-neuron factor ("Affinity-Aware
Sharding for Delayed Tensor Parallelism", §3 "Affinity scores"), so the
calibration tokens split into disjoint shards with no exchange while the
scores are computed: each rank runs the whole pass on its own shard.  The one
exchange step merges the shards' results, a token-weighted mean done in fixed
rank order by ``affinity_combine_shards`` so every rank gets identical bits.

PyTorch supplies the process group (``gloo`` for host tensors, ``nccl`` for
device tensors); the merge arithmetic is the library's.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

from . import binding as B


def token_range(T: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous [start, stop) of the T calibration tokens owned by `rank`:
    T // world each, the first T % world ranks one more."""
    if world < 1 or not 0 <= rank < world or T < 0:
        raise ValueError("need 0 <= rank < world and T >= 0")
    base, extra = divmod(T, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def allgather_combine(S_local, T_local: int, group=None) -> np.ndarray:
    """Merge this rank's S (a torch tensor, host or device, any shape) with every
    other rank's: all-gather the shards' values and token counts, then the
    token-weighted mean in rank order.  Returns the merged fp32 array on the
    host, identical on every rank."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    on_device = dist.get_backend(group) == "nccl"
    dev = S_local.device if on_device else torch.device("cpu")
    S = S_local.detach().to(dev, torch.float32).contiguous()
    T = torch.tensor([int(T_local)], dtype=torch.int64, device=dev)
    S_all = [torch.empty_like(S) for _ in range(world)]
    T_all = [torch.empty_like(T) for _ in range(world)]
    dist.all_gather(T_all, T, group=group)
    dist.all_gather(S_all, S, group=group)
    S_host = [s.cpu().numpy() for s in S_all]
    T_host = [int(t.item()) for t in T_all]
    return B.combine_shards(S_host, T_host)
