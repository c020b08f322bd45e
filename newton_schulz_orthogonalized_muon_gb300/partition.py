"""Layer-wise ownership for running the Muon step on several GPUs.

Whole matrices are assigned to ranks ("Muon 优化器" MindSpeed feature doc,
§ZeRO 兼容适配): sort the parameters by size, then deal them out to the ranks
in ping-pong order (0, 1, ..., N-1, N-1, ..., 0, 0, 1, ...) so every rank
gets a similar number of elements.  Each rank runs the Muon step on the
matrices it owns (they are independent, so the step itself needs no
collective); afterwards every rank needs every updated parameter, which
``broadcast_owned`` provides: one broadcast per owner rank of the
parameters it owns, packed into one byte buffer (the page's all-gather of
unequal-length updated parameters).
"""
from __future__ import annotations


def layerwise_owners(sizes, world_size: int):
    """Owner rank of each item, by size-sorted ping-pong dealing."""
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    order = sorted(range(len(sizes)), key=lambda i: (-int(sizes[i]), i))
    owners = [0] * len(sizes)
    for k, idx in enumerate(order):
        lap, pos = divmod(k, world_size)
        owners[idx] = pos if lap % 2 == 0 else world_size - 1 - pos
    return owners


def owned(sizes, world_size: int, rank: int):
    """Indices owned by `rank`."""
    return [i for i, o in enumerate(layerwise_owners(sizes, world_size)) if o == rank]


def broadcast_owned(params, owners, group=None):
    """Give every rank the parameters updated by their owners, in place.

    ``params``: this rank's full list of contiguous tensors (all ranks hold
    the same shapes and dtypes in the same order); ``owners[i]``: the rank
    that updated params[i].  For each rank r that owns something, r packs
    the bytes of its parameters into one buffer, broadcasts it, and the
    other ranks unpack it into their copies; the owner's own tensors are not
    touched.  Works with any torch.distributed backend that broadcasts
    uint8 tensors (NCCL with CUDA tensors, gloo with CPU tensors)."""
    import torch
    import torch.distributed as dist
    if len(params) != len(owners):
        raise ValueError("one owner per parameter")
    world = dist.get_world_size(group)
    me = dist.get_rank(group)
    for r in range(world):
        idx = [i for i, o in enumerate(owners) if o == r]
        if not idx:
            continue
        for i in idx:
            if not params[i].is_contiguous():
                raise ValueError(f"params[{i}] must be contiguous")
        nbytes = [params[i].numel() * params[i].element_size() for i in idx]
        device = params[idx[0]].device
        if me == r:
            buf = torch.cat([params[i].reshape(-1).view(torch.uint8) for i in idx])
        else:
            buf = torch.empty(sum(nbytes), dtype=torch.uint8, device=device)
        src = dist.get_global_rank(group, r) if group is not None else r
        dist.broadcast(buf, src=src, group=group)
        if me != r:
            off = 0
            for i, nb in zip(idx, nbytes):
                params[i].reshape(-1).view(torch.uint8).copy_(buf[off:off + nb])
                off += nb
