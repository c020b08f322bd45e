"""Layer-wise owner assignment for running the Muon step on several GPUs.

Whole matrices are assigned to ranks ("Muon 优化器" MindSpeed feature doc,
§ZeRO 兼容适配): sort the parameters by size, then deal them out to the ranks
in ping-pong order (0, 1, ..., N-1, N-1, ..., 0, 0, 1, ...) so every rank
gets a similar number of elements.  Each rank then runs the Muon step on the
matrices it owns; the matrices are independent, so no collective is needed
inside the step.  (The page's design all-gathers the updated parameters
afterwards; that exchange belongs to the data-parallel training loop.)
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
