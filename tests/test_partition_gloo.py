"""Multi-rank host logic on CPU: the layer-wise owner assignment used when
several GPUs share the Muon step, run as world_size-2 gloo ranks.

Checks: every matrix is owned by exactly one rank and the element counts
are balanced; and, with 2 and 3 gloo ranks, each rank running the fp64
oracle's Muon step on the matrices it owns, then handing the updated
parameters to every rank with partition.broadcast_owned, ends with exactly
(bit for bit) the parameters one process stepping every matrix produces, on
every rank.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from newton_schulz_orthogonalized_muon_gb300 import partition, workloads as wl


def test_owners_cover_and_balance():
    specs = wl.llama3_8b(32).muon
    sizes = [s.shape[0] * s.shape[1] for s in specs]
    for world in (1, 2, 3, 4, 8):
        owners = partition.layerwise_owners(sizes, world)
        assert sorted(set(owners)) == list(range(min(world, len(sizes))))
        load = np.bincount(owners, weights=sizes, minlength=world)
        assert load.max() / load.mean() < 1.05
        got = sorted(i for r in range(world) for i in partition.owned(sizes, world, r))
        assert got == list(range(len(sizes)))


def test_ping_pong_order():
    owners = partition.layerwise_owners([10, 9, 8, 7, 6, 5, 4, 3], 3)
    # sorted by size, dealt 0 1 2 | 2 1 0 | 0 1
    assert owners == [0, 1, 2, 2, 1, 0, 0, 1]
    with pytest.raises(ValueError):
        partition.layerwise_owners([1], 0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, result_path):
    """One gloo rank: run the fp64 oracle's Muon step on the matrices this
    rank owns (a small GPT-2-like set with a Muon-Split matrix), hand the
    updated parameters to every rank with broadcast_owned, and (rank 0)
    compare the reassembled set with one process stepping every matrix."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    specs = _specs()
    sizes = [s.shape[0] * s.shape[1] for s in specs]
    owners = partition.layerwise_owners(sizes, world)
    params, grads = _inputs(specs)
    for i in partition.owned(sizes, world, rank):
        w_new, _ = oracle.muon_step(params[i].numpy(), grads[i], np.zeros(specs[i].shape), lr=0.02, wd=0.1,
                                    split_heads=specs[i].split_heads)
        params[i].copy_(torch.from_numpy(w_new))
    partition.broadcast_owned(params, owners)
    # every rank ends with the same parameters: compare each rank's bytes with rank 0's
    flat = torch.cat([p.reshape(-1) for p in params])
    copies = [torch.empty_like(flat) for _ in range(world)]
    dist.all_gather(copies, flat)
    if rank == 0:
        start, _ = _inputs(specs)
        single = [torch.from_numpy(oracle.muon_step(start[i].numpy(), grads[i], np.zeros(s.shape), lr=0.02, wd=0.1,
                                                    split_heads=s.split_heads)[0]) for i, s in enumerate(specs)]
        torch.save({"ok": all(torch.equal(a, b) for a, b in zip(params, single)),
                    "same_on_all_ranks": all(torch.equal(c, copies[0]) for c in copies),
                    "owned_by": [len(partition.owned(sizes, world, r)) for r in range(world)]}, result_path)
    dist.destroy_process_group()


def _specs():
    return wl.gpt2_small(layers=1, d=64).muon + [wl.ParamSpec("attn.qkv", (96, 64), split_heads=3),
                                                 wl.ParamSpec("odd", (40, 72))]


def _inputs(specs):
    params = [torch.from_numpy(wl.weight(10 + i, s.shape).astype(np.float64)) for i, s in enumerate(specs)]
    grads = [wl.lowrank_grad(20 + i, s.shape[0], s.shape[1], 8).astype(np.float64) for i, s in enumerate(specs)]
    return params, grads


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_oracle_steps_reassemble_to_the_single_rank_step(tmp_path, world):
    path = str(tmp_path / "res.pt")
    mp.spawn(_rank_main, args=(world, _free_port(), path), nprocs=world, join=True)
    res = torch.load(path)
    assert res["ok"] and res["same_on_all_ranks"]
    assert all(n > 0 for n in res["owned_by"])       # every rank did part of the step
