"""Multi-rank host logic on CPU: the layer-wise owner assignment used when
several GPUs share the Muon step, run as world_size-2 gloo ranks.

Checks: every matrix is owned by exactly one rank, the element counts are
balanced, and an all-gather of per-rank results (standing in for the updated
parameters) reassembles exactly what one rank computing everything produces.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    specs = wl.gpt2_small(2).muon
    sizes = [s.shape[0] * s.shape[1] for s in specs]
    mine = partition.owned(sizes, world, rank)
    # each rank "updates" the matrices it owns (a deterministic stand-in)
    flat = torch.cat([torch.full((sizes[i],), float(i + 1)) for i in mine]) if mine else torch.zeros(0)
    lens = torch.tensor([flat.numel()])
    all_lens = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(all_lens, lens)
    maxlen = int(max(x.item() for x in all_lens))
    padded = torch.zeros(maxlen)
    padded[:flat.numel()] = flat
    gathered = [torch.zeros(maxlen) for _ in range(world)]
    dist.all_gather(gathered, padded)
    if rank == 0:
        out = [None] * len(specs)
        for r in range(world):
            idx = partition.owned(sizes, world, r)
            off = 0
            for i in idx:
                out[i] = gathered[r][off:off + sizes[i]]
                off += sizes[i]
        full = torch.cat(out)
        expect = torch.cat([torch.full((sz,), float(i + 1)) for i, sz in enumerate(sizes)])
        torch.save({"ok": bool(torch.equal(full, expect))}, result_path)
    dist.destroy_process_group()


def test_two_gloo_ranks_reassemble(tmp_path):
    path = str(tmp_path / "res.pt")
    mp.spawn(_rank_main, args=(2, _free_port(), path), nprocs=2, join=True)
    assert torch.load(path)["ok"]
