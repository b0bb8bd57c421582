"""Sharded optimizer step across ranks: world-size-2 gloo process groups on CPU.

Each rank owns block-aligned slices of the flattened parameters and steps them
with the oracle (the GPU library is not needed for the host-side logic); the
gathered shards must equal the unsharded step bit for bit, including the 8-bit
path whose per-block absmax would be wrong if a shard split a block.  The
found-inf flags are combined with an all-reduce MAX, so one rank's non-finite
grad skips the step on every rank.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from adamw_optimizer_step_tensor_gb300 import shard

NUMELS = [1000, 1, 256, 4097, 0, 70001, 300]


def test_slices_cover_every_element_once_and_respect_blocks():
    for world in (1, 2, 3, 8):
        seen = [np.zeros(n, np.int32) for n in NUMELS]
        for r in range(world):
            for s in shard.shard_slices(NUMELS, world, r):
                assert s.start % 256 == 0 and 0 <= s.start < s.stop <= NUMELS[s.tensor]
                seen[s.tensor][s.start:s.stop] += 1
        assert all(np.all(x == 1) for x in seen)


def test_bounds_are_balanced():
    offs, total = shard.padded_offsets(NUMELS)
    sizes = [b - a for a, b in (shard.shard_bounds(total, 4, r) for r in range(4))]
    assert sum(sizes) == total and max(sizes) - min(sizes) <= 256


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, inject_rank, q):
    import torch
    import torch.distributed as dist

    from oracle import adamw as OA
    from oracle import q8 as OQ

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(5)          # same full inputs on every rank
        ps = [rng.normal(0, 0.02, n).astype(np.float32) for n in NUMELS]
        gs = [rng.normal(0, 1e-3, n).astype(np.float32) * 1024 for n in NUMELS]
        if inject_rank is not None:
            gs[5][12345] = np.inf                # owned by exactly one rank
        mine = shard.shard_slices(NUMELS, world, rank)
        # local non-finite check on the owned slices only, then MAX across ranks
        local = any(not np.all(np.isfinite(gs[s.tensor][s.start:s.stop])) for s in mine)
        found = torch.tensor([1.0 if local else 0.0])
        shard.allreduce_found_inf(found)
        out = {}
        if found.item() == 0.0:
            for s in mine:
                p = ps[s.tensor][s.start:s.stop].copy()
                g = gs[s.tensor][s.start:s.stop]
                x = OA.Tensor(p=p.copy(), g=g, m=np.zeros_like(p), v=np.zeros_like(p), wd=0.1)
                OA.step_f32([x], lr=0.01, beta1=0.9, beta2=0.999, eps=1e-8, t=1, grad_scale=1024.0)
                nb = OQ.n_blocks(p.size)
                cm, cv = np.zeros(p.size, np.uint8), np.zeros(p.size, np.uint8)
                am, av = np.zeros(nb, np.float32), np.zeros(nb, np.float32)
                p8 = p.copy()
                OQ.step_f32(p8, g, cm, cv, am, av, lr=0.01, beta1=0.9, beta2=0.999, eps=1e-8,
                            wd=0.1, t=1, grad_scale=1024.0)
                out[(s.tensor, s.start)] = (x.p, x.m, x.v, p8, cm, cv, am, av)
        gathered = [None] * world
        dist.all_gather_object(gathered, (local, found.item(), out))
        if rank == 0:
            q.put(gathered)
    finally:
        dist.destroy_process_group()


def _run(inject_rank):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, inject_rank, q)) for r in range(2)]
    for p in procs:
        p.start()
    result = q.get(timeout=240)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return result


def test_sharded_step_equals_unsharded_step():
    from oracle import adamw as OA
    from oracle import q8 as OQ

    gathered = _run(inject_rank=None)
    assert all(found == 0.0 for _, found, _ in gathered)
    pieces = {}
    for _, _, out in gathered:
        pieces.update(out)
    rng = np.random.default_rng(5)
    ps = [rng.normal(0, 0.02, n).astype(np.float32) for n in NUMELS]
    gs = [rng.normal(0, 1e-3, n).astype(np.float32) * 1024 for n in NUMELS]
    for i, (p, g) in enumerate(zip(ps, gs)):
        if p.size == 0:
            continue
        x = OA.Tensor(p=p.copy(), g=g, m=np.zeros_like(p), v=np.zeros_like(p), wd=0.1)
        OA.step_f32([x], lr=0.01, beta1=0.9, beta2=0.999, eps=1e-8, t=1, grad_scale=1024.0)
        nb = OQ.n_blocks(p.size)
        cm, cv = np.zeros(p.size, np.uint8), np.zeros(p.size, np.uint8)
        am, av = np.zeros(nb, np.float32), np.zeros(nb, np.float32)
        p8 = p.copy()
        OQ.step_f32(p8, g, cm, cv, am, av, lr=0.01, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1,
                    t=1, grad_scale=1024.0)
        parts = sorted((k[1], v) for k, v in pieces.items() if k[0] == i)
        cat = [np.concatenate([v[j] for _, v in parts]) for j in range(8)]
        assert np.array_equal(cat[0].view(np.uint32), x.p.view(np.uint32))
        assert np.array_equal(cat[1].view(np.uint32), x.m.view(np.uint32))
        assert np.array_equal(cat[2].view(np.uint32), x.v.view(np.uint32))
        assert np.array_equal(cat[3].view(np.uint32), p8.view(np.uint32))
        assert np.array_equal(cat[4], cm) and np.array_equal(cat[5], cv)
        assert np.array_equal(cat[6].view(np.uint32), am.view(np.uint32))
        assert np.array_equal(cat[7].view(np.uint32), av.view(np.uint32))


def test_one_ranks_nonfinite_grad_skips_every_rank():
    gathered = _run(inject_rank=1)
    local = [loc for loc, _, _ in gathered]
    assert sum(local) == 1                        # only the owning rank saw it
    assert all(found == 1.0 and out == {} for _, found, out in gathered)
