"""The multi-rank host logic on CPU: two gloo ranks (world_size 2).

Checks that the head and q-block shards cover every unit exactly once with
balanced work, that max_over_ranks returns the slowest rank's time on every
rank, and that sharded per-head attention (the oracle stands in for a GPU
rank's kernels here) reassembles into the single-process result.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from exact_attention_59_gb300 import dist as D


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as tdist
    import oracle.attention as OR
    from exact_attention_59_gb300 import inputs as IN
    r, ws = D.init("gloo")
    assert (r, ws) == (rank, world)
    D.barrier()
    slowest = D.max_over_ranks(10.0 + rank)
    # per-head sharded attention, gathered on every rank
    c = IN.make_case(2, 3, 8, 8, 4, "f32", with_key_mask=True)
    heads = [(b, h) for b in range(2) for h in range(3)]
    mine = [heads[i] for i in D.shard_heads(len(heads), ws, r)]
    q, k, v = (c[n].double().numpy() for n in ("q", "k", "v"))
    o, _ = OR.attn_fwd(q, k, v, key_mask=c["key_mask"].numpy(), score_mod="alibi", heads=mine)
    part = torch.from_numpy(np.nan_to_num(o, nan=0.0))
    tdist.all_reduce(part)          # shards are disjoint: the sum reassembles them
    out[rank] = (slowest, part.numpy(), mine)
    tdist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()   # no fork of this (threaded) process
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    import oracle.attention as OR
    from exact_attention_59_gb300 import inputs as IN
    c = IN.make_case(2, 3, 8, 8, 4, "f32", with_key_mask=True)
    q, k, v = (c[n].double().numpy() for n in ("q", "k", "v"))
    ref, _ = OR.attn_fwd(q, k, v, key_mask=c["key_mask"].numpy(), score_mod="alibi")
    covered = []
    for r in range(world):
        slowest, gathered, mine = out[r]
        assert slowest == 11.0
        np.testing.assert_allclose(gathered, ref, rtol=1e-12, atol=1e-14)
        covered += list(mine)
    assert sorted(covered) == sorted((b, h) for b in range(2) for h in range(3))


@pytest.mark.parametrize("n,world", [(64, 8), (2, 8), (7, 3), (1, 1), (5, 2)])
def test_shard_heads_cover_once(n, world):
    got = [i for r in range(world) for i in D.shard_heads(n, world, r)]
    assert got == list(range(n))
    sizes = [len(D.shard_heads(n, world, r)) for r in range(world)]
    assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("nqb,world", [(1024, 8), (16, 4), (16, 3), (5, 2)])
def test_shard_qblocks_balance_causal_work(nqb, world):
    shards = [D.shard_qblocks(nqb, world, r) for r in range(world)]
    assert sorted(q for s in shards for q in s) == list(range(nqb))
    work = [sum(qb + 1 for qb in s) for s in shards]          # kv tiles per rank (causal)
    assert max(work) - min(work) <= nqb                      # within one longest row
    assert all(s == sorted(s, reverse=True) for s in shards)  # longest first
