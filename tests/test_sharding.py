"""Sharding a batch over ranks (CPU, gloo, world size 2).

Each rank verifies its contiguous range of sequences with the global index of its first
sequence as the random-number base, then the ranks all-gather tokens and accepted counts;
the result must equal one verify over the whole batch.  The oracle stands in for the GPU
library here (the test runs without a GPU); the CUDA path's own seq_index_base is checked
against a single call in the GPU tests.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verification_31_gb300.sharding import shard_range


def test_shard_range_partitions():
    for total in (0, 1, 7, 64, 255, 256):
        for world in (1, 2, 3, 8):
            ranges = [shard_range(total, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == total
            for (a, b), (c, d) in zip(ranges, ranges[1:]):
                assert b == c
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_range(10, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import oracle
    import workloads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.generic(B=7, gamma=5, V=3000, dtype="bf16", seed=3, sigma=0.9, T=0.9,
                              Td=0.4)
        lo, hi = shard_range(w.B, world, rank)
        sub = w.subset(range(lo, hi))
        r = oracle.get().verify(sub.target, sub.draft, sub.tokens, sub.T, sub.Td, seed=11,
                                b_base=lo)
        # pad to the largest shard for all_gather
        width = -(-w.B // world)
        tok = torch.full((width, w.gamma + 1), -9, dtype=torch.int32)
        n = torch.full((width,), -9, dtype=torch.int32)
        tok[:hi - lo] = torch.from_numpy(r.tokens)
        n[:hi - lo] = torch.from_numpy(r.n_accepted)
        toks = [torch.empty_like(tok) for _ in range(world)]
        ns = [torch.empty_like(n) for _ in range(world)]
        dist.all_gather(toks, tok)
        dist.all_gather(ns, n)
        if rank == 0:
            parts_t, parts_n = [], []
            for rr in range(world):
                a, b = shard_range(w.B, world, rr)
                parts_t.append(toks[rr][:b - a].numpy())
                parts_n.append(ns[rr][:b - a].numpy())
            whole = oracle.get().verify(w.target, w.draft, w.tokens, w.T, w.Td, seed=11)
            q.put((np.array_equal(np.concatenate(parts_t), whole.tokens),
                   np.array_equal(np.concatenate(parts_n), whole.n_accepted)))
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_reproduce_the_whole_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    assert q.get(timeout=10) == (True, True)
