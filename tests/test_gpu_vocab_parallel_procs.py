"""The vocabulary split across processes on the CUDA library (marked gpu).

Two processes, each its own rank of a gloo group and its own CUDA context on this GPU, hold
one column block each of every target and draft row and run ``verify_vocab_parallel`` with
``LibraryBackend``: the four library steps on the device, the all-gather of the statistics
and the two max all-reduces through the gloo group.  No kernel of one rank waits for
another rank's: the ranks meet only in the host-side collectives.  Both ranks must return
the same tokens, and those must be the oracle's verify of the whole rows, except on
sequences the oracle flags as near-ties.  ("How speculative decoding makes LLMs go brrr",
module 3; the race keyed by the global token index.)
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads

pytestmark = pytest.mark.gpu

CASES = [
    dict(B=6, gamma=5, V=20011, dtype="bf16", seed=41, sigma=0.7, T=0.9, Td=0.45),
    dict(B=3, gamma=0, V=9000, dtype="f32", seed=42, sigma=0.7, T=1.1, Td=1.1),
    dict(B=4, gamma=8, V=128256, dtype="bf16", seed=43, sigma=1.0, T=0.7, Td=0.35),
]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    import torch.distributed as dist
    import speculative_decoding_verification_31_gb300 as sv
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        for k, case in enumerate(CASES):
            w = workloads.generic(**case)
            lo, hi = sv.vocab_range(w.V, world, rank)

            def to_dev(a):
                a = np.ascontiguousarray(a[:, :, lo:hi])
                if w.dtype == "bf16":
                    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
                return torch.from_numpy(a).to(dev)

            tok = torch.from_numpy(w.tokens).to(dev)
            Tq = torch.from_numpy(w.T.astype(np.float32)).to(dev)
            Tdq = torch.from_numpy(w.Td.astype(np.float32)).to(dev)
            shard = sv.VocabShard(to_dev(w.target), to_dev(w.draft), tok, lo, w.V,
                                  float(w.T[0]), float(w.Td[0]), T_per_seq=Tq, Td_per_seq=Tdq)
            for seed in range(3):
                t, n = sv.verify_vocab_parallel(shard, seed, backend=sv.LibraryBackend())
                torch.cuda.synchronize()
                np.savez(os.path.join(out_dir, f"r{rank}_c{k}_s{seed}.npz"),
                         tokens=t.cpu().numpy(), n=n.cpu().numpy())
            assert sv.spec_verify_check() == sv.SPEC_OK
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_on_the_library_match_the_oracle(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    world = 2
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    orc = oracle.get()
    near = oracle.FLAG_ACCEPT_NEAR_TIE | oracle.FLAG_RACE_NEAR_TIE | oracle.FLAG_RESIDUAL_EMPTY
    for k, case in enumerate(CASES):
        w = workloads.generic(**case)
        for seed in range(3):
            res = [np.load(os.path.join(tmp_path, f"r{r}_c{k}_s{seed}.npz")) for r in range(world)]
            for r in range(1, world):
                np.testing.assert_array_equal(res[r]["tokens"], res[0]["tokens"])
                np.testing.assert_array_equal(res[r]["n"], res[0]["n"])
            ref = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
            for b in range(w.B):
                j = int(res[0]["n"][b])
                assert 0 <= j <= w.gamma
                if ref.flags[b] & near:
                    continue
                assert j == ref.n_accepted[b], (k, seed, b)
                np.testing.assert_array_equal(res[0]["tokens"][b], ref.tokens[b])
