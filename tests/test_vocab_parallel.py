"""The vocabulary-parallel merge on CPU ranks (gloo, world sizes 2 and 3).

Each rank holds a column block of every target and draft row.  The orchestration in
``vocab_parallel.verify_vocab_parallel`` (the all-gather of per-row statistics, the max
all-reduce of the logits at the draft tokens, the max all-reduce of the race keys) runs
unchanged; the four per-rank steps, which the GPU library computes, are played here by a
plain fp64 numpy backend with the oracle's random numbers.  The merged result must be the
oracle's verify of the whole rows, except on sequences the oracle flags as near-ties.
The CUDA steps themselves are compared with the oracle in tests/test_gpu_vocab_parallel.py.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _order_key(score: float, idx: int) -> int:
    """Signed key whose maximum is the highest float32 score, then the lowest index."""
    if idx < 0:
        return -(2 ** 63)
    u = int(np.float32(score).view(np.uint32))
    u = (~u & 0xFFFFFFFF) if u & 0x80000000 else (u | 0x80000000)
    key = (u << 32) | (~idx & 0xFFFFFFFF)
    return key - 2 ** 63


def _key_index(key: int) -> int:
    if key == -(2 ** 63):
        return -1
    return (~(key + 2 ** 63)) & 0xFFFFFFFF


class NumpyBackend:
    """fp64 stand-in for the library's four per-rank steps (natural-log statistics)."""

    def __init__(self, orc):
        self.orc = orc

    def partials(self, sh):
        import workloads
        t = workloads.as_f32(sh.target_np, sh.dtype).astype(np.float64)
        d = workloads.as_f32(sh.draft_np, sh.dtype).astype(np.float64)
        B, g1, Vs = t.shape
        g = g1 - 1
        stats = np.zeros((B, 2 * g + 1, 2))
        for b in range(B):
            for r in range(2 * g + 1):
                z = t[b, r] / sh.Tv[b] if r <= g else d[b, r - g - 1] / sh.Tdv[b]
                m = z.max()
                stats[b, r] = (m, np.exp(z - m).sum())
        gathered = np.full((B, g, 2), -np.inf)
        for b in range(B):
            for i in range(g):
                x = int(sh.tokens_np[b, i]) - sh.x_offset
                if 0 <= x < Vs:
                    gathered[b, i] = (t[b, i, x], d[b, i, x])
        return torch.from_numpy(stats), torch.from_numpy(gathered)

    def decide(self, stats_all, gathered, sh, seed):
        st = stats_all.numpy()
        ga = gathered.numpy()
        W, B, R, _ = st.shape
        g = (R - 1) // 2
        M = st[..., 0].max(axis=0)
        logZ = M + np.log((st[..., 1] * np.exp(st[..., 0] - M)).sum(axis=0))
        u = self.orc.accept_uniforms(seed, B, g)
        tokens = np.full((B, g + 1), -1, np.int32)
        n = np.zeros(B, np.int32)
        state = []
        for b in range(B):
            if np.any((sh.tokens_np[b] < 0) | (sh.tokens_np[b] >= sh.V)):
                n[b] = -1
                state.append((-1, 0.0, 0.0))
                continue
            j = g
            for i in range(g):
                lp = ga[b, i, 0] / sh.Tv[b] - logZ[b, i]
                lq = ga[b, i, 1] / sh.Tdv[b] - logZ[b, g + 1 + i]
                if not (np.isfinite(lp) and u[b, i] < np.exp(lp - lq)):
                    j = i
                    break
            tokens[b, :j] = sh.tokens_np[b, :j]
            n[b] = j
            state.append((j, logZ[b, j], logZ[b, g + 1 + j] if j < g else 0.0))
        return torch.from_numpy(tokens), torch.from_numpy(n), state

    def race(self, sh, state, seed):
        import workloads
        t = workloads.as_f32(sh.target_np, sh.dtype).astype(np.float64)
        d = workloads.as_f32(sh.draft_np, sh.dtype).astype(np.float64)
        B, g1, Vs = t.shape
        g = g1 - 1
        keys = np.full((B, 2), -(2 ** 63), np.int64)
        for b, (j, lzp, lzq) in enumerate(state):
            if j < 0:
                continue
            E = self.orc.race_exponentials(seed, b, j, Vs, sh.x_offset)
            p = np.exp(t[b, j] / sh.Tv[b] - lzp)
            w = np.maximum(0.0, p - np.exp(d[b, j] / sh.Tdv[b] - lzq)) if j < g else p
            for slot, weight in ((0, w), (1, p if j < g and not np.any(w > 0) else None)):
                if weight is None or not np.any(weight > 0):
                    continue
                with np.errstate(divide="ignore"):
                    score = np.where(weight > 0, np.log(weight) - np.log(E), -np.inf)
                x = int(np.argmax(score))  # lowest index among equal scores
                keys[b, slot] = _order_key(score[x], x + sh.x_offset)
        return torch.from_numpy(keys)

    def finish(self, keys, state, tokens):
        k = keys.numpy()
        for b, (j, _, _) in enumerate(state):
            if j < 0:
                continue
            y = _key_index(int(k[b, 0]))
            tokens[b, j] = y if y >= 0 else _key_index(int(k[b, 1]))
        return tokens


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, cfg, q):
    import oracle
    import workloads
    from speculative_decoding_verification_31_gb300.vocab_parallel import (VocabShard, verify_vocab_parallel,
                                                                           vocab_range)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, gamma, V, dtype, seed = cfg
        w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=V + gamma, sigma=0.8,
                              T=0.9, Td=0.45)
        lo, hi = vocab_range(V, world, rank)
        sh = VocabShard(None, None, None, lo, V, float(w.T[0]), float(w.Td[0]))
        sh.target_np = np.ascontiguousarray(w.target[:, :, lo:hi])
        sh.draft_np = np.ascontiguousarray(w.draft[:, :, lo:hi])
        sh.tokens_np, sh.dtype, sh.Tv, sh.Tdv = w.tokens, w.dtype, w.T, w.Td
        orc = oracle.get()
        tokens, n = verify_vocab_parallel(sh, seed, backend=NumpyBackend(orc))
        if rank == 0:
            r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
            near = oracle.FLAG_ACCEPT_NEAR_TIE | oracle.FLAG_RACE_NEAR_TIE | oracle.FLAG_RESIDUAL_EMPTY
            ok = (r.flags & near) == 0
            q.put((bool(ok.any()),
                   np.array_equal(n.numpy()[ok], r.n_accepted[ok]),
                   np.array_equal(tokens.numpy()[ok], r.tokens[ok])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,cfg", [(2, (5, 4, 3001, "bf16", 7)), (3, (4, 6, 2000, "f32", 3)),
                                       (2, (3, 0, 1500, "bf16", 1))])
def test_vocab_split_reproduces_the_whole_rows(world, cfg):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cfg, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    assert q.get(timeout=10) == (True, True, True)
