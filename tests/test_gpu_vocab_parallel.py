"""The vocabulary-parallel steps on the GPU (marked gpu): W ranks emulated one after another
on one device (each rank's steps are separate calls on its own column block; the two
collectives are a max and a stack of the ranks' outputs), compared with the oracle's verify
of the whole rows and with the one-GPU verify, except on near-tie sequences."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import NEAR_TIE, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_31_gb300 as m
    m.load_library()
    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def emulate(sv, w, world, seed, tokens=None, per_seq=False):
    dev = torch.device("cuda:0")
    tok = torch.from_numpy(np.ascontiguousarray(w.tokens if tokens is None else tokens)).to(dev)
    Tq = torch.from_numpy(w.T.astype(np.float32)).to(dev) if per_seq else None
    Tdq = torch.from_numpy(w.Td.astype(np.float32)).to(dev) if per_seq else None
    shards = []
    for r in range(world):
        lo, hi = sv.vocab_range(w.V, world, r)
        t = to_device(np.ascontiguousarray(w.target[:, :, lo:hi]), w.dtype, dev)
        d = to_device(np.ascontiguousarray(w.draft[:, :, lo:hi]), w.dtype, dev)
        shards.append(sv.VocabShard(t, d, tok, lo, w.V, float(w.T[0]), float(w.Td[0]), Tq, Tdq))
    be = sv.LibraryBackend()
    parts = [be.partials(sh) for sh in shards]
    stats_all = torch.stack([p[0] for p in parts]).contiguous()
    gathered = parts[0][1]
    for p in parts[1:]:
        gathered = torch.maximum(gathered, p[1])
    tokens_out, n, state = be.decide(stats_all, gathered.contiguous(), shards[0], seed)
    keys = be.race(shards[0], state, seed)
    for sh in shards[1:]:
        keys = torch.maximum(keys, be.race(sh, state, seed))
    be.finish(keys, state, tokens_out)
    torch.cuda.synchronize()
    return tokens_out.cpu().numpy(), n.cpu().numpy()


CASES = [(5, 4, 3001, "bf16", 2), (4, 6, 2000, "f32", 3), (3, 0, 1500, "bf16", 2),
         (3, 40, 20000, "bf16", 4), (6, 3, 40001, "f32", 2), (2, 5, 152064, "bf16", 8),
         # each shard with more row pieces than the streaming grid has warps (its claiming launch)
         (32, 8, 128256, "bf16", 2)]


@pytest.mark.parametrize("B,gamma,V,dtype,world", CASES)
def test_vocab_split_matches_oracle_and_one_gpu(sv, orc, B, gamma, V, dtype, world):
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=V + world, sigma=0.8, T=0.9,
                          Td=0.45)
    dev = torch.device("cuda:0")
    t_full, d_full = to_device(w.target, w.dtype, dev), to_device(w.draft, w.dtype, dev)
    tok = torch.from_numpy(w.tokens).to(dev)
    for seed in (0, 3):
        vt, vn = emulate(sv, w, world, seed)
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        ok = (r.flags & NEAR_TIE) == 0
        assert ok.any()
        np.testing.assert_array_equal(vn[ok], r.n_accepted[ok])
        np.testing.assert_array_equal(vt[ok], r.tokens[ok])
        gt, gn, _ = sv.spec_verify_ex(t_full, d_full, tok, float(w.T[0]), float(w.Td[0]), seed)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(vt[ok], gt.cpu().numpy()[ok])
        np.testing.assert_array_equal(vn[ok], gn.cpu().numpy()[ok])
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_vocab_split_per_sequence_temperatures(sv, orc):
    w = workloads.config(3, B=6)
    vt, vn = emulate(sv, w, 4, 11, per_seq=True)
    r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, 11)
    ok = (r.flags & NEAR_TIE) == 0
    np.testing.assert_array_equal(vn[ok], r.n_accepted[ok])
    np.testing.assert_array_equal(vt[ok], r.tokens[ok])
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_vocab_split_bad_tokens(sv, orc):
    w = workloads.generic(B=4, gamma=5, V=3000, dtype="bf16", seed=12)
    tok = w.tokens.copy()
    tok[1, 2] = w.V
    tok[2, 0] = -5
    vt, vn = emulate(sv, w, 2, 0, tokens=tok)
    assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
    assert vn[1] == -1 and vn[2] == -1
    assert np.all(vt[1] == -1) and np.all(vt[2] == -1)
    r = orc.verify(w.target, w.draft, tok, w.T, w.Td, 0)
    for b in (0, 3):
        if not (r.flags[b] & NEAR_TIE):
            assert vn[b] == r.n_accepted[b]
            np.testing.assert_array_equal(vt[b], r.tokens[b])


def test_one_rank_orchestration_on_the_gpu(sv, orc):
    """verify_vocab_parallel without a process group: one rank holding every column."""
    w = workloads.generic(B=3, gamma=4, V=5003, dtype="bf16", seed=5, sigma=0.8)
    dev = torch.device("cuda:0")
    sh = sv.VocabShard(to_device(w.target, w.dtype, dev), to_device(w.draft, w.dtype, dev),
                       torch.from_numpy(w.tokens).to(dev), 0, w.V, float(w.T[0]), float(w.Td[0]))
    t, n = sv.verify_vocab_parallel(sh, 9)
    torch.cuda.synchronize()
    r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, 9)
    ok = (r.flags & NEAR_TIE) == 0
    np.testing.assert_array_equal(n.cpu().numpy()[ok], r.n_accepted[ok])
    np.testing.assert_array_equal(t.cpu().numpy()[ok], r.tokens[ok])
