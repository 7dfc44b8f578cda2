"""GPU parity of libspecverify against the CPU oracle (marked gpu).

Every call goes through the C ABI (the ctypes binding).  Sizes span several row pieces
with ragged tails, unaligned rows (V not a multiple of 8), gamma = 0, fp32 and bf16,
scalar and per-sequence temperatures; the five named workloads run in the launch
configuration the benchmark times (full size; the two batched ones compared on sampled
sequences, which the oracle can compute one by one).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import DeviceWorkload, compare_greedy, compare_sampling, run_gpu

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


SMALL_SHAPES = [
    # B, gamma, V, dtype
    (1, 5, 1024, "f32"),
    (3, 4, 5003, "bf16"),    # unaligned rows, ragged last piece
    (2, 7, 9000, "f32"),     # several pieces
    (4, 0, 777, "bf16"),     # plain sampling
    (2, 3, 1, "f32"),        # V = 1
    (5, 2, 7, "bf16"),       # V < one vector
    (2, 6, 20000, "bf16"),   # several pieces, aligned rows
    (3, 1, 8, "bf16"),       # V = one bf16 vector, gamma = 1
    (2, 1, 9, "f32"),        # V = two f32 vectors and one, rows off 16-byte boundaries
    (1, 1, 4100, "f32"),     # piece boundary + 4
]


TINY_SHAPES = [
    # B, gamma, V, dtype: rows of at most 4 KB (the one-launch small-sequence path)
    (4, 7, 2048, "bf16"),
    (3, 0, 1024, "f32"),
    (8, 3, 512, "bf16"),
    (2, 6, 64, "f32"),
    (5, 2, 8, "bf16"),
]


@pytest.mark.parametrize("B,gamma,V,dtype", TINY_SHAPES)
def test_tiny_sequences(sv, orc, B, gamma, V, dtype):
    """Tiny sequences (the one-launch small-sequence path) with per-sequence temperatures,
    diagnostics, a bad draft token and a sequence whose draft equals its target, against
    the oracle."""
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B * 100 + V + gamma, sigma=0.7,
                          T=0.8, Td=0.5)
    T = np.linspace(0.4, 1.6, B).astype(np.float32)
    Td = (T * np.linspace(0.3, 1.0, B)).astype(np.float32)
    draft, tok = w.draft.copy(), w.tokens.copy()
    if gamma and B > 2:
        draft[1] = w.target[1, :gamma]
        Td[1] = T[1]
        tok[2, gamma - 1] = V  # out of range: sequence 2 is marked
    w2 = workloads.Workload("tiny", B, gamma, V, dtype, w.target, draft, tok, T, Td)
    dw = DeviceWorkload(w2)
    for seed in range(3):
        r = orc.verify(w2.target, w2.draft, w2.tokens, w2.T, w2.Td, seed)
        g = run_gpu(sv, dw, seed, diagnostics=(seed == 0))
        compare_sampling(w2, g, r, check_values=(seed == 0))
        if gamma and B > 2:
            assert g["n"][2] == -1 and np.all(g["tokens"][2] == -1)
            assert g["n"][1] == gamma  # p = q: every draft token accepted
    if gamma and B > 2:
        assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
    assert sv.spec_verify_check() == sv.SPEC_OK


@pytest.mark.parametrize("B,gamma,V,dtype", SMALL_SHAPES)
def test_greedy_small(sv, orc, B, gamma, V, dtype):
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B * 1000 + V, greedy=True)
    dw = DeviceWorkload(w)
    # make some drafts disagree so the first mismatch moves
    tok = w.tokens.copy()
    if gamma:
        tok[0, gamma // 2] = (tok[0, gamma // 2] + 1) % V if V > 1 else tok[0, gamma // 2]
    dtok = torch.from_numpy(tok).cuda()
    out_t, out_n = sv.spec_verify_greedy_ex(dw.target, dtok)
    torch.cuda.synchronize()
    rt, rn, _ = orc.verify_greedy(w.target, tok)
    compare_greedy(out_t.cpu().numpy(), out_n.cpu().numpy(), rt, rn)
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_greedy_ties_lowest_index(sv, orc):
    w = workloads.generic(B=2, gamma=3, V=30000, dtype="bf16", seed=3, greedy=True)
    t = w.target.copy()
    tf = workloads.as_f32(t, "bf16")
    for b in range(2):
        for i in range(4):
            m = int(np.argmax(tf[b, i]))
            for off in (9001, 17, 4096 * 3):       # equal maxima after the first
                t[b, i, (m + off) % w.V] = t[b, i, m]
            if m > 5:
                t[b, i, m - 5] = t[b, i, m]        # ... and one before it
    dt = torch.from_numpy(t.view(np.int16)).view(torch.bfloat16).cuda()
    out_t, out_n = sv.spec_verify_greedy(dt, torch.from_numpy(w.tokens).cuda())
    torch.cuda.synchronize()
    rt, rn, _ = orc.verify_greedy(t, w.tokens)
    compare_greedy(out_t.cpu().numpy(), out_n.cpu().numpy(), rt, rn)


@pytest.mark.parametrize("B,gamma,V,dtype", SMALL_SHAPES)
@pytest.mark.parametrize("temps", [(1.0, 1.0), (0.6, 0.2), (1.3, 0.8)])
def test_sampling_small(sv, orc, B, gamma, V, dtype, temps):
    T, Td = temps
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B * 7 + V, sigma=0.7, T=T,
                          Td=Td)
    dw = DeviceWorkload(w)
    for seed in range(6):
        g = run_gpu(sv, dw, seed, per_seq_temps=(seed % 2 == 0))
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        compare_sampling(w, g, r)
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_per_sequence_temperatures(sv, orc):
    w = workloads.config(3, B=6)          # first 6 sequences of the batched workload
    assert len(np.unique(w.T)) == 6
    dw = DeviceWorkload(w)
    for seed in range(3):
        g = run_gpu(sv, dw, seed, per_seq_temps=True)
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        compare_sampling(w, g, r)


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_named_single_sequence_workloads(sv, orc, cfg):
    w = workloads.config(cfg)
    dw = DeviceWorkload(w)
    nseeds = {0: 200, 1: 12, 2: 6}[cfg]
    for seed in range(nseeds):
        g = run_gpu(sv, dw, seed, per_seq_temps=False, diagnostics=(seed < 3))
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        compare_sampling(w, g, r, check_values=(seed < 3))


def test_named_single_sequence_greedy(sv, orc):
    w = workloads.config(1, greedy=True)
    dw = DeviceWorkload(w)
    out_t, out_n = sv.spec_verify_greedy(dw.target, dw.tokens)
    torch.cuda.synchronize()
    rt, rn, _ = orc.verify_greedy(w.target, w.tokens)
    compare_greedy(out_t.cpu().numpy(), out_n.cpu().numpy(), rt, rn)
    assert rn[0] == w.gamma or rt[0, rn[0]] != w.tokens[0, rn[0]]


def test_batched_serving_workload_full(sv, orc):
    """B=64, gamma=8, V=128256 with per-sequence temperatures: every sequence checked."""
    w = workloads.config(3)
    dw = DeviceWorkload(w)
    for seed in range(2):
        g = run_gpu(sv, dw, seed, per_seq_temps=True, diagnostics=(seed == 0))
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        compare_sampling(w, g, r, check_values=(seed == 0))
    wg = workloads.config(3, greedy=True)
    dg = DeviceWorkload(wg)
    out_t, out_n = sv.spec_verify_greedy(dg.target, dg.tokens)
    torch.cuda.synchronize()
    rt, rn, _ = orc.verify_greedy(wg.target, wg.tokens)
    compare_greedy(out_t.cpu().numpy(), out_n.cpu().numpy(), rt, rn)


def _oracle_pool_verify(cfg, seeds):
    """The oracle's verify of every sequence of named workload `cfg` for each seed, the seeds
    spread over processes (spawned: the parent holds a CUDA context; each regenerates the
    workload from its seeded recipe).  Returns {seed: OracleResult}."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import os
    workers = max(1, min(len(seeds), (os.cpu_count() or 1)))
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        futs = {s: ex.submit(_oracle_verify_config, cfg, s) for s in seeds}
        return {s: f.result() for s, f in futs.items()}


def _oracle_verify_config(cfg, seed):
    # runs in a spawned worker
    import oracle as orc_mod
    import workloads as wl
    w = wl.config(cfg)
    return orc_mod.get().verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)


def test_throughput_workload_full_size_every_sequence(sv, orc):
    """B=256, gamma=12, V=152064 bf16 (1.95 GB) in the benchmark's launch configuration:
    every one of the 256 sequences against the oracle for four seeds, on the full read and
    on the early-exit path (the oracle's result is the same for both)."""
    seeds = (0, 1, 2, 3)
    refs = _oracle_pool_verify(4, seeds)
    w = workloads.config(4)
    dw = DeviceWorkload(w)
    for seed in seeds:
        r = refs[seed]
        g = run_gpu(sv, dw, seed, per_seq_temps=False, diagnostics=(seed < 2))
        compare_sampling(w, g, r, check_values=(seed < 2))
        assert np.all((g["n"] >= 0) & (g["n"] <= w.gamma))
        ge = run_gpu(sv, dw, seed, per_seq_temps=False, diagnostics=False,
                     flags=sv.SPEC_FLAG_EARLY_EXIT)
        compare_sampling(w, ge, r, check_values=False, count=False)


@pytest.mark.parametrize("sigma,T,Td", [(0.0, 1.0, 1.0), (0.1, 1.0, 1.0), (0.1, 0.7, 0.7), (0.3, 1.0, 0.8)])
def test_long_accepted_prefixes(sv, orc, sigma, T, Td):
    """Drafts close to the target (draft = target at sigma = 0): long accepted prefixes, bonus
    races, and residual races where q is close to p, so that many tokens pass the race
    filter and are scored exactly.  Every sequence against the oracle, on the full read and
    on the early-exit path."""
    w = workloads.generic(B=16, gamma=8, V=128256, dtype="bf16", seed=77, scale=3.0,
                          sigma=sigma, T=T, Td=Td, kind="zipf")
    dw = DeviceWorkload(w)
    for seed in (0, 1):
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        g = run_gpu(sv, dw, seed, diagnostics=(seed == 0))
        compare_sampling(w, g, r, check_values=(seed == 0))
        ge = run_gpu(sv, dw, seed, diagnostics=False, flags=sv.SPEC_FLAG_EARLY_EXIT)
        compare_sampling(w, ge, r, check_values=False, count=False)
    if sigma == 0.0 and T == Td:
        assert np.all(r.n_accepted == w.gamma)  # p / q = 1 accepts every draft token
    assert sv.spec_verify_check() == sv.SPEC_OK


@pytest.mark.parametrize("B,gamma,V,dtype,sigma", [(2, 2048, 40, "f32", 0.0), (3, 2048, 33, "bf16", 0.01),
                                                   (4, 300, 257, "bf16", 0.01)])
def test_longest_drafts(sv, orc, B, gamma, V, dtype, sigma):
    """Draft lengths past the positions the scan gathers ahead (256) up to the largest gamma
    the library takes (2048), with drafts so close to the target that the first rejection
    falls deep in the draft (sigma = 0: never), on the full read, the early-exit path and in
    greedy mode, against the oracle; gamma = 2049 is refused."""
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=gamma + V, scale=2.0,
                          sigma=sigma, T=1.0, Td=1.0)
    dw = DeviceWorkload(w)
    accepted = []
    for seed in (0, 1):
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        g = run_gpu(sv, dw, seed, diagnostics=(seed == 0))
        compare_sampling(w, g, r, check_values=(seed == 0))
        ge = run_gpu(sv, dw, seed, diagnostics=False, flags=sv.SPEC_FLAG_EARLY_EXIT)
        compare_sampling(w, ge, r, check_values=False, count=False)
        accepted.append(r.n_accepted)
    accepted = np.concatenate(accepted)
    if sigma == 0.0:
        assert np.all(accepted == gamma)
    else:
        assert np.any(accepted > 256)  # some rejection past the gathered-ahead positions
    wg = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=gamma + V + 1, scale=2.0,
                           sigma=sigma, greedy=True)
    dg = DeviceWorkload(wg)
    out_t, out_n = sv.spec_verify_greedy_ex(dg.target, dg.tokens)
    torch.cuda.synchronize()
    rt, rn, _ = orc.verify_greedy(wg.target, wg.tokens)
    compare_greedy(out_t.cpu().numpy(), out_n.cpu().numpy(), rt, rn)
    assert sv.spec_verify_check() == sv.SPEC_OK
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_ex(torch.zeros((1, 2050, 8), dtype=torch.float32, device="cuda"),
                          torch.zeros((1, 2049, 8), dtype=torch.float32, device="cuda"),
                          torch.zeros((1, 2049), dtype=torch.int32, device="cuda"), 1.0, 1.0, 0)
    assert e.value.code == sv.SPEC_EINVAL


@pytest.mark.parametrize("B", [180, 240, 400])
def test_batch_sizes_around_the_race_wave(sv, orc, B):
    """The race's three grid layouts by batch size against one resident wave of race blocks
    (304 on a 152-SM GPU): chunks shared evenly with blocks straddling two sequences (180),
    one block per sequence when the batch fills three quarters of the wave (240), and more
    sequences than the wave holds (400) -- every sequence against the oracle."""
    w = workloads.generic(B=B, gamma=3, V=3001, dtype="bf16", seed=B, sigma=0.8, T=0.9, Td=0.6)
    dw = DeviceWorkload(w)
    for seed in (0, 1):
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        g = run_gpu(sv, dw, seed, diagnostics=(seed == 0))
        compare_sampling(w, g, r, check_values=(seed == 0))
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_a_million_token_vocabulary(sv, orc):
    """V = 2^20 + 3 (1024 race chunks and a ragged tail per raced row) against the oracle, on
    the full read and the early-exit path."""
    w = workloads.generic(B=2, gamma=2, V=(1 << 20) + 3, dtype="bf16", seed=11, sigma=0.9,
                          T=1.0, Td=0.7)
    dw = DeviceWorkload(w)
    for seed in (0, 1, 2):
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        g = run_gpu(sv, dw, seed, diagnostics=(seed == 0))
        compare_sampling(w, g, r, check_values=(seed == 0))
        ge = run_gpu(sv, dw, seed, diagnostics=False, flags=sv.SPEC_FLAG_EARLY_EXIT)
        compare_sampling(w, ge, r, check_values=False, count=False)
    assert sv.spec_verify_check() == sv.SPEC_OK


@pytest.mark.parametrize("B,gamma,V,dtype", [(24, 8, 128257, "bf16"), (20, 8, 65537, "f32")])
def test_streaming_claim_launch_unaligned_rows(sv, orc, B, gamma, V, dtype):
    """Calls with more row pieces than the streaming grid has warps take the claiming launch
    (one block per SM, pieces claimed from a shared counter); here with rows that start off
    16-byte boundaries (odd V), against the oracle, in sampling and greedy mode."""
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B + V, sigma=0.8, T=0.9, Td=0.45)
    dw = DeviceWorkload(w)
    for seed in (0, 3):
        g = run_gpu(sv, dw, seed, diagnostics=(seed == 0))
        compare_sampling(w, g, orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed),
                         check_values=(seed == 0))
    out_t, out_n = sv.spec_verify_greedy_ex(dw.target, dw.tokens)
    torch.cuda.synchronize()
    rt, rn, _ = orc.verify_greedy(w.target, w.tokens)
    compare_greedy(out_t.cpu().numpy(), out_n.cpu().numpy(), rt, rn)
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_seq_index_base_splits_a_batch(sv, orc):
    """Two half-batch calls with seq_index_base give exactly the one-call result."""
    w = workloads.generic(B=8, gamma=5, V=6000, dtype="bf16", seed=9, T=0.8, Td=0.4)
    dw = DeviceWorkload(w)
    full = run_gpu(sv, dw, 5, per_seq_temps=False, diagnostics=False)
    halves = []
    for lo in (0, 4):
        sub = w.subset(range(lo, lo + 4))
        halves.append(run_gpu(sv, DeviceWorkload(sub), 5, per_seq_temps=False,
                              seq_index_base=lo, diagnostics=False))
    np.testing.assert_array_equal(full["tokens"], np.concatenate([h["tokens"] for h in halves]))
    np.testing.assert_array_equal(full["n"], np.concatenate([h["n"] for h in halves]))


def test_seq_index_base_wraps_like_the_oracle(sv, orc):
    """Global sequence indices are 32-bit counter words: a base of 2^32 - 3 wraps to 0 within
    the batch, on the device exactly as in the oracle (full read and early exit)."""
    w = workloads.generic(B=6, gamma=4, V=7001, dtype="bf16", seed=12, sigma=0.6, T=0.9, Td=0.5)
    dw = DeviceWorkload(w)
    base = (1 << 32) - 3
    for seed in (0, 1):
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed, b_base=base)
        g = run_gpu(sv, dw, seed, seq_index_base=base, diagnostics=(seed == 0))
        compare_sampling(w, g, r, check_values=(seed == 0))
        ge = run_gpu(sv, dw, seed, seq_index_base=base, diagnostics=False,
                     flags=sv.SPEC_FLAG_EARLY_EXIT)
        compare_sampling(w, ge, r, check_values=False, count=False)


def test_repeatable_and_caller_workspace(sv, orc):
    w = workloads.generic(B=5, gamma=6, V=33000, dtype="bf16", seed=4, T=1.0, Td=0.3)
    dw = DeviceWorkload(w)
    a = run_gpu(sv, dw, 77, per_seq_temps=False, diagnostics=False)
    nbytes = sv.spec_verify_workspace_bytes(w.B, w.gamma, w.V, sv.SPEC_BF16)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):  # tickets must be left at zero by every call
        t, n, _ = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]),
                                    float(w.Td[0]), 77, workspace=ws, d_status=status)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(t.cpu().numpy(), a["tokens"])
        np.testing.assert_array_equal(n.cpu().numpy(), a["n"])
    assert sv.spec_verify_check(d_status=status) == sv.SPEC_OK
    small = torch.zeros(nbytes // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, 1.0, 1.0, 0, workspace=small)
    assert e.value.code == sv.SPEC_ENOMEM


def test_bad_tokens_are_reported(sv, orc):
    w = workloads.generic(B=4, gamma=3, V=500, dtype="bf16", seed=6)
    tok = w.tokens.copy()
    tok[1, 1] = 500
    tok[3, 0] = -1
    dw = DeviceWorkload(w)
    dtok = torch.from_numpy(tok).cuda()
    t, n, _ = sv.spec_verify_ex(dw.target, dw.draft, dtok, 1.0, 1.0, 3)
    assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
    assert sv.spec_verify_check() == sv.SPEC_OK  # reading clears it
    r = orc.verify(w.target, w.draft, tok, w.T, w.Td, 3)
    np.testing.assert_array_equal(n.cpu().numpy(), r.n_accepted)
    np.testing.assert_array_equal(t.cpu().numpy(), r.tokens)
    tg, ng = sv.spec_verify_greedy(dw.target, dtok)
    assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
    assert ng.cpu().numpy()[1] == -1 and ng.cpu().numpy()[3] == -1


def test_degenerate_distributions(sv, orc):
    """-inf draft logits (q = 0 outside the draft token), identical draft and target."""
    V, g = 3000, 4
    w = workloads.generic(B=3, gamma=g, V=V, dtype="f32", seed=8, T=0.9, Td=0.9)
    draft = w.draft.copy()
    # sequence 0: one-hot q on its draft tokens (draft logits -inf elsewhere)
    draft[0] = -np.inf
    for i in range(g):
        draft[0, i, w.tokens[0, i]] = 0.0
    # sequence 1: draft identical to target, same temperature -> never rejects
    draft[1] = w.target[1, :g]
    tok = w.tokens.copy()
    tok[1] = np.argmax(w.target[1, :g], axis=-1)
    w2 = workloads.Workload("degenerate", 3, g, V, "f32", w.target, draft, tok, w.T, w.Td)
    dw = DeviceWorkload(w2)
    for seed in range(20):
        gres = run_gpu(sv, dw, seed, per_seq_temps=False)
        r = orc.verify(w2.target, w2.draft, w2.tokens, w2.T, w2.Td, seed)
        compare_sampling(w2, gres, r)
        assert gres["n"][1] == g


@pytest.mark.parametrize("dtype,T,Td", [("bf16", 1.0, 0.5), ("f32", 0.05, 0.05), ("bf16", 20.0, 8.0)])
def test_masked_vocabulary_and_extreme_temperatures(sv, orc, dtype, T, Td):
    """Logits masked to -inf (a third of the vocabulary, the same tokens in target and
    draft, as a constrained or padded vocabulary gives), one sequence whose target rows keep
    a single token (p one-hot), one whose draft tokens are masked in the target (p(d) = 0:
    rejected at position 0), at sharp and flat temperatures -- against the oracle, on the
    full read and the early-exit path."""
    B, g, V = 6, 5, 20011
    w = workloads.generic(B=B, gamma=g, V=V, dtype="f32", seed=int(T * 100) + V, sigma=0.4,
                          T=T, Td=Td)
    rng = np.random.default_rng(5)
    mask = rng.random(V) < 1.0 / 3.0
    tgt, drf, tok = w.target.copy(), w.draft.copy(), w.tokens.copy()
    tgt[:, :, mask] = -np.inf
    drf[:, :, mask] = -np.inf
    live = np.flatnonzero(~mask)
    for b in range(B):  # draft tokens drawn from the masked draft rows
        tok[b] = workloads.draw_drafts(rng, drf[b], float(Td))
    keep = live[7]
    tgt[1] = -np.inf
    tgt[1, :, keep] = 0.5                              # p one-hot on `keep`
    tgt[2, 0, tok[2, 0]] = -np.inf                     # p(d_0) = 0 for sequence 2
    enc = (lambda a: workloads.to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a.astype(np.float32))
    w2 = workloads.Workload("masked", B, g, V, dtype, enc(tgt), enc(drf), tok, w.T, w.Td)
    dw = DeviceWorkload(w2)
    for seed in range(4):
        r = orc.verify(w2.target, w2.draft, w2.tokens, w2.T, w2.Td, seed)
        gres = run_gpu(sv, dw, seed, diagnostics=(seed == 0))
        compare_sampling(w2, gres, r, check_values=(seed == 0))
        ge = run_gpu(sv, dw, seed, diagnostics=False, flags=sv.SPEC_FLAG_EARLY_EXIT)
        compare_sampling(w2, ge, r, check_values=False, count=False)
        assert r.n_accepted[2] == 0
        assert not mask[gres["tokens"][np.arange(B), gres["n"]]].any()  # no masked token drawn
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_empty_batch_and_invalid_arguments(sv):
    e = torch.empty((0, 4, 100), dtype=torch.bfloat16, device="cuda")
    d = torch.empty((0, 3, 100), dtype=torch.bfloat16, device="cuda")
    tok = torch.empty((0, 3), dtype=torch.int32, device="cuda")
    t, n = sv.spec_verify(e, d, tok, 1.0, 1.0, 0)
    assert t.shape == (0, 4) and n.shape == (0,)
    w = workloads.generic(B=2, gamma=3, V=64, dtype="bf16", seed=1)
    dw = DeviceWorkload(w)
    for T, Td in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        with pytest.raises(sv.SpecVerifyError) as ex:
            sv.spec_verify(dw.target, dw.draft, dw.tokens, T, Td, 0)
        assert ex.value.code == sv.SPEC_EINVAL
    # misaligned logit pointer
    flat = torch.zeros(2 * 4 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    mis = flat[1:].view(2, 4, 64)
    with pytest.raises(sv.SpecVerifyError) as ex:
        sv.spec_verify(mis, dw.draft, dw.tokens, 1.0, 1.0, 0)
    assert ex.value.code == sv.SPEC_EINVAL


def test_bounded_wait_times_out_and_context_survives(sv, orc):
    """The early-exit kernel's waits are bounded: with the test flag under which no race unit
    publishes its winner, each sequence's last race unit waits for them until the wait
    gives up (about half a second), records SPEC_ETIMEOUT and finishes; the context stays
    usable and the next normal call is correct."""
    import time
    w = workloads.generic(B=2, gamma=3, V=3000, dtype="bf16", seed=77)
    dw = DeviceWorkload(w)
    t0 = time.time()
    sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, 1.0, 1.0, 0,
                      flags=sv.SPEC_FLAG_EARLY_EXIT | sv.SPEC_DEBUG_NEVER_READY)
    assert sv.spec_verify_check() == sv.SPEC_ETIMEOUT
    assert time.time() - t0 < 30
    for flags in (0, sv.SPEC_FLAG_EARLY_EXIT):
        g = run_gpu(sv, dw, 0, per_seq_temps=False, diagnostics=False, flags=flags)
        assert sv.spec_verify_check() == sv.SPEC_OK
        compare_sampling(w, g, orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, 0))


def test_unknown_flag_bits_are_refused(sv):
    w = workloads.generic(B=2, gamma=3, V=300, dtype="bf16", seed=1)
    dw = DeviceWorkload(w)
    for bad in (1, 32, 1 << 31):
        with pytest.raises(sv.SpecVerifyError) as e:
            sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, 1.0, 1.0, 0, flags=bad)
        assert e.value.code == sv.SPEC_EINVAL
