"""GPU parity of the early-exit sampling path (SPEC_FLAG_EARLY_EXIT) against the oracle and
the full-read path (marked gpu).

The early-exit path reads a sequence's rows one position at a time and stops after its first
rejection.  Its outputs follow the same rules as the full read: tokens and counts equal the
oracle's except at flagged near-ties.  The cases run gamma = 0..13 and 48, draft noise from
small (long accepted prefixes, the bonus row) to large (early rejections), and include bad
tokens in a late position, degenerate distributions, per-sequence temperatures, split
batches, repeated calls on one caller workspace, and the two batched workloads at full
size.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import DeviceWorkload, compare_sampling, gpu_near_ties, run_gpu

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


def early(sv, dw, seed, **kw):
    return run_gpu(sv, dw, seed, diagnostics=False, flags=sv.SPEC_FLAG_EARLY_EXIT, **kw)


SHAPES = [
    # B, gamma, V, dtype, draft noise sigma
    (1, 5, 1024, "f32", 0.5),
    (3, 4, 5003, "bf16", 0.3),
    (2, 7, 9000, "f32", 0.2),
    (4, 0, 777, "bf16", 1.0),
    (2, 3, 1, "f32", 1.0),
    (5, 2, 7, "bf16", 0.5),
    (6, 1, 4100, "f32", 0.8),
    (8, 8, 20000, "bf16", 0.1),
    (7, 9, 6001, "bf16", 0.05),
    (5, 13, 3000, "f32", 0.02),
    (3, 48, 2500, "bf16", 0.01),
    (33, 6, 12000, "bf16", 1.2),
]


@pytest.mark.parametrize("B,gamma,V,dtype,sigma", SHAPES)
def test_early_exit_small(sv, orc, B, gamma, V, dtype, sigma):
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B * 7 + V + gamma,
                          sigma=sigma, T=0.9, Td=0.7)
    dw = DeviceWorkload(w)
    for seed in range(4):
        g = early(sv, dw, seed, per_seq_temps=False)
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        compare_sampling(w, g, r)
        full = run_gpu(sv, dw, seed, per_seq_temps=False, diagnostics=False)
        flagged = (r.flags & (oracle.FLAG_ACCEPT_NEAR_TIE | oracle.FLAG_RACE_NEAR_TIE |
                              oracle.FLAG_RESIDUAL_EMPTY)) != 0
        ok = ~flagged
        np.testing.assert_array_equal(g["n"][ok], full["n"][ok])
        np.testing.assert_array_equal(g["tokens"][ok], full["tokens"][ok])
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_early_exit_reaches_every_position(sv, orc):
    """Draft = target at the same temperature accepts every position, so the bonus row
    decides; the other sequences reject at planted positions (p(d) = 0) from 0 to 12."""
    B, gamma, V = 6, 13, 4000
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype="bf16", seed=5, T=1.0, Td=1.0)
    draft = w.target[:, :gamma].copy()
    tok = w.tokens.copy()
    # p(d) = 0 rejects: make target logit -inf at the planted token of sequence b
    target = w.target.copy()
    ninf = workloads.to_bf16_bits(np.array([-np.inf], dtype=np.float32))[0]
    for b, i in enumerate([None, 0, 1, 3, 7, 12]):
        if i is not None:
            target[b, i, tok[b, i]] = ninf
    w2 = workloads.Workload("every-position", B, gamma, V, "bf16", target, draft, tok, w.T, w.Td)
    dw = DeviceWorkload(w2)
    for seed in range(3):
        g = early(sv, dw, seed, per_seq_temps=False)
        r = orc.verify(w2.target, w2.draft, w2.tokens, w2.T, w2.Td, seed)
        compare_sampling(w2, g, r)
        assert list(g["n"]) == [gamma, 0, 1, 3, 7, 12]


def test_early_exit_per_sequence_temperatures_and_split(sv, orc):
    w = workloads.generic(B=10, gamma=6, V=7000, dtype="bf16", seed=21, sigma=0.4)
    rng = np.random.default_rng(3)
    w.T[:] = rng.uniform(0.3, 1.2, size=w.B)
    w.Td[:] = 0.5 * w.T
    dw = DeviceWorkload(w)
    for seed in range(3):
        g = early(sv, dw, seed, per_seq_temps=True)
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        compare_sampling(w, g, r)
    full = early(sv, dw, 9, per_seq_temps=True)
    halves = [early(sv, DeviceWorkload(w.subset(range(lo, lo + 5))), 9, per_seq_temps=True,
                    seq_index_base=lo) for lo in (0, 5)]
    np.testing.assert_array_equal(full["tokens"], np.concatenate([h["tokens"] for h in halves]))
    np.testing.assert_array_equal(full["n"], np.concatenate([h["n"] for h in halves]))


def test_early_exit_bad_token_in_a_late_position(sv, orc):
    w = workloads.generic(B=4, gamma=12, V=900, dtype="bf16", seed=6, sigma=0.05)
    tok = w.tokens.copy()
    tok[1, 11] = 900    # checked at position 0 although position 11 is never reached
    tok[2, 0] = -1
    dw = DeviceWorkload(w)
    dtok = torch.from_numpy(tok).cuda()
    t, n, _ = sv.spec_verify_ex(dw.target, dw.draft, dtok, 1.0, 1.0, 3,
                                flags=sv.SPEC_FLAG_EARLY_EXIT)
    assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
    assert sv.spec_verify_check() == sv.SPEC_OK
    r = orc.verify(w.target, w.draft, tok, w.T, w.Td, 3)
    np.testing.assert_array_equal(n.cpu().numpy(), r.n_accepted)
    np.testing.assert_array_equal(t.cpu().numpy(), r.tokens)


def test_early_exit_degenerate_distributions(sv, orc):
    V, g = 3000, 5
    w = workloads.generic(B=3, gamma=g, V=V, dtype="f32", seed=8, T=0.9, Td=0.9)
    draft = w.draft.copy()
    draft[0] = -np.inf
    for i in range(g):
        draft[0, i, w.tokens[0, i]] = 0.0
    draft[1] = w.target[1, :g]
    tok = w.tokens.copy()
    tok[1] = np.argmax(w.target[1, :g], axis=-1)
    w2 = workloads.Workload("degenerate", 3, g, V, "f32", w.target, draft, tok, w.T, w.Td)
    dw = DeviceWorkload(w2)
    for seed in range(10):
        gres = early(sv, dw, seed, per_seq_temps=False)
        compare_sampling(w2, gres, orc.verify(w2.target, w2.draft, w2.tokens, w2.T, w2.Td, seed))
        assert gres["n"][1] == g


def test_early_exit_workspace_reuse_and_path_mixing(sv, orc):
    """Repeated early-exit calls on one caller workspace, interleaved with full-read calls
    on the same workspace, give the same outputs every time; diagnostics requested with the
    flag run the full read."""
    w = workloads.generic(B=9, gamma=7, V=11000, dtype="bf16", seed=4, sigma=0.3, T=1.0, Td=0.5)
    dw = DeviceWorkload(w)
    nbytes = sv.spec_verify_workspace_bytes(w.B, w.gamma, w.V, sv.SPEC_BF16)
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, 12)
    outs = []
    for k in range(6):
        t, n, d = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, 1.0, 0.5, 12, workspace=ws,
                                    d_status=status, diagnostics=(k == 5),
                                    flags=sv.SPEC_FLAG_EARLY_EXIT if k % 2 == 0 or k == 5 else 0)
        torch.cuda.synchronize()
        outs.append((t.cpu().numpy(), n.cpu().numpy()))
        if k == 5:
            assert d is not None and "logZp" in d
    assert sv.spec_verify_check(d_status=status) == sv.SPEC_OK
    for t, n in outs:
        compare_sampling(w, {"tokens": t, "n": n}, ref)
        np.testing.assert_array_equal(t, outs[0][0])
        np.testing.assert_array_equal(n, outs[0][1])


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_early_exit_named_single_sequence_workloads(sv, orc, cfg):
    w = workloads.config(cfg)
    dw = DeviceWorkload(w)
    for seed in range(6 if cfg == 0 else 3):
        g = early(sv, dw, seed)
        compare_sampling(w, g, orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed))


def test_early_exit_batched_serving_workload_full(sv, orc):
    """B=64, gamma=8, V=128256, per-sequence temperatures: every sequence checked."""
    w = workloads.config(3)
    dw = DeviceWorkload(w)
    for seed in range(2):
        g = early(sv, dw, seed, per_seq_temps=True)
        compare_sampling(w, g, orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed))


def test_early_exit_throughput_workload_full_size(sv, orc):
    """B=256, gamma=12, V=152064 (1.95 GB): 24 sampled sequences against the oracle, and
    all 256 against the full-read path (equal except near-ties that the full read's own
    diagnostics flag)."""
    w = workloads.config(4)
    dw = DeviceWorkload(w)
    idx = np.sort(np.random.default_rng(1).choice(w.B, size=24, replace=False))
    sub = w.subset(idx)
    for seed in (0, 3):
        g = early(sv, dw, seed, per_seq_temps=False)
        full = run_gpu(sv, dw, seed, per_seq_temps=False, diagnostics=True)
        flagged = gpu_near_ties(full, w.gamma)
        ok = ~flagged
        assert flagged.sum() <= 2
        np.testing.assert_array_equal(g["n"][ok], full["n"][ok])
        np.testing.assert_array_equal(g["tokens"][ok], full["tokens"][ok])
        parts = [orc.verify(sub.target[k:k + 1], sub.draft[k:k + 1], sub.tokens[k:k + 1],
                            sub.T[k:k + 1], sub.Td[k:k + 1], seed, b_base=int(b))
                 for k, b in enumerate(idx)]
        r = oracle.OracleResult(**{f: np.concatenate([getattr(p, f) for p in parts])
                                   for f in oracle.OracleResult.__dataclass_fields__})
        compare_sampling(sub, g, r, idx=idx)
