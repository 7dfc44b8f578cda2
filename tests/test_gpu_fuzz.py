"""Seeded random shapes against the oracle (marked gpu): batch size, draft length,
vocabulary size (aligned and not), element type, temperatures (scalar and per sequence),
draft noise and sequence index base drawn at random, each case run on the full read, the
early-exit path and in greedy mode.  A net for the corners the named cases miss: rows off
16-byte boundaries, vocabularies of a few tokens to a few hundred thousand, one-sequence and
many-sequence calls.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import DeviceWorkload, compare_greedy, compare_sampling, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = int(os.environ.get("SPECVERIFY_FUZZ_CASES", "40"))  # more for a longer sweep


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_31_gb300 as m
    m.load_library()
    return m


def draw_case(rng):
    dtype = "bf16" if rng.random() < 0.6 else "f32"
    V = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 5000)),
                        int(rng.integers(5000, 70000)), int(rng.integers(70000, 300000))],
                       p=[0.15, 0.35, 0.3, 0.2]))
    if rng.random() < 0.5:
        V += (-V) % 8  # aligned rows for either element type
    gamma = int(rng.choice([0, 1, 2, 3, 5, 8, 13, 21]))
    max_b = max(1, min(48, 6_000_000 // max(1, (2 * gamma + 1) * V)))
    B = int(rng.integers(1, max_b + 1))
    T = float(rng.uniform(0.2, 2.0))
    return dict(B=B, gamma=gamma, V=V, dtype=dtype, T=T, Td=float(T * rng.uniform(0.3, 1.0)),
                sigma=float(rng.choice([0.05, 0.3, 0.8, 1.5])),
                kind=str(rng.choice(["normal", "zipf", "heavy"])),
                per_seq=bool(rng.random() < 0.5), base=int(rng.integers(0, 1 << 32)))


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_shapes(sv, case):
    rng = np.random.default_rng(20261202 + case)
    c = draw_case(rng)
    target_fn = {"normal": lambda r_, n, v: workloads.normal_rows(r_, n, v, 3.0),
                 "zipf": lambda r_, n, v: workloads.zipf_shaped_rows(r_, n, v, 3.0),
                 "heavy": (workloads.heavy_tailed_rows if c["V"] >= 16
                           else (lambda r_, n, v: workloads.normal_rows(r_, n, v, 3.0)))}[c["kind"]]

    def params(r_):  # per-sequence temperatures, drawn before the sequence's draft tokens
        t = r_.uniform(0.2, 2.0)
        return t, t * r_.uniform(0.3, 1.0), c["sigma"]

    w = workloads.make_workload(f"fuzz{case}", c["B"], c["gamma"], c["V"], c["dtype"], case, target_fn,
                                c["sigma"], c["T"], Td=c["Td"],
                                per_seq_params=params if c["per_seq"] else None)
    orc = oracle.get()
    dw = DeviceWorkload(w)
    r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, case, b_base=c["base"])
    g = run_gpu(sv, dw, case, per_seq_temps=c["per_seq"], seq_index_base=c["base"], diagnostics=True)
    compare_sampling(w, g, r, check_values=True)
    ge = run_gpu(sv, dw, case, per_seq_temps=c["per_seq"], seq_index_base=c["base"],
                 diagnostics=False, flags=sv.SPEC_FLAG_EARLY_EXIT)
    compare_sampling(w, ge, r, check_values=False, count=False)
    assert sv.spec_verify_check() == sv.SPEC_OK, c
    t, n = sv.spec_verify_greedy_ex(dw.target, dw.tokens)
    rt, rn, _ = orc.verify_greedy(w.target, w.tokens)
    compare_greedy(t.cpu().numpy(), n.cpu().numpy(), rt, rn)
    assert sv.spec_verify_check() == sv.SPEC_OK, c


N_SPLIT = int(os.environ.get("SPECVERIFY_FUZZ_SPLIT_CASES", "16"))
N_TREE = int(os.environ.get("SPECVERIFY_FUZZ_TREE_CASES", "16"))


@pytest.mark.parametrize("case", range(N_SPLIT))
def test_random_vocab_splits(sv, case):
    """The vocabulary-parallel steps on random shapes and rank counts (ranks emulated one
    after another on this GPU), against the oracle except at its flagged near-ties."""
    from _parity import NEAR_TIE
    from test_gpu_vocab_parallel import emulate
    rng = np.random.default_rng(7_000_000 + case)
    world = int(rng.integers(2, 9))
    dtype = "bf16" if rng.random() < 0.6 else "f32"
    V = int(rng.integers(8 * world + 1, 200_000))
    gamma = int(rng.choice([0, 1, 3, 6, 12]))
    B = int(rng.integers(1, max(2, min(16, 3_000_000 // ((2 * gamma + 1) * V)) + 1)))
    T = float(rng.uniform(0.3, 1.8))
    sigma = float(rng.choice([0.1, 0.6, 1.2]))
    per_seq = bool(rng.random() < 0.5)
    kind = str(rng.choice(["normal", "zipf", "heavy"]))
    target_fn = {"normal": lambda r_, n, v: workloads.normal_rows(r_, n, v, 3.0),
                 "zipf": lambda r_, n, v: workloads.zipf_shaped_rows(r_, n, v, 3.0),
                 "heavy": workloads.heavy_tailed_rows}[kind]

    def params(r_):
        t = r_.uniform(0.3, 1.8)
        return t, t * r_.uniform(0.3, 1.0), sigma

    w = workloads.make_workload(f"split{case}", B, gamma, V, dtype, case, target_fn, sigma, T,
                                Td=T * float(rng.uniform(0.3, 1.0)),
                                per_seq_params=params if per_seq else None)
    orc = oracle.get()
    seed = int(rng.integers(0, 1 << 31))
    vt, vn = emulate(sv, w, world, seed, per_seq=per_seq)
    r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
    ok = (r.flags & NEAR_TIE) == 0
    np.testing.assert_array_equal(vn[ok], r.n_accepted[ok])
    np.testing.assert_array_equal(vt[ok], r.tokens[ok])
    assert sv.spec_verify_check() == sv.SPEC_OK


@pytest.mark.parametrize("case", range(N_TREE))
def test_random_token_trees(sv, case):
    """Token-tree verifies of random trees, shapes and temperatures against the oracle."""
    from test_gpu_tree import compare_tree, run_tree
    rng = np.random.default_rng(9_000_000 + case)
    N = int(rng.integers(1, 80))
    parent = workloads.random_tree(rng, N, int(rng.integers(1, 6)))
    dtype = "bf16" if rng.random() < 0.6 else "f32"
    V = int(rng.integers(2, 60_000))
    if rng.random() < 0.5:
        V += (-V) % 8
    B = int(rng.integers(1, 6))
    T = float(rng.uniform(0.3, 1.8))
    w = workloads.tree(parent, B=B, V=V, dtype=dtype, seed=case, scale=3.0,
                       sigma=float(rng.choice([0.1, 0.6, 1.2])), T=T, Td=T * float(rng.uniform(0.3, 1.0)))
    orc = oracle.get()
    for seed in range(2):
        compare_tree(w, run_tree(sv, w, seed),
                     orc.verify_tree(w.target, w.draft, w.tokens, w.parent, w.T, w.Td, seed))
    assert sv.spec_verify_check() == sv.SPEC_OK
