"""Pins of the oracle's p, q values and of its greedy mode (CPU only).

* log Z and ln p(d_i), ln q(d_i) against scipy's logsumexp / log_softmax (library routines),
  on fp32 and bf16 inputs, with T != T_d so a temperature mix-up fails.
* Greedy mode against numpy.argmax (first occurrence on ties) and the argmax-match rule,
  including planted ties and bad draft tokens.
* Basic output invariants: 0 <= j <= gamma, exactly j + 1 emitted tokens, -1 padding.
"""
import numpy as np
import pytest
from scipy.special import log_softmax, logsumexp

import oracle
import workloads


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_log_normalisers_and_draft_probabilities_match_scipy(dtype):
    w = workloads.generic(B=3, gamma=4, V=3001, dtype=dtype, seed=5, scale=3.0, sigma=0.8,
                          T=0.7, Td=0.3)
    r = oracle.get().verify(w.target, w.draft, w.tokens, w.T, w.Td, seed=9)
    t = workloads.as_f32(w.target, dtype).astype(np.float64)
    d = workloads.as_f32(w.draft, dtype).astype(np.float64)
    for b in range(w.B):
        Tb, Tdb = float(w.T[b]), float(w.Td[b])
        np.testing.assert_allclose(r.logZp[b], logsumexp(t[b] / Tb, axis=-1), rtol=1e-13)
        np.testing.assert_allclose(r.logZq[b], logsumexp(d[b] / Tdb, axis=-1), rtol=1e-13)
        lp = log_softmax(t[b, :w.gamma] / Tb, axis=-1)[np.arange(w.gamma), w.tokens[b]]
        lq = log_softmax(d[b] / Tdb, axis=-1)[np.arange(w.gamma), w.tokens[b]]
        np.testing.assert_allclose(r.logp[b], lp, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r.logq[b], lq, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r.a[b], np.exp(lp - lq), rtol=1e-12)


def test_row_overlap_matches_scipy():
    w = workloads.generic(B=1, gamma=6, V=777, dtype="bf16", seed=2, T=0.9, Td=0.4)
    t = workloads.as_f32(w.target[0, :6], "bf16").astype(np.float64)
    d = workloads.as_f32(w.draft[0], "bf16").astype(np.float64)
    p = np.exp(log_softmax(t / 0.9, axis=-1))
    q = np.exp(log_softmax(d / np.float64(np.float32(0.4)), axis=-1))
    got = oracle.get().row_overlap(w.target[0, :6], w.draft[0], 0.9,
                                   np.float64(np.float32(0.4)))
    np.testing.assert_allclose(got, np.minimum(p, q).sum(-1), rtol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_matches_numpy_argmax(dtype):
    w = workloads.generic(B=6, gamma=5, V=4099, dtype=dtype, seed=11, greedy=True)
    t = w.target.copy()
    # plant exact ties of the row maximum at a higher index, and one at a lower index
    tf = workloads.as_f32(t, dtype)
    for b in range(w.B):
        for i in range(w.gamma + 1):
            m = int(np.argmax(tf[b, i]))
            t[b, i, (m + 17) % w.V] = t[b, i, m]
    # break some drafts so the first mismatch moves around
    tok = w.tokens.copy()
    tok[1, 0] = (tok[1, 0] + 1) % w.V
    tok[2, 3] = (tok[2, 3] + 5) % w.V
    out_t, out_n, g = oracle.get().verify_greedy(t, tok)
    tf = workloads.as_f32(t, dtype)
    ref_g = np.argmax(tf, axis=-1)
    np.testing.assert_array_equal(g, ref_g)
    for b in range(w.B):
        match = tok[b] == ref_g[b, :w.gamma]
        j = int(np.argmin(match)) if not match.all() else w.gamma
        assert out_n[b] == j
        np.testing.assert_array_equal(out_t[b, :j], tok[b, :j])
        assert out_t[b, j] == ref_g[b, j]
        assert np.all(out_t[b, j + 1:] == -1)


def test_greedy_bad_token_marks_sequence():
    w = workloads.generic(B=3, gamma=4, V=100, dtype="f32", seed=1, greedy=True)
    tok = w.tokens.copy()
    tok[1, 2] = 100
    tok[2, 0] = -3
    out_t, out_n, _ = oracle.get().verify_greedy(w.target, tok)
    assert out_n[0] == 4 and out_n[1] == -1 and out_n[2] == -1
    assert np.all(out_t[1] == -1) and np.all(out_t[2] == -1)


def test_sampling_bad_token_marks_sequence():
    w = workloads.generic(B=2, gamma=3, V=50, dtype="f32", seed=4)
    tok = w.tokens.copy()
    tok[0, 2] = 50
    r = oracle.get().verify(w.target, w.draft, tok, w.T, w.Td, seed=0)
    assert r.n_accepted[0] == -1 and np.all(r.tokens[0] == -1)
    assert r.flags[0] & oracle.FLAG_BAD_TOKEN
    assert 0 <= r.n_accepted[1] <= 3


@pytest.mark.parametrize("gamma,V", [(0, 1), (0, 9), (1, 1), (3, 8), (5, 1024), (7, 1000)])
def test_output_invariants(gamma, V):
    """At least one token per cycle; tau = j + 1 in [1, gamma + 1]; prefix = drafts."""
    w = workloads.generic(B=64, gamma=gamma, V=V, dtype="f32", seed=gamma * 100 + V, sigma=1.0)
    for seed in range(4):
        r = oracle.get().verify(w.target, w.draft, w.tokens, w.T, w.Td, seed=seed)
        assert np.all((r.n_accepted >= 0) & (r.n_accepted <= gamma))
        for b in range(w.B):
            j = r.n_accepted[b]
            np.testing.assert_array_equal(r.tokens[b, :j], w.tokens[b, :j])
            assert 0 <= r.tokens[b, j] < V
            assert np.all(r.tokens[b, j + 1:] == -1)
            # accepted prefix passed the test, the deciding position failed it
            assert np.all(r.u[b, :j] < r.a[b, :j])
            if j < gamma:
                assert r.u[b, j] >= r.a[b, j]
