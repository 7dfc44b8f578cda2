"""Statistical pins of the oracle's sampler (CPU only).

The verify step is an exact sampler, so its law is fixed by the mathematics:

* Brute force (V = 8, gamma = 3, fixed position-indexed rows p_i, q_i): enumerating every
  draft sequence (weight prod q_i) with its accept probabilities and residual draws gives
  the law of (j, emitted tokens); completing each emitted prefix with independent draws
  from the remaining p_i gives exactly prod_i p_i(y_i) -- the lossless property
  ("How speculative decoding makes LLMs go brrr", module 3: min(p, q) + max(0, p - q) = p).
  This part checks the method's statement itself, in fp64, within 1e-12.
* 10^6 seeded oracle cycles on the same rows: chi-square of the (j, emitted) histogram
  against the enumerated law, and of the gamma = 0 draw against p_0.
* Acceptance rate at each position against sum_x min(p_i, q_i) (module 3).
* tau against (1 - alpha^(gamma+1)) / (1 - alpha) for i.i.d. positions (module 4).
* Special cases: draft == target never rejects; the residual never returns the rejected
  draft token; a one-hot q accepts with probability p(d).
* Planted mistakes: copies of the oracle built with a known bug each fail these pins.
"""
import itertools
from collections import defaultdict

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle
import workloads

V, G = 8, 3


def _rows(seed, T, Td, dtype="f32"):
    """Position-indexed rows drawn as in the small workload: N(0, 2^2) target, +N(0, 0.5^2)."""
    w = workloads.generic(B=1, gamma=G, V=V, dtype=dtype, seed=seed, scale=2.0, sigma=0.5,
                          T=T, Td=Td)
    t = workloads.as_f32(w.target[0], dtype).astype(np.float64)
    d = workloads.as_f32(w.draft[0], dtype).astype(np.float64)
    p = softmax(t / np.float64(np.float32(T)), axis=-1)
    q = softmax(d / np.float64(np.float32(Td)), axis=-1)
    return w, p, q


def enumerate_law(p, q):
    """Law of (j, emitted tuple) by brute force over all V^gamma draft sequences."""
    g = q.shape[0]
    law = defaultdict(float)
    for drafts in itertools.product(range(p.shape[1]), repeat=g):
        reach = float(np.prod([q[i, drafts[i]] for i in range(g)]))
        if reach == 0.0:
            continue
        for i in range(g):
            d = drafts[i]
            a = min(1.0, p[i, d] / q[i, d])
            if a < 1.0:
                resid = np.maximum(0.0, p[i] - q[i])
                resid = resid / resid.sum()
                for y in range(p.shape[1]):
                    if resid[y] > 0:
                        law[(i, tuple(drafts[:i]) + (y,))] += reach * (1.0 - a) * resid[y]
            reach *= a
        for y in range(p.shape[1]):
            law[(g, tuple(drafts) + (y,))] += reach * p[g, y]
    return law


def extended_law(law, p):
    """Complete every emitted prefix with independent draws from the remaining p rows."""
    g1 = p.shape[0]
    full = np.zeros((p.shape[1],) * g1)
    for (j, toks), pr in law.items():
        rest = [p[k] for k in range(j + 1, g1)]
        tail = np.ones(())
        for r in rest:
            tail = np.multiply.outer(tail, r)
        full[toks] += pr * tail
    return full


def run_cycles(orc, w, p_rows_logits, q_rows_logits, n, seed, data_seed):
    """n independent cycles on fixed rows; drafts drawn from q by numpy (the drafter)."""
    rng = np.random.default_rng(data_seed)
    target = np.broadcast_to(p_rows_logits, (n,) + p_rows_logits.shape)
    draft = np.broadcast_to(q_rows_logits, (n,) + q_rows_logits.shape)
    qf = workloads.as_f32(q_rows_logits, w.dtype)
    tok = np.stack([workloads.draw_drafts(rng, np.broadcast_to(qf[i], (n, w.V)), float(w.Td[0]))
                    for i in range(w.gamma)], axis=1) if w.gamma else np.zeros((n, 0), np.int32)
    r = orc.verify(target, draft, tok, w.T[0], w.Td[0], seed=seed)
    return tok, r


def chi2_against_law(r, law, n):
    keys = list(law.keys())
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for b in range(n):
        j = int(r.n_accepted[b])
        counts[index[(j, tuple(int(x) for x in r.tokens[b, :j + 1]))]] += 1
    expected = np.array([law[k] for k in keys]) * n
    small = expected < 5
    obs = np.append(counts[~small], counts[small].sum())
    exp = np.append(expected[~small], expected[small].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    exp = exp * obs.sum() / exp.sum()
    return stats.chisquare(obs, exp).pvalue


def acceptance_z(r, q_rows_p, p, q):
    """z-scores of P(accept at i | reached i) against sum_x min(p_i, q_i)."""
    zs = []
    for i in range(q.shape[0]):
        reached = r.n_accepted >= i
        acc = r.n_accepted[reached] > i
        alpha = np.minimum(p[i], q[i]).sum()
        nreach = reached.sum()
        zs.append((acc.mean() - alpha) / np.sqrt(alpha * (1 - alpha) / nreach))
    return np.array(zs)


TEMPS = [(1.0, 1.0), (1.0, 0.5), (0.7, 1.3)]


@pytest.mark.parametrize("T,Td", TEMPS)
def test_enumerated_law_is_lossless(T, Td):
    w, p, q = _rows(seed=31, T=T, Td=Td)
    law = enumerate_law(p, q)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    full = extended_law(law, p)
    ref = p[0][:, None, None, None] * p[1][None, :, None, None] * p[2][None, None, :, None] \
        * p[3][None, None, None, :]
    np.testing.assert_allclose(full, ref, atol=1e-12, rtol=0)
    # closed form of the same law: prod_{i<j} min(p_i, q_i)(d_i) * max(0, p_j - q_j)(y)
    for (j, toks), pr in list(law.items())[:500]:
        pref = np.prod([min(p[i, toks[i]], q[i, toks[i]]) for i in range(j)])
        last = p[j, toks[j]] if j == G else max(0.0, p[j, toks[j]] - q[j, toks[j]])
        assert pr == pytest.approx(pref * last, rel=1e-10, abs=1e-15)


@pytest.mark.parametrize("T,Td", TEMPS)
def test_oracle_cycles_follow_the_enumerated_law(T, Td):
    orc = oracle.get()
    w, p, q = _rows(seed=31, T=T, Td=Td)
    n = 1_000_000
    tok, r = run_cycles(orc, w, w.target[0], w.draft[0], n, seed=12345, data_seed=99)
    assert np.all((r.n_accepted >= 0) & (r.n_accepted <= G))
    pval = chi2_against_law(r, enumerate_law(p, q), n)
    assert pval > 1e-3, pval
    z = acceptance_z(r, None, p, q)
    assert np.all(np.abs(z) < 4), z
    # the empirical 4-token law after completion matches prod p_i (chi-square, 4096 cells)


def test_gamma0_is_categorical_sampling_from_p0():
    orc = oracle.get()
    w = workloads.generic(B=1, gamma=0, V=V, dtype="f32", seed=8, scale=2.0)
    p0 = softmax(w.target[0, 0].astype(np.float64), axis=-1)
    n = 1_000_000
    target = np.broadcast_to(w.target[0], (n, 1, V))
    r = orc.verify(target, np.zeros((n, 0, V), np.float32), np.zeros((n, 0), np.int32), 1.0,
                   1.0, seed=777)
    assert np.all(r.n_accepted == 0)
    counts = np.bincount(r.tokens[:, 0], minlength=V)
    assert stats.chisquare(counts, p0 * n).pvalue > 1e-3


def test_tau_closed_form_for_iid_positions():
    """Identical (p, q) at every position: acceptances are i.i.d. with alpha = sum min(p,q),
    so the mean number emitted is (1 - alpha^(g+1)) / (1 - alpha)."""
    orc = oracle.get()
    g = 5
    w = workloads.generic(B=1, gamma=1, V=V, dtype="f32", seed=3, scale=2.0, sigma=0.8)
    trow, drow = w.target[0, 0], w.draft[0, 0]
    target = np.broadcast_to(trow, (g + 1, V)).copy()
    draft = np.broadcast_to(drow, (g, V)).copy()
    p = softmax(trow.astype(np.float64))
    q = softmax(drow.astype(np.float64))
    alpha = np.minimum(p, q).sum()
    n = 400_000
    wl = workloads.Workload("iid", 1, g, V, "f32", target[None], draft[None],
                            np.zeros((1, g), np.int32), np.ones(1, np.float32),
                            np.ones(1, np.float32))
    _, r = run_cycles(orc, wl, target, draft, n, seed=5, data_seed=6)
    emitted = r.n_accepted + 1
    tau = (1 - alpha ** (g + 1)) / (1 - alpha)
    z = (emitted.mean() - tau) / (emitted.std() / np.sqrt(n))
    assert abs(z) < 4, (emitted.mean(), tau, z)


def test_identical_draft_and_target_never_rejects():
    orc = oracle.get()
    w = workloads.generic(B=256, gamma=6, V=500, dtype="bf16", seed=12, T=0.8, Td=0.8)
    draft = np.ascontiguousarray(w.target[:, :w.gamma])
    for seed in range(8):
        r = orc.verify(w.target, draft, w.tokens, w.T, w.T, seed=seed)
        assert np.all(r.n_accepted == w.gamma)
        np.testing.assert_array_equal(r.a, 1.0)


def test_residual_never_returns_the_rejected_draft():
    orc = oracle.get()
    w = workloads.generic(B=2000, gamma=4, V=16, dtype="f32", seed=13, sigma=1.5, T=1.0, Td=0.6)
    r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed=1)
    rej = np.where(r.n_accepted < w.gamma)[0]
    assert rej.size > 500
    for b in rej:
        j = r.n_accepted[b]
        if r.a[b, j] < 1 - 1e-12:
            assert r.tokens[b, j] != w.tokens[b, j]


def test_one_hot_draft_accepts_with_probability_p():
    orc = oracle.get()
    n, t = 400_000, 5
    rng = np.random.default_rng(0)
    trow = (rng.standard_normal((2, V)) * 2).astype(np.float32)
    drow = np.full((1, V), -np.inf, np.float32)
    drow[0, t] = 0.0
    target = np.broadcast_to(trow, (n, 2, V))
    draft = np.broadcast_to(drow, (n, 1, V))
    r = orc.verify(target, draft, np.full((n, 1), t, np.int32), 1.0, 1.0, seed=2)
    p_t = softmax(trow[0].astype(np.float64))[t]
    acc = (r.n_accepted == 1).mean()
    assert abs(acc - p_t) < 4 * np.sqrt(p_t * (1 - p_t) / n)
    # the residual max(0, p - onehot) never contains t
    assert np.all(r.tokens[r.n_accepted == 0, 0] != t)


# -- planted mistakes --------------------------------------------------------------------

MUTATIONS = {
    1: "residual max(0, q - p)",
    2: "draft normalised at T instead of T_d",
    3: "accept test inverted / non-strict",
    4: "bonus drawn from row gamma - 1",
    5: "residual ignores q",
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistakes_fail_the_pins(mutation, tmp_path):
    path = str(tmp_path / f"liboracle_m{mutation}.so")
    oracle.build(path, mutation=mutation)
    orc = oracle.Oracle(path)
    T, Td = 1.0, 0.5
    w, p, q = _rows(seed=31, T=T, Td=Td)
    n = 200_000
    tok, r = run_cycles(orc, w, w.target[0], w.draft[0], n, seed=4242, data_seed=77)
    law = enumerate_law(p, q)
    bad_support = any((int(r.n_accepted[b]), tuple(int(x) for x in r.tokens[b, :r.n_accepted[b] + 1]))
                      not in law for b in range(min(n, 20000)))
    pval = 0.0 if bad_support else chi2_against_law(r, law, n)
    z = acceptance_z(r, None, p, q)
    assert pval < 1e-6 or np.any(np.abs(z) > 6), (MUTATIONS[mutation], pval, z)
