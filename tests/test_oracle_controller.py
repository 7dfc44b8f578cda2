"""Pins of the oracle's per-position statistics and of the adaptive draft length
([SPARSESPEC] "投机解码的第二本账", section 3.3; KL as quoted by [SUBSPEC]).

Entropies and KL divergences are checked against scipy (library routines with their own
softmax and log), against closed forms (uniform rows, one-hot rows, KL(p || p) = 0, q = 0
under p > 0), and against Gibbs' inequality.  The class-centre update and the k* rule are
checked on hand-worked cases and against the closed form of a geometric series.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import entropy

import oracle
import workloads


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("temp", [0.2, 0.6, 1.0, 1.7])
def test_entropy_matches_scipy(orc, dtype, temp):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((6, 777)) * 3).astype(np.float32)
    rows = workloads.to_bf16_bits(x) if dtype == "bf16" else x
    wide = workloads.as_f32(rows, dtype).astype(np.float64)
    want = [entropy(softmax(r / temp)) for r in wide]
    np.testing.assert_allclose(orc.row_entropies(rows, temp), want, rtol=1e-12, atol=1e-12)


def test_entropy_special_cases(orc):
    V = 1000
    flat = np.zeros((1, V), np.float32)
    assert orc.row_entropies(flat, 1.0)[0] == pytest.approx(math.log(V), abs=1e-12)
    one_hot = np.full((1, V), -np.inf, np.float32)
    one_hot[0, 17] = 3.0
    assert orc.row_entropies(one_hot, 0.7)[0] == 0.0
    two = np.full((1, V), -np.inf, np.float32)
    two[0, [3, 9]] = 1.0
    assert orc.row_entropies(two, 1.0)[0] == pytest.approx(math.log(2), abs=1e-15)


@pytest.mark.parametrize("T,Td", [(1.0, 1.0), (0.6, 0.2), (1.3, 0.8)])
def test_kl_matches_scipy_and_gibbs(orc, T, Td):
    rng = np.random.default_rng(5)
    t = (rng.standard_normal((5, 911)) * 2).astype(np.float32)
    d = (t + rng.standard_normal(t.shape) * 0.7).astype(np.float32)
    got = orc.row_kl(t, d, T, Td)
    want = [entropy(softmax(a.astype(np.float64) / T), softmax(b.astype(np.float64) / Td))
            for a, b in zip(t, d)]
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-13)
    assert np.all(got >= 0)
    # KL(p || p) = 0 at equal temperatures
    np.testing.assert_allclose(orc.row_kl(t, t, T, T), 0.0, atol=1e-13)


def test_kl_infinite_when_q_misses_support(orc):
    t = np.zeros((1, 8), np.float32)
    d = np.zeros((1, 8), np.float32)
    d[0, 2] = -np.inf
    assert orc.row_kl(t, d, 1.0, 1.0)[0] == np.inf
    # q covering p's support: finite even with p = 0 elsewhere
    t2 = np.full((1, 8), -np.inf, np.float32)
    t2[0, 4] = 0.0
    assert orc.row_kl(t2, np.zeros((1, 8), np.float32), 1.0, 1.0)[0] == pytest.approx(math.log(8))


def test_position_stats_against_scipy(orc):
    """H(p_i) over target rows 0..g, H(q_i) and KL(p_i || q_i) pairing target and draft row
    i, with per-sequence temperatures."""
    w = workloads.generic(B=3, gamma=4, V=600, dtype="bf16", seed=11, sigma=0.8)
    T = np.array([0.5, 1.0, 1.4])
    Td = T * 0.5
    hp, hq, kl = orc.position_stats(w.target, w.draft, T, Td)
    tw = workloads.as_f32(w.target, "bf16").astype(np.float64)
    dw = workloads.as_f32(w.draft, "bf16").astype(np.float64)
    for b in range(3):
        for i in range(5):
            assert hp[b, i] == pytest.approx(entropy(softmax(tw[b, i] / T[b])), rel=1e-11)
        for i in range(4):
            p, q = softmax(tw[b, i] / T[b]), softmax(dw[b, i] / Td[b])
            assert hq[b, i] == pytest.approx(entropy(q), rel=1e-11, abs=1e-13)
            assert kl[b, i] == pytest.approx(entropy(p, q), rel=1e-10, abs=1e-13)


def test_centre_update_hand_worked(orc):
    H = np.array([[1.0, 2.0, 3.0, 4.0]] * 4)
    c0 = np.array([[10.0, 20.0]] * 4)
    n = np.array([2, 4, 0, -1], np.int32)
    c = orc.entropy_centres_update(H, n, 0.5, c0)
    # rejected at 2: positions 0, 1 accepted (10 -> 5.5 -> 3.75), position 2 rejected
    assert c[0].tolist() == [3.75, 11.5]
    # all accepted: four updates of the accepted centre, the rejected one untouched
    assert c[1].tolist() == [3.6875, 20.0]  # 10 -> 5.5 -> 3.75 -> 3.375 -> 3.6875
    # rejected at 0: only the rejected centre moves
    assert c[2].tolist() == [10.0, 10.5]
    # bad draft: unchanged
    assert c[3].tolist() == [10.0, 20.0]


def test_soft_accept_rule(orc):
    assert orc.soft_accept(1.0, 1.0, 3.0) == 1.0      # on the accepted centre
    assert orc.soft_accept(3.0, 1.0, 3.0) == 0.0      # on the rejected centre
    assert orc.soft_accept(2.0, 1.0, 3.0) == 0.5      # midway
    assert orc.soft_accept(2.0, 2.0, 2.0) == 0.5      # centres coincide
    assert orc.soft_accept(1.5, 1.0, 3.0) == pytest.approx(0.75)
    assert orc.soft_accept(0.0, 1.0, 3.0) == pytest.approx(0.75)  # beyond the accepted centre
    # lower entropy than the accepted centre is more confident than higher
    assert orc.soft_accept(0.5, 1.0, 3.0) > orc.soft_accept(1.8, 1.0, 3.0)


@pytest.mark.parametrize("a,Cd,Cv", [(0.75, 0.2, 1.0), (0.9, 0.2, 1.0), (0.5, 0.7, 1.0),
                                     (0.95, 0.05, 1.0), (0.3, 1.0, 1.0)])
def test_adaptive_k_geometric_closed_form(orc, a, Cd, Cv):
    """Every draft token at the same entropy gives p_i = a, so
    sum_{m=1..k} prod_{i<=m} p_i = a (1 - a^k) / (1 - a)."""
    K = 24
    c_acc, c_rej = 0.0, 1.0
    H = np.full((2, K), 1.0 - a)  # d_acc = 1 - a, d_rej = a  ->  p = a
    cand = np.array([1, 2, 3, 4, 6, 8, 10, 12, 16, 20, 24], np.int32)
    k, eff = orc.adaptive_k(H, np.array([[c_acc, c_rej]] * 2), cand, Cd, Cv)
    effs = [(1 + a * (1 - a ** kk) / (1 - a)) / (kk * Cd + Cv) for kk in cand]
    assert k[0] == cand[int(np.argmax(effs))] and k[1] == k[0]
    assert eff[0] == pytest.approx(max(effs), rel=1e-12)


def test_adaptive_k_limits(orc):
    K = 8
    cand = np.array([2, 4, 8], np.int32)
    H = np.full((1, K), 0.25)
    c = np.array([[0.0, 1.0]])
    # free drafts: the longest candidate wins; hopeless drafts: the shortest
    assert orc.adaptive_k(H, c, cand, 0.0, 1.0)[0][0] == 8
    assert orc.adaptive_k(np.full((1, K), 1.0), c, cand, 0.5, 1.0)[0][0] == 2
    # confidence that drops after the third token stops the draft there
    Hs = np.array([[0.0, 0.0, 0.0, 1.0, 1.0, 1.0, 1.0, 1.0]])
    assert orc.adaptive_k(Hs, c, np.arange(1, 9, dtype=np.int32), 0.1, 1.0)[0][0] == 3
    with pytest.raises(ValueError):
        orc.adaptive_k(H, c, np.array([0, 3], np.int32), 0.1, 1.0)


CONTROLLER_MUTATIONS = {6: "centres swapped", 7: "soft classification inverted",
                        8: "yield sums p_i", 9: "entropy sign"}


@pytest.mark.parametrize("mutation", sorted(CONTROLLER_MUTATIONS))
def test_planted_controller_mistakes_fail_the_pins(mutation, tmp_path):
    """Each planted mistake in a rebuilt oracle fails one of the pins above."""
    path = str(tmp_path / f"liboracle_m{mutation}.so")
    oracle.build(path, mutation=mutation)
    bad = oracle.Oracle(path)
    failed = []
    for name, fn in (("entropy", lambda: test_entropy_special_cases(bad)),
                     ("centres", lambda: test_centre_update_hand_worked(bad)),
                     ("soft", lambda: test_soft_accept_rule(bad)),
                     ("geometric", lambda: test_adaptive_k_geometric_closed_form(bad, 0.75, 0.2, 1.0))):
        try:
            fn()
        except AssertionError:
            failed.append(name)
    assert failed, CONTROLLER_MUTATIONS[mutation]
